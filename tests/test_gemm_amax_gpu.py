"""The GEMM that reduces its output's tensor amaxes, and the one-read dual
quantizer that takes them.

nvfp4_gemm_amax must write exactly nvfp4_gemm's bf16 output, and its two
maxima must equal the oracle's max |D| and max |RHT(D)| of that output
(bit-exact: both are plain maxima of values computed in the same binary32
order).  nvfp4_quantize_dual_from_amax must then write exactly what the oracle's
1x16 and Hadamard quantizers write for the same tensor ("I ricercatori di
Nvidia ...", "Come funziona NVFP4?": the tensor scale from the tensor's amax;
"Entrenamiento ...", "Metodología de Entrenamiento": the Hadamard form).
"""
import numpy as np
import pytest
import torch

import nvfp4_bit_quantized_quantize_gb300 as nv
import oracle as O
from nvfp4_bit_quantized_quantize_gb300 import synth
from gpu_helpers import gemm, gemm_amax, quantize_dual_from_amax

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed, outliers=0.001):
    a = synth.normal_bf16((M, K), seed, 0, 1.0, 0.0, outliers, 100.0)
    b = synth.normal_bf16((N, K), seed, 1, 0.05)
    qa, sfa, ga = O.quantize(a, O.RN, 0)
    qb, sfb, gb = O.quantize(b, O.RN, 0)
    return qa, sfa, ga, qb, sfb, gb


def _same(got, want, what):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, what
    bad = np.flatnonzero(got.ravel() != want.ravel())
    assert bad.size == 0, f"{what}: {bad.size} differ, first at {bad[0]}"


# M <= 128 (one 256-row pair tile, the odd CTA's rows all padding), one pair
# tile, ragged N and K, several tiles with ragged edges, a tile grid
SHAPES = [(16, 48, 64), (128, 256, 256), (256, 272, 320), (528, 1040, 512), (1024, 2048, 1024)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_amax_output_and_maxima(M, N, K):
    ops = _operands(M, N, K, seed=M + N)
    d_bits, amax, st = gemm_amax(*ops, M, N, K, rht_seed=7)
    assert st == 0
    got = synth.bf16_bits_to_f32(d_bits).astype(np.float64)
    if M > 128:
        # the same paired-SM kernel as the plain GEMM: its output bit for bit
        plain, st2 = gemm(*ops, M, N, K)
        assert st2 == 0
        _same(got, plain, "D")
    else:
        # (the plain GEMM runs these on the one-SM kernel): the GEMM tolerance
        ref, dabs = O.gemm_f64(*ops, M, N, K)
        assert np.all(np.abs(got - ref) <= 1e-5 * dabs + 2.0 ** -8 * np.abs(ref))
    assert amax[0] == O.amax(d_bits)
    assert amax[1] == O.rht_amax(d_bits, 7)


def test_gemm_amax_seeds_and_extremes_at_the_edges():
    # the largest |D| in the last row and last column of a ragged grid, once
    # negative: an A row and a B row scaled up
    M, N, K = 400, 784, 256
    a = synth.normal_bf16((M, K), 3, 0, 1.0)
    b = synth.normal_bf16((N, K), 3, 1, 0.05)
    a[M - 1] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(a[M - 1]) * 40.0)
    b[N - 1] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(b[N - 1]) * -40.0)
    qa, sfa, ga = O.quantize(a, O.RN, 0)
    qb, sfb, gb = O.quantize(b, O.RN, 0)
    ws = nv.alloc_workspace()
    for seed in (0, 1, 12345):
        d_bits, amax, st = gemm_amax(qa, sfa, ga, qb, sfb, gb, M, N, K, rht_seed=seed, ws=ws)
        assert st == 0
        dm = np.abs(synth.bf16_bits_to_f32(d_bits))
        assert np.unravel_index(np.argmax(dm), dm.shape) == (M - 1, N - 1)
        assert amax[0] == O.amax(d_bits)
        assert amax[1] == O.rht_amax(d_bits, seed)


def test_gemm_amax_starts_afresh_on_every_call():
    # one workspace: a call with small outputs after one with large outputs
    # must report its own maxima (the grid's last warp clears the partials)
    M, N, K = 512, 512, 256
    ws = nv.alloc_workspace()
    big = _operands(M, N, K, seed=1, outliers=0.01)
    small = list(_operands(M, N, K, seed=2, outliers=0.0))
    small[2] *= 1e-3
    for ops in (big, tuple(small), big):
        d_bits, amax, st = gemm_amax(*ops, M, N, K, rht_seed=3, ws=ws)
        assert st == 0
        assert amax[0] == O.amax(d_bits) and amax[1] == O.rht_amax(d_bits, 3)


@pytest.mark.parametrize("modes", [(nv.RN, nv.RN), (nv.SR, nv.SR)])
def test_gemm_then_one_read_dual_matches_oracle(modes):
    M, N, K = 528, 1040, 512
    mode, mode_t = modes
    d_bits, amax, st = gemm_amax(*_operands(M, N, K, seed=5), M, N, K, rht_seed=11)
    assert st == 0
    q, sf, g, qT, sfT, gT, st = quantize_dual_from_amax(d_bits, amax, mode, 21, 11, mode_t, 22)
    assert st == 0
    rq, rsf, rg = O.quantize(d_bits, mode, 21)
    rqT, rsfT, rgT = O.rht_quantize(d_bits, 11, mode_t, 22)
    assert g == rg and gT == rgT
    _same(q, rq, "row codes")
    _same(sf, rsf, "row scales")
    _same(qT, rqT, "Hadamard codes")
    _same(sfT, rsfT, "Hadamard scales")


@pytest.mark.parametrize("T,C", [(16, 16), (80, 272), (1040, 528), (4096, 1536)])
def test_one_read_dual_with_oracle_maxima(T, C):
    # maxima from the oracle, every tile shape including ragged token and
    # channel tiles; SR on both forms
    x = synth.normal_bf16((T, C), T + C, 0, 1.0, 0.0, 0.001, 100.0)
    amax = [O.amax(x), O.rht_amax(x, 4)]
    q, sf, g, qT, sfT, gT, st = quantize_dual_from_amax(x, amax, nv.SR, 8, 4, nv.SR, 9)
    assert st == 0
    rq, rsf, rg = O.quantize(x, O.SR, 8)
    rqT, rsfT, rgT = O.rht_quantize(x, 4, O.SR, 9)
    assert g == rg and gT == rgT
    _same(q, rq, "row codes")
    _same(sf, rsf, "row scales")
    _same(qT, rqT, "Hadamard codes")
    _same(sfT, rsfT, "Hadamard scales")


def test_one_read_dual_reports_a_nonfinite_amax():
    x = synth.normal_bf16((64, 256), 1, 0)
    for amax in ([np.inf, 1.0], [1.0, np.nan]):
        assert quantize_dual_from_amax(x, amax, nv.RN, 0, 1, nv.SR, 2)[6] == 4
    # a GEMM whose bf16 output overflows hands on an infinite amax
    M, N, K = 256, 256, 256
    qa, sfa, ga, qb, sfb, gb = _operands(M, N, K, seed=9)
    d_bits, amax, st = gemm_amax(qa, sfa, 3.0e38, qb, sfb, 1.0, M, N, K, rht_seed=1)
    assert not np.isfinite(amax[0])
    assert quantize_dual_from_amax(d_bits, amax, nv.RN, 0, 1, nv.SR, 2)[6] == 4


def test_argument_errors_are_returned_before_launch():
    ws = nv.alloc_workspace()
    fake = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    g = torch.ones(2, dtype=torch.float32, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:   # M % 16 != 0
        nv.nvfp4_gemm_amax(fake, fake, g, fake, fake, g, 24, 32, 64, fake, 32, 0, g, ws)
    assert e.value.status == 2
    with pytest.raises(nv.NVFP4Error) as e:   # no amax output
        nv.nvfp4_gemm_amax(fake, fake, g, fake, fake, g, 32, 32, 64, fake, 32, 0, None, ws)
    assert e.value.status == 1
    with pytest.raises(nv.NVFP4Error) as e:   # no amax input
        nv.nvfp4_quantize_dual_from_amax(fake, 32, 32, 32, None, 0, 0, fake, fake, g, 1, 1, 0, fake, fake, g, ws)
    assert e.value.status == 1
