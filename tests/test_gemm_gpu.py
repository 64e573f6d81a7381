"""Block-scaled GEMM parity: the tcgen05 kernel against the oracle's binary64
dequantize-and-accumulate, within |D - ref| <= 1e-5 * ga*gb*sum|a*b| (binary32
output) plus one bf16 rounding, 2^-8 |ref|, for bf16 output."""
import json
import os

import numpy as np
import pytest

import oracle as O
from nvfp4_bit_quantized_quantize_gb300 import synth

from gpu_helpers import gemm

pytestmark = pytest.mark.gpu

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
REL = 1e-5
BF16_REL = 2.0 ** -8


def _check(d, ref, dabs, bf16, what=""):
    tol = REL * dabs + (BF16_REL * np.abs(ref) if bf16 else 0.0)
    err = np.abs(d - ref)
    bad = np.flatnonzero((err > tol).ravel())
    ratio = float(np.max(err / np.maximum(REL * dabs, 1e-300)))
    assert bad.size == 0, f"{what}: {bad.size} out of tolerance, first {bad[:5]}, max err/(1e-5 sum|ab|) = {ratio}"
    return ratio


def _random_operand(rows, K, rng, sf_lo=0x30, sf_hi=0x48):
    """Arbitrary NVFP4 operand: uniform codes over all 16, scale bytes drawn
    from [sf_lo, sf_hi) (E4M3 2^-1 .. 2^2), padding zero."""
    q = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    sf = np.zeros(O.sf_bytes(rows, K), np.uint8)
    kb = K // 16
    r = np.arange(rows)[:, None]
    k = np.arange(kb)[None, :]
    cp = (kb + 3) // 4
    off = ((r // 128) * cp + k // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (k % 4)
    sf[off.ravel()] = rng.integers(sf_lo, sf_hi, rows * kb, dtype=np.uint8)
    return q, sf


def test_worked_example_E4():
    # A row 0 = E1's codes (scale 448), B row 0 = 1.0 x 16 (scale 1.0); K = 64
    # with the other blocks zero; D[0, 0] = gA * 448 * 7.
    e1 = GOLD["E1"]
    x = np.zeros((128, 64), np.float32)
    x[0, :16] = [float(s) for s in e1["x"]]
    qa, sfa, ga = O.quantize(synth.f32_to_bf16_bits(x))
    qb = np.zeros((128, 32), np.uint8)
    qb[0, :8] = 0x22
    sfb = np.zeros(O.sf_bytes(128, 64), np.uint8)
    sfb[O.sf_offset(0, 0, 4)] = 0x38
    for f32 in (True, False):
        d, st = gemm(qa, sfa, ga, qb, sfb, 1.0, 128, 128, 64, out_f32=f32)
        assert st == 0
        expect = float(np.float32(ga)) * 448.0 * GOLD["E4"]["sum_codes"]
        assert d[0, 0] == pytest.approx(expect, rel=1e-6 if f32 else 2 ** -8)
        assert np.count_nonzero(d) == (1 if expect != 0 else 0)


@pytest.mark.parametrize("f32", [True, False])
def test_tiny_linear_layer_full(f32):
    # configs: X, W 256 x 256 from N(0,1) with 0.5% outliers x50 (seed 0),
    # 1x16 RN on both, Y = X W^T
    wl = synth.make_workload("tiny_linear_256")
    qa, sfa, ga = O.quantize(wl["X"])
    qb, sfb, gb = O.quantize(wl["W"])
    ref, dabs = O.gemm_f64(qa, sfa, ga, qb, sfb, gb, 256, 256, 256)
    d, st = gemm(qa, sfa, ga, qb, sfb, gb, 256, 256, 256, out_f32=f32)
    assert st == 0
    _check(d, ref, dabs, not f32, "tiny linear")


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (128, 256, 256), (256, 384, 320), (384, 128, 192),
                                   (128, 640, 576), (512, 512, 1024)])
def test_gemm_shapes_full_compare(M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    qa, sfa = _random_operand(M, K, rng)
    qb, sfb = _random_operand(N, K, rng)
    ga, gb = 0.75, 1.5
    ref, dabs = O.gemm_f64(qa, sfa, ga, qb, sfb, gb, M, N, K)
    for f32 in (True, False):
        d, st = gemm(qa, sfa, ga, qb, sfb, gb, M, N, K, out_f32=f32)
        assert st == 0
        _check(d, ref, dabs, not f32, f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 5, 32), (100, 136, 96), (130, 300, 160), (64, 40, 224),
                                   (257, 129, 4128), (200, 520, 288), (129, 257, 32)])
def test_gemm_ragged_shapes(M, N, K):
    """M, N off the 128/256 tiles and K off the 64/256 steps: the on-chip
    padding must not change any written value, and nothing past N is written."""
    rng = np.random.default_rng(M * 11 + N * 5 + K)
    qa, sfa = _random_operand(M, K, rng)
    qb, sfb = _random_operand(N, K, rng)
    ga, gb = 1.25, 0.5
    ref, dabs = O.gemm_f64(qa, sfa, ga, qb, sfb, gb, M, N, K)
    for f32 in (True, False):
        d, st = gemm(qa, sfa, ga, qb, sfb, gb, M, N, K, out_f32=f32)
        assert st == 0
        _check(d, ref, dabs, not f32, f"ragged {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(8192, 4096, 64), (6000, 2100, 96)])
def test_gemm_many_tiles_short_k(M, N, K):
    """One or two K stages per tile and ~14 tiles per CTA: the stage ring,
    the scale slots and the accumulator hand-over wrap around many times."""
    rng = np.random.default_rng(M + N + K)
    qa, sfa = _random_operand(M, K, rng)
    qb, sfb = _random_operand(N, K, rng)
    ga, gb = 0.5, 0.25
    d, st = gemm(qa, sfa, ga, qb, sfb, gb, M, N, K)
    assert st == 0
    ms = np.concatenate([rng.integers(0, M, 8192), np.arange(M), np.full(N, M - 1)])
    ns = np.concatenate([rng.integers(0, N, 8192), np.arange(M) % N, np.arange(N)])
    ref, dabs = O.gemm_f64_sampled(qa, sfa, ga, qb, sfb, gb, M, N, K, ms, ns)
    _check(d[ms, ns], ref, dabs, True, f"many tiles {M}x{N}x{K}")


def test_ragged_linear_layer_from_quantizers():
    """Quantize X [200, 96] and W [136, 96] with the CUDA quantizers (whose
    scale padding the GEMM relies on) and multiply: Y = X W^T."""
    from gpu_helpers import quantize
    x = synth.normal_bf16((200, 96), 51, 0, 1.0, 0.0, 0.01, 20.0)
    w = synth.normal_bf16((136, 96), 51, 1, 0.02)
    qa, sfa, ga, st_a = quantize(x)
    qb, sfb, gb, st_b = quantize(w)
    assert st_a == 0 and st_b == 0
    ref, dabs = O.gemm_f64(qa, sfa, ga, qb, sfb, gb, 200, 136, 96)
    d, st = gemm(qa, sfa, ga, qb, sfb, gb, 200, 136, 96, out_f32=True)
    assert st == 0
    _check(d, ref, dabs, False, "ragged layer")


@pytest.mark.parametrize("M", [128, 256, 384])
def test_scale_layout_one_hot(M):
    # Distinct power-of-two scale per (row, 16-block) of A: each output
    # element isolates one scale, so a wrong scale-factor layout shows up.
    # M = 128 runs the one-SM kernel, larger M the paired-SM kernel (both
    # CTAs' A rows, and a ragged second pair tile at 384).
    N, K = 128, 256
    rng = np.random.default_rng(5)
    qa = np.full((M, K // 2), 0x22, np.uint8)              # all 1.0
    qb = np.zeros((N, K // 2), np.uint8)
    kb = K // 16
    for n in range(N):
        blk = n % kb
        qb[n, blk * 8:(blk + 1) * 8] = 0x22                # B row n selects block n % kb
    sfa = np.zeros(O.sf_bytes(M, K), np.uint8)
    vals = rng.integers(0x20, 0x50, (M, kb), dtype=np.uint8)
    for r in range(M):
        for k in range(kb):
            sfa[O.sf_offset(r, k, kb)] = vals[r, k]
    sfb = np.zeros(O.sf_bytes(N, K), np.uint8)
    for n in range(N):
        for k in range(kb):
            sfb[O.sf_offset(n, k, kb)] = 0x38 + (n // kb) % 4 * 8  # 1, 2, 4, 8
    ref, dabs = O.gemm_f64(qa, sfa, 1.0, qb, sfb, 1.0, M, N, K)
    d, st = gemm(qa, sfa, 1.0, qb, sfb, 1.0, M, N, K, out_f32=True)
    assert st == 0
    assert np.array_equal(d, ref)


@pytest.mark.parametrize("M,N", [(128, 384), (256, 384), (512, 512)])
def test_scale_layout_one_hot_b(M, N):
    # The B side: a distinct scale per (row n, 16-block) of B, and A row m
    # selecting 16-block m % kb, so output (m, n) isolates B's scale of (n,
    # m % kb).  N = 384 and 512 cover both halves of a pair tile's 256 B rows
    # (each CTA of a pair stages one half) and a second N tile.
    K = 256
    kb = K // 16
    rng = np.random.default_rng(6)
    qa = np.zeros((M, K // 2), np.uint8)
    for m in range(M):
        blk = m % kb
        qa[m, blk * 8:(blk + 1) * 8] = 0x22                # A row m selects block m % kb
    qb = np.full((N, K // 2), 0x22, np.uint8)              # all 1.0
    sfa = np.zeros(O.sf_bytes(M, K), np.uint8)
    for r in range(M):
        for k in range(kb):
            sfa[O.sf_offset(r, k, kb)] = 0x38
    sfb = np.zeros(O.sf_bytes(N, K), np.uint8)
    vals = rng.integers(0x20, 0x50, (N, kb), dtype=np.uint8)
    for n in range(N):
        for k in range(kb):
            sfb[O.sf_offset(n, k, kb)] = vals[n, k]
    ref, dabs = O.gemm_f64(qa, sfa, 1.0, qb, sfb, 1.0, M, N, K)
    d, st = gemm(qa, sfa, 1.0, qb, sfb, 1.0, M, N, K, out_f32=True)
    assert st == 0
    assert np.array_equal(d, ref)


# ------------------------------------------------- full workload shapes ----
FULL = [
    ("fprop_w2d", 8192, 20480, 5120),
    ("wgrad_rht", 5120, 5120, 16384),
    ("mlp_up_fprop", 8192, 11008, 4096),
    ("mlp_down_fprop", 8192, 4096, 11008),
    ("mlp_up_wgrad", 11008, 4096, 8192),
    ("mlp_down_wgrad", 4096, 11008, 8192),
]


@pytest.mark.parametrize("name,M,N,K", FULL)
def test_gemm_full_size_sampled(name, M, N, K):
    rng = np.random.default_rng(K)
    qa, sfa = _random_operand(M, K, rng)
    qb, sfb = _random_operand(N, K, rng)
    ga, gb = 0.01, 0.02
    d, st = gemm(qa, sfa, ga, qb, sfb, gb, M, N, K, out_f32=True)
    assert st == 0
    ms = np.concatenate([rng.integers(0, M, 4096), np.full(N, 7), np.full(N, M - 1), np.arange(M), np.arange(M)])
    ns = np.concatenate([rng.integers(0, N, 4096), np.arange(N), np.arange(N), np.full(M, 3), np.full(M, N - 2)])
    ref, dabs = O.gemm_f64_sampled(qa, sfa, ga, qb, sfb, gb, M, N, K, ms, ns)
    _check(d[ms, ns], ref, dabs, False, name)
