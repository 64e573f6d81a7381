"""Quantizer parity: the CUDA kernels against the oracle, bit for bit (codes,
raw swizzled scale bytes including padding, and the binary32 tensor scale)."""
import json
import os

import numpy as np
import pytest

import oracle as O
import nvfp4_bit_quantized_quantize_gb300 as nv
from nvfp4_bit_quantized_quantize_gb300 import synth

from gpu_helpers import quantize, quantize_2d, quantize_dual, rht_quantize

pytestmark = pytest.mark.gpu

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def _assert_same(gpu, ref, what):
    g = np.asarray(gpu)
    r = np.asarray(ref)
    assert g.shape == r.shape, what
    bad = np.flatnonzero(g.ravel() != r.ravel())
    assert bad.size == 0, f"{what}: {bad.size} mismatches, first at {bad[:8]}: gpu {g.ravel()[bad[:8]]} ref {r.ravel()[bad[:8]]}"


SHAPES = [(256, 256), (1, 16), (16, 48), (200, 80), (130, 1040), (384, 192), (1024, 1024)]


@pytest.mark.parametrize("mode", [nv.RN, nv.SR])
@pytest.mark.parametrize("shape", SHAPES)
def test_quantize_1x16_parity(shape, mode):
    x = synth.normal_bf16(shape, 11, shape[0] % 7, 1.0, 0.0, 0.005, 50.0)
    q, sf, g, st = quantize(x, mode, seed=1234)
    rq, rsf, rg = O.quantize(x, mode, 1234)
    assert st == 0
    assert np.float32(g) == np.float32(rg)
    _assert_same(q, rq, "codes")
    _assert_same(sf, rsf, "scales")


def test_quantize_leading_dimension_and_workspace_reuse():
    x = synth.normal_bf16((136, 96), 5, 0)
    ws = nv.alloc_workspace()
    for mode in (nv.RN, nv.SR, nv.RN):
        q, sf, g, st = quantize(x, mode, seed=7, ld=136, ws=ws)
        rq, rsf, rg = O.quantize(x, mode, 7)
        assert st == 0 and g == rg
        _assert_same(q, rq, "codes")
        _assert_same(sf, rsf, "scales")


def test_worked_examples_on_gpu():
    e1, e2 = GOLD["E1"], GOLD["E2"]
    x = synth.f32_to_bf16_bits(np.array([[float(s) for s in e1["x"] + e2["x"]]], np.float32))
    q, sf, g, st = quantize(x, nv.RN)
    assert st == 0
    assert q[0, :8].tobytes().hex() == e1["packed_hex"]
    assert q[0, 8:].tobytes().hex() == e2["packed_hex"]
    assert sf[0] == int(e1["scale_byte"], 16) and sf[1] == int(e2["scale_byte"], 16)
    assert np.float32(g).view(np.uint32) == int(e1["g_f32_hex"], 16)


def test_zero_tensor_and_signed_zero():
    x = synth.f32_to_bf16_bits(np.array([[0.0] * 8 + [-0.0] * 8] * 3, np.float32))
    for mode in (nv.RN, nv.SR):
        q, sf, g, st = quantize(x, mode, 3)
        assert st == 0 and g == 0.0
        assert np.all(sf == 0)
        assert q[0].tobytes().hex() == "0000000088888888"


def test_tiny_values_and_saturating_scales():
    # amax in the bf16 subnormal range: s_enc saturates to FLT_MAX; zeros stay zero
    x = np.zeros((4, 32), np.float32)
    x[0, :5] = [2.0 ** -133, -2.0 ** -130, 2.0 ** -127, 0.0, -0.0]
    x[3, 17] = 2.0 ** -126
    xb = synth.f32_to_bf16_bits(x)
    for mode in (nv.RN, nv.SR):
        q, sf, g, st = quantize(xb, mode, 9)
        rq, rsf, rg = O.quantize(xb, mode, 9)
        assert st == 0 and g == rg
        _assert_same(q, rq, "codes")
        _assert_same(sf, rsf, "scales")


def test_nonfinite_input_is_reported():
    x = synth.normal_bf16((64, 64), 3, 0)
    x[5, 7] = 0x7F80  # +inf
    _, _, _, st = quantize(x)
    assert st == 4
    x[5, 7] = 0xFFC1  # NaN
    _, _, _, st = quantize(x)
    assert st == 4


# (48, 80), (144, 208), (80, 192), (176, 320): rows not a multiple of 32 (the
# transposed rows leave as 8-byte halves) and of 128; (16, 16), (80, 192),
# (176, 320): an odd count of 64-column tiles (zero padding rows in the last
# transposed scale atom)
@pytest.mark.parametrize("shape", [(256, 256), (48, 80), (144, 208), (16, 16), (512, 1024), (80, 192), (176, 320)])
def test_quantize_2d_parity(shape):
    w = synth.normal_bf16(shape, 21, 0, 0.02, 0.0, 0.002, 100.0)
    q, sf, qT, sfT, g, st = quantize_2d(w)
    rq, rsf, rqT, rsfT, rg = O.quantize_2d(w)
    assert st == 0 and g == rg
    _assert_same(q, rq, "codes")
    _assert_same(sf, rsf, "scales")
    _assert_same(qT, rqT, "transposed codes")
    _assert_same(sfT, rsfT, "transposed scales")


def test_quantize_2d_without_transpose():
    w = synth.normal_bf16((96, 64), 22, 0, 0.02)
    q, sf, _, _, g, st = quantize_2d(w, transpose=False)
    rq, rsf, _, _, rg = O.quantize_2d(w, transpose=False)
    assert st == 0 and g == rg
    _assert_same(q, rq, "codes")
    _assert_same(sf, rsf, "scales")


@pytest.mark.parametrize("mode", [nv.RN, nv.SR])
@pytest.mark.parametrize("shape", [(64, 128), (48, 40), (272, 200), (16, 8), (1024, 384)])
def test_rht_quantize_parity(shape, mode):
    x = synth.normal_bf16(shape, 31, 1, 1e-3 if mode == nv.SR else 1.0)
    qT, sfT, g, st = rht_quantize(x, rht_seed=77, mode=mode, sr_seed=5)
    rqT, rsfT, rg = O.rht_quantize(x, 77, mode, 5)
    assert st == 0 and g == rg
    _assert_same(qT, rqT, "codes")
    _assert_same(sfT, rsfT, "scales")


@pytest.mark.parametrize("modes", [(nv.RN, nv.SR), (nv.SR, nv.RN)])
@pytest.mark.parametrize("shape", [(64, 128), (48, 80), (272, 208), (16, 16), (1024, 384), (192, 1040)])
def test_quantize_dual_parity(shape, modes):
    """One read, two outputs: each equals the single-form oracle quantizer."""
    mode, mode_t = modes
    x = synth.normal_bf16(shape, 41, shape[1] % 5, 1.0, 0.0, 0.01, 30.0)
    q, sf, g, qT, sfT, gT, st = quantize_dual(x, mode, 9, 123, mode_t, 10)
    rq, rsf, rg = O.quantize(x, mode, 9)
    rqT, rsfT, rgT = O.rht_quantize(x, 123, mode_t, 10)
    assert st == 0 and g == rg and gT == rgT
    _assert_same(q, rq, "row codes")
    _assert_same(sf, rsf, "row scales")
    _assert_same(qT, rqT, "transformed codes")
    _assert_same(sfT, rsfT, "transformed scales")


def test_quantize_dual_leading_dimension():
    x = synth.normal_bf16((128, 96), 42, 0, 1.0)
    q, sf, g, qT, sfT, gT, st = quantize_dual(x, nv.RN, 0, 3, nv.SR, 4, ld=136)
    rq, rsf, rg = O.quantize(x, O.RN, 0)
    rqT, rsfT, rgT = O.rht_quantize(x, 3, O.SR, 4)
    assert st == 0 and g == rg and gT == rgT
    _assert_same(q, rq, "row codes")
    _assert_same(sf, rsf, "row scales")
    _assert_same(qT, rqT, "transformed codes")
    _assert_same(sfT, rsfT, "transformed scales")


# ---------------------------------------------- full-size workload tensors ----

@pytest.mark.parametrize("name", ["A1024", "A4096", "A8192"])
def test_quantize_sweep_full_size(name):
    x = synth.make_workload("quantize_sweep", only={name})[name]
    seed = synth.WORKLOADS["quantize_sweep"]["seed"]
    for mode in (nv.RN, nv.SR):
        q, sf, g, st = quantize(x, mode, seed)
        rq, rsf, rg = O.quantize(x, mode, seed)
        assert st == 0 and g == rg
        _assert_same(q, rq, "codes")
        _assert_same(sf, rsf, "scales")


def test_weight_2d_full_size_fprop_workload():
    w = synth.make_workload("fprop_w2d_8192x20480x5120", only={"W"})["W"]
    q, sf, qT, sfT, g, st = quantize_2d(w)
    rq, rsf, rqT, rsfT, rg = O.quantize_2d(w)
    assert st == 0 and g == rg
    _assert_same(q, rq, "codes")
    _assert_same(sf, rsf, "scales")
    _assert_same(qT, rqT, "transposed codes")
    _assert_same(sfT, rsfT, "transposed scales")


def test_rht_sr_full_size_wgrad_workload():
    wl = synth.make_workload("wgrad_rht_sr_16384x5120", only={"dY"})
    seed = synth.WORKLOADS["wgrad_rht_sr_16384x5120"]["seed"]
    qT, sfT, g, st = rht_quantize(wl["dY"], rht_seed=seed + 1, mode=nv.SR, sr_seed=seed)
    rqT, rsfT, rg = O.rht_quantize(wl["dY"], seed + 1, O.SR, seed)
    assert st == 0 and g == rg
    _assert_same(qT, rqT, "codes")
    _assert_same(sfT, rsfT, "scales")


def test_quantize_dual_full_size_activation():
    """The MLP input X [8192, 4096] (outlier channels): forward RN row form
    and the Hadamard SR form, as the MLP step quantizes it."""
    wl = synth.make_workload("mlp7b_fwd_bwd_h4096_f11008_t8192", only={"X"})
    x = wl["X"]
    q, sf, g, qT, sfT, gT, st = quantize_dual(x, nv.RN, 0, 17, nv.SR, 18)
    rq, rsf, rg = O.quantize(x, O.RN, 0)
    rqT, rsfT, rgT = O.rht_quantize(x, 17, O.SR, 18)
    assert st == 0 and g == rg and gT == rgT
    _assert_same(q, rq, "row codes")
    _assert_same(sf, rsf, "row scales")
    _assert_same(qT, rqT, "transformed codes")
    _assert_same(sfT, rsfT, "transformed scales")


# ------------------------------------------- degenerate inputs, every form ----

def test_rht_dual_2d_on_zero_and_tiny_tensors():
    """amax = 0 gives g = 0, zero scales and sign-only codes in every form; a
    subnormal-range tensor saturates s_enc like the oracle does."""
    z = synth.f32_to_bf16_bits(np.array([[0.0, -0.0] * 24] * 32, np.float32))  # 32 x 48
    qT, sfT, g, st = rht_quantize(z, 3, nv.SR, 1)
    rqT, rsfT, rg = O.rht_quantize(z, 3, O.SR, 1)
    assert st == 0 and g == 0.0 == rg
    _assert_same(qT, rqT, "rht codes")
    _assert_same(sfT, rsfT, "rht scales")
    q, sf, g, qT, sfT, gT, st = quantize_dual(z, nv.SR, 2, 3, nv.SR, 4)
    assert st == 0 and g == 0.0 and gT == 0.0
    _assert_same(q, O.quantize(z, O.SR, 2)[0], "dual row codes")
    _assert_same(qT, O.rht_quantize(z, 3, O.SR, 4)[0], "dual rht codes")
    q, sf, qT, sfT, g, st = quantize_2d(z)
    assert st == 0 and g == 0.0 and not sf.any() and not sfT.any()
    tiny = np.zeros((32, 48), np.float32)
    tiny[3, 5], tiny[17, 40], tiny[30, 0] = 2.0 ** -130, -2.0 ** -126, 2.0 ** -133
    tb = synth.f32_to_bf16_bits(tiny)
    q, sf, g, qT, sfT, gT, st = quantize_dual(tb, nv.RN, 0, 5, nv.SR, 6)
    rq, rsf, rg = O.quantize(tb, O.RN, 0)
    rqT, rsfT, rgT = O.rht_quantize(tb, 5, O.SR, 6)
    assert st == 0 and g == rg and gT == rgT
    _assert_same(q, rq, "tiny row codes")
    _assert_same(qT, rqT, "tiny rht codes")
    _assert_same(sfT, rsfT, "tiny rht scales")


def test_nonfinite_input_is_reported_by_every_form():
    x = synth.normal_bf16((64, 128), 4, 0)
    x[9, 70] = 0x7F80  # +inf
    assert rht_quantize(x, 1, nv.SR, 2)[3] == 4
    assert quantize_dual(x, nv.RN, 0, 1, nv.SR, 2)[6] == 4
    assert quantize_2d(x)[5] == 4
    # finite input whose Hadamard sums overflow binary32: the transformed amax
    # is not finite, which the Hadamard forms report
    big = np.full((16, 16), 3.0e38, np.float32)
    bb = synth.f32_to_bf16_bits(big)
    assert rht_quantize(bb, 0, nv.RN, 0)[3] == 4
    with pytest.raises(O.OracleError):
        O.rht_quantize(bb, 0, O.RN, 0)


def test_grid_barrier_time_limit_is_reported():
    """The grid barrier counts CTA arrivals in word 2 of the workspace, from 0
    up to the grid size.  Started at 2^32 - 1 the count wraps to one below the
    grid size, so the barrier can only end by its 2 s time limit: the kernel
    must finish, report NVFP4_ERR_TIMEOUT, and the workspace must work again
    after nvfp4_workspace_init.  Nothing faults or hangs."""
    import torch
    x = synth.normal_bf16((512, 256), 61, 0)
    ws = nv.alloc_workspace()
    ws.view(torch.int32)[2] = -1
    _, _, _, st = quantize(x, nv.RN, 0, ws=ws)
    assert st == 5, nv.nvfp4_status_str(st)
    nv.nvfp4_workspace_init(ws)
    q, sf, g, st = quantize(x, nv.RN, 0, ws=ws)
    rq, rsf, rg = O.quantize(x, O.RN, 0)
    assert st == 0 and g == rg
    _assert_same(q, rq, "codes after recovery")
    _assert_same(sf, rsf, "scales after recovery")


def _edge_value_tensor(rows, cols, seed):
    """Blocks of the method's edge cases, tiled over the tensor: all-equal
    blocks of both signs, one outlier among zeros, one outlier among tiny
    values, alternating +-amax, bf16 subnormals, values at the E2M1 grid
    points of their block scale, and plain N(0, 1)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    blocks = x.reshape(rows, cols // 16, 16)
    kinds = rng.integers(0, 7, (rows, cols // 16))
    for r in range(rows):
        for b in range(cols // 16):
            k = kinds[r, b]
            v = blocks[r, b]
            if k == 0:
                v[:] = rng.choice([-1, 1]) * rng.uniform(0.1, 100)
            elif k == 1:
                v[:] = 0.0
                v[rng.integers(16)] = rng.choice([-1, 1]) * rng.uniform(1, 1000)
            elif k == 2:
                v[:] = rng.uniform(-1e-6, 1e-6, 16)
                v[rng.integers(16)] = 50.0
            elif k == 3:
                v[:] = np.where(np.arange(16) % 2 == 0, 3.0, -3.0)
            elif k == 4:
                v[:] = rng.uniform(-1, 1, 16) * 2.0 ** -130
            elif k == 5:
                v[:] = rng.choice([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], 16) * rng.choice([-1, 1], 16) * 0.25
    return synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("mode", [nv.RN, nv.SR])
def test_edge_value_blocks_every_form(mode):
    x = _edge_value_tensor(256, 384, 71)
    q, sf, g, st = quantize(x, mode, seed=9)
    rq, rsf, rg = O.quantize(x, mode, 9)
    assert st == 0 and g == rg
    _assert_same(q, rq, "1x16 codes")
    _assert_same(sf, rsf, "1x16 scales")
    qT, sfT, gT, st = rht_quantize(x, 4, mode, 10)
    rqT, rsfT, rgT = O.rht_quantize(x, 4, mode, 10)
    assert st == 0 and gT == rgT
    _assert_same(qT, rqT, "rht codes")
    _assert_same(sfT, rsfT, "rht scales")
    q, sf, g, qT, sfT, gT, st = quantize_dual(x, mode, 9, 4, mode, 10)
    assert st == 0 and g == rg and gT == rgT
    _assert_same(q, rq, "dual row codes")
    _assert_same(qT, rqT, "dual rht codes")
    if mode == nv.RN:
        q, sf, qT2, sfT2, g, st = quantize_2d(x)
        rq2, rsf2, rqT2, rsfT2, rg2 = O.quantize_2d(x)
        assert st == 0 and g == rg2
        _assert_same(q, rq2, "2-D codes")
        _assert_same(sf, rsf2, "2-D scales")
        _assert_same(qT2, rqT2, "2-D transposed codes")
        _assert_same(sfT2, rsfT2, "2-D transposed scales")
