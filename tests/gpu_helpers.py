"""Run the CUDA path through the C ABI on numpy inputs (used by -m gpu tests)."""
from __future__ import annotations

import numpy as np
import torch

import nvfp4_bit_quantized_quantize_gb300 as nv


def dev_bf16(x_bits: np.ndarray, ld: int | None = None) -> torch.Tensor:
    """Upload uint16 bf16 bits; with ld > cols the rows are padded."""
    rows, cols = x_bits.shape
    ld = cols if ld is None else ld
    buf = torch.zeros((rows, ld), dtype=torch.int16)
    buf[:, :cols] = torch.from_numpy(x_bits.view(np.int16))
    return buf.cuda().view(torch.bfloat16)


def quantize(x_bits, mode=nv.RN, seed=0, ld=None, ws=None):
    rows, cols = x_bits.shape
    x = dev_bf16(x_bits, ld)
    q, sf, g = nv.alloc_quantized(rows, cols)
    q.fill_(0xEE)
    sf.fill_(0xEE)
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_quantize(x, rows, cols, x.shape[1], mode, seed, q, sf, g, ws)
    st = nv.nvfp4_device_status(ws)
    return q.cpu().numpy(), sf.cpu().numpy(), float(g.cpu()[0]), st


def quantize_2d(w_bits, transpose=True, ld=None, ws=None):
    rows, cols = w_bits.shape
    w = dev_bf16(w_bits, ld)
    q, sf, g = nv.alloc_quantized(rows, cols)
    q.fill_(0xEE)
    sf.fill_(0xEE)
    qT = sfT = None
    if transpose:
        qT, sfT, _ = nv.alloc_quantized(cols, rows)
        qT.fill_(0xEE)
        sfT.fill_(0xEE)
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_quantize_2d(w, rows, cols, w.shape[1], q, sf, qT, sfT, g, ws)
    st = nv.nvfp4_device_status(ws)
    out = [q.cpu().numpy(), sf.cpu().numpy(), None, None, float(g.cpu()[0]), st]
    if transpose:
        out[2] = qT.cpu().numpy()
        out[3] = sfT.cpu().numpy()
    return tuple(out)


def rht_quantize(x_bits, rht_seed, mode=nv.SR, sr_seed=0, ld=None, ws=None):
    T, C = x_bits.shape
    x = dev_bf16(x_bits, ld)
    qT, sfT, g = nv.alloc_quantized(C, T)
    qT.fill_(0xEE)
    sfT.fill_(0xEE)
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_rht_quantize(x, T, C, x.shape[1], rht_seed, mode, sr_seed, qT, sfT, g, ws)
    st = nv.nvfp4_device_status(ws)
    return qT.cpu().numpy(), sfT.cpu().numpy(), float(g.cpu()[0]), st


def quantize_dual(x_bits, mode, sr_seed, rht_seed, mode_t, sr_seed_t, ld=None, ws=None):
    T, C = x_bits.shape
    x = dev_bf16(x_bits, ld)
    q, sf, g = nv.alloc_quantized(T, C)
    qT, sfT, gT = nv.alloc_quantized(C, T)
    for t in (q, sf, qT, sfT):
        t.fill_(0xEE)
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_quantize_dual(x, T, C, x.shape[1], mode, sr_seed, q, sf, g, rht_seed, mode_t, sr_seed_t,
                           qT, sfT, gT, ws)
    st = nv.nvfp4_device_status(ws)
    return (q.cpu().numpy(), sf.cpu().numpy(), float(g.cpu()[0]),
            qT.cpu().numpy(), sfT.cpu().numpy(), float(gT.cpu()[0]), st)


def gemm(qa, sfa, ga, qb, sfb, gb, M, N, K, out_f32=False, ws=None, ldd=None):
    """Run the GEMM; the output rows are padded to ldd (a multiple of 16 bytes),
    32 spare rows follow row M, all pre-filled with NaN, and the padding must
    come back untouched."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    unit = 4 if out_f32 else 8
    ldd = ((N + unit - 1) // unit) * unit if ldd is None else ldd
    # 32 spare rows below M: a write past row M would land there
    d = torch.full((M + 32, ldd), float("nan"), dtype=torch.float32 if out_f32 else torch.bfloat16,
                   device="cuda")
    gat = torch.tensor([ga], dtype=torch.float32, device="cuda")
    gbt = torch.tensor([gb], dtype=torch.float32, device="cuda")
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_gemm(t(qa), t(sfa), gat, t(qb), t(sfb), gbt, M, N, K, d, ldd,
                  nv.OUT_F32 if out_f32 else nv.OUT_BF16, ws)
    st = nv.nvfp4_device_status(ws)
    out = d.float().cpu().numpy().astype(np.float64)
    assert np.isnan(out[:M, N:]).all(), "GEMM wrote past column N"
    assert np.isnan(out[M:]).all(), "GEMM wrote past row M"
    return np.ascontiguousarray(out[:M, :N]), st


def quant_noise(x_bits, q, sf, g, ld=None):
    """The CUDA noise meter on host arrays: returns (sum (Q-x)^2, sum x^2)."""
    rows, cols = x_bits.shape
    x = dev_bf16(x_bits, ld)
    qt = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    sft = torch.from_numpy(np.ascontiguousarray(sf)).cuda()
    gt = torch.tensor([g], dtype=torch.float32, device="cuda")
    sums = torch.full((2,), float("nan"), dtype=torch.float64, device="cuda")
    nv.nvfp4_quant_noise(x, rows, cols, x.shape[1], qt, sft, gt, sums)
    torch.cuda.synchronize()
    s = sums.cpu().numpy()
    return float(s[0]), float(s[1])


def mx_quantize(x_bits, ld=None, ws=None):
    rows, cols = x_bits.shape
    x = dev_bf16(x_bits, ld)
    q = torch.full((rows, cols // 2), 0xEE, dtype=torch.uint8, device="cuda")
    sf = torch.full((nv.nvfp4_sf_bytes(rows, cols),), 0xEE, dtype=torch.uint8, device="cuda")
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_mxfp4_quantize(x, rows, cols, x.shape[1], q, sf, ws)
    st = nv.nvfp4_device_status(ws)
    return q.cpu().numpy(), sf.cpu().numpy(), st


def mx_gemm(qa, sfa, qb, sfb, M, N, K, out_f32=False, ws=None):
    """MXFP4 GEMM with the same NaN-filled, padded output check as gemm()."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    unit = 4 if out_f32 else 8
    ldd = ((N + unit - 1) // unit) * unit
    d = torch.full((M + 32, ldd), float("nan"), dtype=torch.float32 if out_f32 else torch.bfloat16,
                   device="cuda")
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_mxfp4_gemm(t(qa), t(sfa), t(qb), t(sfb), M, N, K, d, ldd, nv.OUT_F32 if out_f32 else nv.OUT_BF16, ws)
    st = nv.nvfp4_device_status(ws)
    out = d.float().cpu().numpy().astype(np.float64)
    assert np.isnan(out[:M, N:]).all(), "GEMM wrote past column N"
    assert np.isnan(out[M:]).all(), "GEMM wrote past row M"
    return np.ascontiguousarray(out[:M, :N]), st


def gemm_amax(qa, sfa, ga, qb, sfb, gb, M, N, K, rht_seed, ws=None):
    """nvfp4_gemm_amax into a NaN-filled, padded bf16 output (the padding must
    come back untouched).  Returns (D as bf16 bits [M, N], amax[2], status)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ldd = ((N + 7) // 8) * 8
    d = torch.full((M + 32, ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    gat = torch.tensor([ga], dtype=torch.float32, device="cuda")
    gbt = torch.tensor([gb], dtype=torch.float32, device="cuda")
    amax = torch.full((2,), float("nan"), dtype=torch.float32, device="cuda")
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_gemm_amax(t(qa), t(sfa), gat, t(qb), t(sfb), gbt, M, N, K, d, ldd, rht_seed, amax, ws)
    st = nv.nvfp4_device_status(ws)
    out = d.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all(out[:M, N:] == 0x7FC0), "GEMM wrote past column N"
    assert np.all(out[M:] == 0x7FC0), "GEMM wrote past row M"
    return np.ascontiguousarray(out[:M, :N]), amax.cpu().numpy(), st


def quantize_dual_from_amax(x_bits, amax, mode, sr_seed, rht_seed, mode_t, sr_seed_t, ld=None, ws=None):
    """nvfp4_quantize_dual_from_amax with the two maxima given as host floats."""
    T, C = x_bits.shape
    x = dev_bf16(x_bits, ld)
    q, sf, g = nv.alloc_quantized(T, C)
    qT, sfT, gT = nv.alloc_quantized(C, T)
    for t in (q, sf, qT, sfT):
        t.fill_(0xEE)
    am = torch.tensor(np.asarray(amax, np.float32), device="cuda")
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_quantize_dual_from_amax(x, T, C, x.shape[1], am, mode, sr_seed, q, sf, g, rht_seed, mode_t,
                                     sr_seed_t, qT, sfT, gT, ws)
    st = nv.nvfp4_device_status(ws)
    return (q.cpu().numpy(), sf.cpu().numpy(), float(g.cpu()[0]),
            qT.cpu().numpy(), sfT.cpu().numpy(), float(gT.cpu()[0]), st)
