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


def gemm(qa, sfa, ga, qb, sfb, gb, M, N, K, out_f32=False, ws=None):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    d = torch.empty((M, N), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    gat = torch.tensor([ga], dtype=torch.float32, device="cuda")
    gbt = torch.tensor([gb], dtype=torch.float32, device="cuda")
    ws = nv.alloc_workspace() if ws is None else ws
    nv.nvfp4_gemm(t(qa), t(sfa), gat, t(qb), t(sfb), gbt, M, N, K, d, N,
                  nv.OUT_F32 if out_f32 else nv.OUT_BF16, ws)
    st = nv.nvfp4_device_status(ws)
    return d.float().cpu().numpy().astype(np.float64), st
