"""NVFP4 quantize + block-scaled GEMM for GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libnvfp4_gb300.so`` (C ABI in ``include/nvfp4.h``).
Each function has the name of the C entry point it calls and only marshals
arguments: torch tensors become device pointers, ``stream=None`` becomes
torch's current stream, a non-OK status raises ``NVFP4Error``.  All compute
runs in the library's CUDA kernels; there is no other implementation here and
no fallback — calling any entry point without the built library raises.

The ``alloc_*`` helpers only allocate output tensors of the right size.
"""
from __future__ import annotations

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libnvfp4_gb300.so")

RN, SR = 0, 1
OUT_BF16, OUT_F32 = 0, 1

STATUS = {0: "OK", 1: "ERR_ARG", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_NONFINITE",
          5: "ERR_TIMEOUT", 6: "ERR_CUDA", 7: "ERR_UNSUPPORTED"}

EXPORTS = ["nvfp4_sf_bytes", "nvfp4_workspace_bytes", "nvfp4_workspace_init", "nvfp4_quantize",
           "nvfp4_quantize_2d", "nvfp4_rht_quantize", "nvfp4_quantize_dual", "nvfp4_quant_noise", "nvfp4_gemm",
           "nvfp4_mxfp4_quantize", "nvfp4_mxfp4_gemm", "nvfp4_device_status", "nvfp4_status_str",
           "nvfp4_encode_probe", "nvfp4_quantize_noalloc", "nvfp4_gemm_amax", "nvfp4_quantize_dual_from_amax"]


class NVFP4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS.get(status, status)}")
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Load the built library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                           "(python -m nvfp4_bit_quantized_quantize_gb300.build)")
    L = ctypes.CDLL(LIB_PATH)
    p, i64, u64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
    sig = {
        "nvfp4_sf_bytes": ([i64, i64], ctypes.c_size_t),
        "nvfp4_workspace_bytes": ([i64, i64], ctypes.c_size_t),
        "nvfp4_workspace_init": ([p, p], i32),
        "nvfp4_quantize": ([p, i64, i64, i64, i32, u64, p, p, p, p, p], i32),
        "nvfp4_quantize_2d": ([p, i64, i64, i64, p, p, p, p, p, p, p], i32),
        "nvfp4_rht_quantize": ([p, i64, i64, i64, u64, i32, u64, p, p, p, p, p], i32),
        "nvfp4_quantize_dual": ([p, i64, i64, i64, i32, u64, p, p, p, u64, i32, u64, p, p, p, p, p], i32),
        "nvfp4_quant_noise": ([p, i64, i64, i64, p, p, p, p, p], i32),
        "nvfp4_gemm": ([p, p, p, p, p, p, i64, i64, i64, p, i64, i32, p, p], i32),
        "nvfp4_mxfp4_quantize": ([p, i64, i64, i64, p, p, p, p], i32),
        "nvfp4_mxfp4_gemm": ([p, p, p, p, i64, i64, i64, p, i64, i32, p, p], i32),
        "nvfp4_device_status": ([p, p], i32),
        "nvfp4_status_str": ([i32], ctypes.c_char_p),
        "nvfp4_encode_probe": ([p, p, i64, p, p, p, p], i32),
        "nvfp4_quantize_noalloc": ([p, i64, i64, i64, i32, u64, p, p, p, p], i32),
        "nvfp4_gemm_amax": ([p, p, p, p, p, p, i64, i64, i64, p, i64, u64, p, p, p], i32),
        "nvfp4_quantize_dual_from_amax": ([p, i64, i64, i64, p, i32, u64, p, p, p, u64, i32, u64, p, p, p, p, p],
                                          i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn: str, st: int):
    if st != 0:
        raise NVFP4Error(fn, st)


# ------------------------------------------------------------ entry points ----

def nvfp4_sf_bytes(rows: int, cols: int) -> int:
    return int(load().nvfp4_sf_bytes(rows, cols))


def nvfp4_workspace_bytes(rows: int = 0, cols: int = 0) -> int:
    return int(load().nvfp4_workspace_bytes(rows, cols))


def nvfp4_workspace_init(ws, stream=None) -> None:
    _check("nvfp4_workspace_init", load().nvfp4_workspace_init(_ptr(ws), _stream(stream)))


def nvfp4_quantize(x, rows, cols, ld, mode, sr_seed, q, sf, g_dec, ws, stream=None) -> None:
    _check("nvfp4_quantize", load().nvfp4_quantize(
        _ptr(x), rows, cols, ld, mode, sr_seed, _ptr(q), _ptr(sf), _ptr(g_dec), _ptr(ws), _stream(stream)))


def nvfp4_quantize_2d(w, rows, cols, ld, q, sf, qT, sfT, g_dec, ws, stream=None) -> None:
    _check("nvfp4_quantize_2d", load().nvfp4_quantize_2d(
        _ptr(w), rows, cols, ld, _ptr(q), _ptr(sf), _ptr(qT), _ptr(sfT), _ptr(g_dec), _ptr(ws),
        _stream(stream)))


def nvfp4_rht_quantize(x, T, C, ld, rht_seed, mode, sr_seed, qT, sfT, g_dec, ws, stream=None) -> None:
    _check("nvfp4_rht_quantize", load().nvfp4_rht_quantize(
        _ptr(x), T, C, ld, rht_seed, mode, sr_seed, _ptr(qT), _ptr(sfT), _ptr(g_dec), _ptr(ws),
        _stream(stream)))


def nvfp4_mxfp4_quantize(x, rows, cols, ld, q, sf, ws, stream=None) -> None:
    _check("nvfp4_mxfp4_quantize", load().nvfp4_mxfp4_quantize(
        _ptr(x), rows, cols, ld, _ptr(q), _ptr(sf), _ptr(ws), _stream(stream)))


def nvfp4_mxfp4_gemm(a, sfa, b, sfb, M, N, K, d, ldd, out_dtype, ws, stream=None) -> None:
    _check("nvfp4_mxfp4_gemm", load().nvfp4_mxfp4_gemm(
        _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), M, N, K, _ptr(d), ldd, out_dtype, _ptr(ws), _stream(stream)))


def nvfp4_quant_noise(x, rows, cols, ld, q, sf, g_dec, sums, stream=None) -> None:
    _check("nvfp4_quant_noise", load().nvfp4_quant_noise(
        _ptr(x), rows, cols, ld, _ptr(q), _ptr(sf), _ptr(g_dec), _ptr(sums), _stream(stream)))


def nvfp4_quantize_dual(x, T, C, ld, mode, sr_seed, q, sf, g_dec, rht_seed, mode_t, sr_seed_t,
                        qT, sfT, g_dec_t, ws, stream=None) -> None:
    _check("nvfp4_quantize_dual", load().nvfp4_quantize_dual(
        _ptr(x), T, C, ld, mode, sr_seed, _ptr(q), _ptr(sf), _ptr(g_dec), rht_seed, mode_t, sr_seed_t,
        _ptr(qT), _ptr(sfT), _ptr(g_dec_t), _ptr(ws), _stream(stream)))


def nvfp4_quantize_dual_from_amax(x, T, C, ld, amax, mode, sr_seed, q, sf, g_dec, rht_seed, mode_t, sr_seed_t,
                                  qT, sfT, g_dec_t, ws, stream=None) -> None:
    _check("nvfp4_quantize_dual_from_amax", load().nvfp4_quantize_dual_from_amax(
        _ptr(x), T, C, ld, _ptr(amax), mode, sr_seed, _ptr(q), _ptr(sf), _ptr(g_dec), rht_seed, mode_t,
        sr_seed_t, _ptr(qT), _ptr(sfT), _ptr(g_dec_t), _ptr(ws), _stream(stream)))


def nvfp4_gemm_amax(a, sfa, ga, b, sfb, gb, M, N, K, d, ldd, rht_seed, amax, ws, stream=None) -> None:
    _check("nvfp4_gemm_amax", load().nvfp4_gemm_amax(
        _ptr(a), _ptr(sfa), _ptr(ga), _ptr(b), _ptr(sfb), _ptr(gb), M, N, K, _ptr(d), ldd, rht_seed,
        _ptr(amax), _ptr(ws), _stream(stream)))


def nvfp4_gemm(a, sfa, ga, b, sfb, gb, M, N, K, d, ldd, out_dtype, ws, stream=None) -> None:
    _check("nvfp4_gemm", load().nvfp4_gemm(
        _ptr(a), _ptr(sfa), _ptr(ga), _ptr(b), _ptr(sfb), _ptr(gb), M, N, K, _ptr(d), ldd, out_dtype,
        _ptr(ws), _stream(stream)))


def nvfp4_device_status(ws, stream=None) -> int:
    return int(load().nvfp4_device_status(_ptr(ws), _stream(stream)))


def nvfp4_status_str(status: int) -> str:
    return load().nvfp4_status_str(status).decode()


def nvfp4_encode_probe(v, r, n, e4m3_out, e2m1_rn_out, e2m1_sr_out, stream=None) -> None:
    _check("nvfp4_encode_probe", load().nvfp4_encode_probe(
        _ptr(v), _ptr(r), n, _ptr(e4m3_out), _ptr(e2m1_rn_out), _ptr(e2m1_sr_out), _stream(stream)))


def nvfp4_quantize_noalloc(x, rows, cols, ld, mode, sr_seed, q, sf, g_dec, stream=None) -> None:
    """nvfp4_quantize without a workspace, for callers that cannot allocate
    device memory: the library keeps the scratch in a static device array."""
    _check("nvfp4_quantize_noalloc", load().nvfp4_quantize_noalloc(
        _ptr(x), rows, cols, ld, mode, sr_seed, _ptr(q), _ptr(sf), _ptr(g_dec), _stream(stream)))


# ------------------------------------------------------- output allocation ----

def alloc_workspace(device="cuda", stream=None):
    """Allocate and zero one workspace (torch allocation + nvfp4_workspace_init)."""
    import torch
    ws = torch.empty(nvfp4_workspace_bytes(), dtype=torch.uint8, device=device)
    nvfp4_workspace_init(ws, stream)
    return ws


def alloc_quantized(rows: int, cols: int, device="cuda"):
    """(codes [rows, cols/2] uint8, scales nvfp4_sf_bytes uint8, g_dec float32[1])."""
    import torch
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
    sf = torch.empty(nvfp4_sf_bytes(rows, cols), dtype=torch.uint8, device=device)
    g = torch.empty(1, dtype=torch.float32, device=device)
    return q, sf, g
