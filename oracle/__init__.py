"""NVFP4 oracle — TEST INFRASTRUCTURE ONLY.

A ctypes view of ``nvfp4_oracle.c``: a plain, slow, single-threaded CPU
restatement of the NVFP4 quantizers and the block-scaled matmul, written from
the pages' definition of the format (E2M1 elements, one E4M3 scale per 16
contiguous elements, a tensor-level scale, 2-D weight blocks, random Hadamard
transform, stochastic rounding).  Only the tests, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The library
path never does, and this package imports nothing from the library.

Parity status: every function is pinned by ``tests/test_oracle_pins.py``,
including the Philox generator's exact bit stream (the known-answer vectors
published with the method).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "libnvfp4_oracle.so")

# Plain IEEE binary32 semantics: no contraction into FMA, no fast-math.
CFLAGS = ["-O1", "-ffp-contract=off", "-fno-fast-math", "-fno-strict-aliasing",
          "-std=c11", "-fPIC", "-shared"]

OK, ERR_SHAPE, ERR_NONFINITE = 0, 2, 4
RN, SR = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no SIMD intrinsics, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        u64 = ctypes.c_uint64
        L.or_e2m1_value.argtypes = [ctypes.c_int]
        L.or_e2m1_value.restype = ctypes.c_float
        L.or_e2m1_rn.argtypes = [ctypes.c_float]
        L.or_e2m1_rn.restype = ctypes.c_int
        L.or_e2m1_sr.argtypes = [ctypes.c_float, ctypes.c_uint]
        L.or_e2m1_sr.restype = ctypes.c_int
        L.or_e4m3_value.argtypes = [ctypes.c_int]
        L.or_e4m3_value.restype = ctypes.c_float
        L.or_e4m3_rn_sat.argtypes = [ctypes.c_float]
        L.or_e4m3_rn_sat.restype = ctypes.c_int
        L.or_philox4x32_10.argtypes = [p, p, p]
        L.or_philox4x32_10.restype = None
        L.or_rht_signs.argtypes = [u64]
        L.or_rht_signs.restype = ctypes.c_uint32
        L.or_rht16.argtypes = [p, ctypes.c_uint32, p]
        L.or_rht16.restype = None
        L.or_sf_bytes.argtypes = [i64, i64]
        L.or_sf_bytes.restype = ctypes.c_size_t
        L.or_sf_offset.argtypes = [i64, i64, i64]
        L.or_sf_offset.restype = ctypes.c_size_t
        L.or_amax.argtypes = [p, i64, i64, i64, p]
        L.or_amax.restype = ctypes.c_int
        L.or_rht_amax.argtypes = [p, i64, i64, i64, u64, p]
        L.or_rht_amax.restype = ctypes.c_int
        L.or_quantize.argtypes = [p, i64, i64, i64, ctypes.c_int, u64, p, p, p]
        L.or_quantize.restype = ctypes.c_int
        L.or_quantize_2d.argtypes = [p, i64, i64, i64, p, p, p, p, p]
        L.or_quantize_2d.restype = ctypes.c_int
        L.or_rht_quantize.argtypes = [p, i64, i64, i64, u64, ctypes.c_int, u64, p, p, p]
        L.or_rht_quantize.restype = ctypes.c_int
        L.or_dequantize.argtypes = [p, p, ctypes.c_float, i64, i64, p]
        L.or_dequantize.restype = None
        L.or_gemm_f64.argtypes = [p, p, ctypes.c_float, p, p, ctypes.c_float, i64, i64, i64, p, p]
        L.or_gemm_f64.restype = None
        L.or_gemm_f64_sampled.argtypes = [p, p, ctypes.c_float, p, p, ctypes.c_float,
                                          i64, i64, i64, p, p, i64, p, p]
        L.or_gemm_f64_sampled.restype = None
        L.or_quant_noise.argtypes = [p, i64, i64, i64, p, p, ctypes.c_float, p]
        L.or_quant_noise.restype = None
        L.or_e8m0_value.argtypes = [ctypes.c_int]
        L.or_e8m0_value.restype = ctypes.c_double
        L.or_mx_sf_offset.argtypes = [i64, i64, i64]
        L.or_mx_sf_offset.restype = ctypes.c_size_t
        L.or_mx_quantize.argtypes = [p, i64, i64, i64, p, p]
        L.or_mx_quantize.restype = ctypes.c_int
        L.or_mx_dequantize.argtypes = [p, p, i64, i64, p]
        L.or_mx_dequantize.restype = None
        L.or_mx_gemm_f64_sampled.argtypes = [p, p, p, p, i64, p, p, i64, p, p]
        L.or_mx_gemm_f64_sampled.restype = None
        L.or_e2m1_rn_many.argtypes = [p, i64, p]
        L.or_e2m1_sr_many.argtypes = [p, p, i64, p]
        L.or_sr_values.argtypes = [u64, u64, p]
        L.or_sr_values.restype = None
        L.or_e4m3_rn_sat_many.argtypes = [p, i64, p]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"oracle status {status}")
        self.status = status


# ---------------------------------------------------------------- codecs ----

def e2m1_value(code: int) -> float:
    return lib().or_e2m1_value(int(code))


def e2m1_rn(v: float) -> int:
    return lib().or_e2m1_rn(float(v))


def e2m1_sr(v: float, R: int) -> int:
    """Stochastic rounding of v with the 16-bit random value R."""
    return lib().or_e2m1_sr(float(v), int(R))


def e4m3_value(code: int) -> float:
    return lib().or_e4m3_value(int(code))


def e4m3_rn_sat(x: float) -> int:
    return lib().or_e4m3_rn_sat(float(x))


def e2m1_rn_many(v: np.ndarray) -> np.ndarray:
    v = _c(v, np.float32)
    out = np.empty(v.size, np.uint8)
    lib().or_e2m1_rn_many(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_sr_many(v: np.ndarray, R: np.ndarray) -> np.ndarray:
    v = _c(v, np.float32)
    r = _c(R, np.uint16)
    out = np.empty(v.size, np.uint8)
    lib().or_e2m1_sr_many(_ptr(v), _ptr(r), v.size, _ptr(out))
    return out


def e4m3_rn_sat_many(v: np.ndarray) -> np.ndarray:
    v = _c(v, np.float32)
    out = np.empty(v.size, np.uint8)
    lib().or_e4m3_rn_sat_many(_ptr(v), v.size, _ptr(out))
    return out


def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.empty(4, np.uint32)
    lib().or_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_values(seed: int, blk: int) -> np.ndarray:
    """The 16-bit random values of the 16 elements of output block blk."""
    out = np.empty(16, np.uint32)
    lib().or_sr_values(seed, blk, _ptr(out))
    return out


def rht_signs(seed: int) -> int:
    return int(lib().or_rht_signs(seed))


def rht16(v, sign_bits: int) -> np.ndarray:
    v = _c(v, np.float32)
    assert v.size == 16
    y = np.empty(16, np.float32)
    lib().or_rht16(_ptr(v), int(sign_bits), _ptr(y))
    return y


def sf_bytes(rows: int, cols: int) -> int:
    return int(lib().or_sf_bytes(rows, cols))


def sf_offset(r: int, kb: int, kblocks: int) -> int:
    return int(lib().or_sf_offset(r, kb, kblocks))


def unswizzle_sf(sf: np.ndarray, rows: int, kblocks: int) -> np.ndarray:
    """Linear [rows, kblocks] view of a swizzled scale buffer (via sf_offset)."""
    out = np.empty((rows, kblocks), np.uint8)
    for r in range(rows):
        for kb in range(kblocks):
            out[r, kb] = sf[sf_offset(r, kb, kblocks)]
    return out


# ------------------------------------------------------------ quantizers ----

def amax(x_bf16: np.ndarray) -> float:
    """max |x| over a bf16 matrix (uint16 bits): the tensor amax."""
    x = _c(x_bf16, np.uint16)
    R, C = x.shape
    out = np.zeros(1, np.float32)
    st = lib().or_amax(_ptr(x), R, C, C, _ptr(out))
    if st != OK:
        raise OracleError(st)
    return float(out[0])


def rht_amax(x_bf16: np.ndarray, rht_seed: int) -> float:
    """max |y| over the 16-token Hadamard transforms of every channel of x [T, C]."""
    x = _c(x_bf16, np.uint16)
    T, C = x.shape
    out = np.zeros(1, np.float32)
    st = lib().or_rht_amax(_ptr(x), T, C, C, rht_seed, _ptr(out))
    if st != OK:
        raise OracleError(st)
    return float(out[0])


def quantize(x_bf16: np.ndarray, mode: int = RN, seed: int = 0):
    """1x16 quantization of a row-major bf16 matrix (given as uint16 bits)."""
    x = _c(x_bf16, np.uint16)
    R, C = x.shape
    q = np.empty((R, C // 2), np.uint8)
    sf = np.empty(sf_bytes(R, C), np.uint8)
    g = np.zeros(1, np.float32)
    st = lib().or_quantize(_ptr(x), R, C, C, mode, seed, _ptr(q), _ptr(sf), _ptr(g))
    if st != OK:
        raise OracleError(st)
    return q, sf, float(g[0])


def quantize_2d(w_bf16: np.ndarray, transpose: bool = True):
    w = _c(w_bf16, np.uint16)
    R, C = w.shape
    q = np.empty((R, C // 2), np.uint8)
    sf = np.empty(sf_bytes(R, C), np.uint8)
    qT = np.empty((C, R // 2), np.uint8) if transpose else None
    sfT = np.empty(sf_bytes(C, R), np.uint8) if transpose else None
    g = np.zeros(1, np.float32)
    st = lib().or_quantize_2d(_ptr(w), R, C, C, _ptr(q), _ptr(sf),
                              _ptr(qT) if transpose else None,
                              _ptr(sfT) if transpose else None, _ptr(g))
    if st != OK:
        raise OracleError(st)
    return q, sf, qT, sfT, float(g[0])


def rht_quantize(x_bf16: np.ndarray, rht_seed: int, mode: int = SR, sr_seed: int = 0):
    x = _c(x_bf16, np.uint16)
    T, C = x.shape
    qT = np.empty((C, T // 2), np.uint8)
    sfT = np.empty(sf_bytes(C, T), np.uint8)
    g = np.zeros(1, np.float32)
    st = lib().or_rht_quantize(_ptr(x), T, C, C, rht_seed, mode, sr_seed, _ptr(qT), _ptr(sfT), _ptr(g))
    if st != OK:
        raise OracleError(st)
    return qT, sfT, float(g[0])


def dequantize(q: np.ndarray, sf: np.ndarray, g: float, rows: int, cols: int) -> np.ndarray:
    q = _c(q, np.uint8)
    sf = _c(sf, np.uint8)
    out = np.empty((rows, cols), np.float64)
    lib().or_dequantize(_ptr(q), _ptr(sf), g, rows, cols, _ptr(out))
    return out


def gemm_f64(a, sfa, ga, b, sfb, gb, M, N, K):
    """D = gA gB sum_k deqA[m,k] deqB[n,k] in binary64, plus the |.| sum."""
    a, sfa, b, sfb = (_c(t, np.uint8) for t in (a, sfa, b, sfb))
    d = np.empty((M, N), np.float64)
    dabs = np.empty((M, N), np.float64)
    lib().or_gemm_f64(_ptr(a), _ptr(sfa), ga, _ptr(b), _ptr(sfb), gb, M, N, K, _ptr(d), _ptr(dabs))
    return d, dabs


def gemm_f64_sampled(a, sfa, ga, b, sfb, gb, M, N, K, ms, ns):
    a, sfa, b, sfb = (_c(t, np.uint8) for t in (a, sfa, b, sfb))
    ms = _c(ms, np.int64)
    ns = _c(ns, np.int64)
    d = np.empty(ms.size, np.float64)
    dabs = np.empty(ms.size, np.float64)
    lib().or_gemm_f64_sampled(_ptr(a), _ptr(sfa), ga, _ptr(b), _ptr(sfb), gb, M, N, K,
                              _ptr(ms), _ptr(ns), ms.size, _ptr(d), _ptr(dabs))
    return d, dabs


def quant_noise(x_bf16: np.ndarray, q: np.ndarray, sf: np.ndarray, g: float):
    """(sum (Q(x) - x)^2, sum x^2) in binary64 for the 1x16 form (q, sf, g) of x."""
    x = _c(x_bf16, np.uint16)
    R, C = x.shape
    q, sf = _c(q, np.uint8), _c(sf, np.uint8)
    out = np.zeros(2, np.float64)
    lib().or_quant_noise(_ptr(x), R, C, C, _ptr(q), _ptr(sf), g, _ptr(out))
    return float(out[0]), float(out[1])


# ----------------------------------------------------------------- MXFP4 ----

def e8m0_value(code: int) -> float:
    return float(lib().or_e8m0_value(int(code)))


def mx_sf_offset(r: int, kb: int, kblocks: int) -> int:
    return int(lib().or_mx_sf_offset(r, kb, kblocks))


def mx_quantize(x_bf16: np.ndarray):
    """MXFP4 (OCP MX v1.0) of a row-major bf16 matrix: (codes, scale bytes)."""
    x = _c(x_bf16, np.uint16)
    R, C = x.shape
    q = np.empty((R, C // 2), np.uint8)
    sf = np.empty(sf_bytes(R, C), np.uint8)
    st = lib().or_mx_quantize(_ptr(x), R, C, C, _ptr(q), _ptr(sf))
    if st != OK:
        raise OracleError(st)
    return q, sf


def mx_dequantize(q: np.ndarray, sf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    q, sf = _c(q, np.uint8), _c(sf, np.uint8)
    out = np.empty((rows, cols), np.float64)
    lib().or_mx_dequantize(_ptr(q), _ptr(sf), rows, cols, _ptr(out))
    return out


def mx_gemm_f64_sampled(a, sfa, b, sfb, K, ms, ns):
    a, sfa, b, sfb = (_c(t, np.uint8) for t in (a, sfa, b, sfb))
    ms = _c(ms, np.int64)
    ns = _c(ns, np.int64)
    d = np.empty(ms.size, np.float64)
    dabs = np.empty(ms.size, np.float64)
    lib().or_mx_gemm_f64_sampled(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), K, _ptr(ms), _ptr(ns), ms.size,
                                 _ptr(d), _ptr(dabs))
    return d, dabs


def mx_gemm_f64(a, sfa, b, sfb, M, N, K):
    """Full D = A B^T of two MXFP4 operands (binary64), with the |.| sums."""
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    d, dabs = mx_gemm_f64_sampled(a, sfa, b, sfb, K, mm.ravel(), nn.ravel())
    return d.reshape(M, N), dabs.reshape(M, N)
