/*
 * nvfp4.h — C ABI of the GB300 (sm_103a) NVFP4 quantize + block-scaled GEMM
 * library (libnvfp4_gb300.so).
 *
 * The format, as the pages define it:
 *  - every element is E2M1 (1 sign, 2 exponent, 1 mantissa bit), one of
 *    ±0, ±0.5, ±1, ±1.5, ±2, ±3, ±4, ±6
 *    ["Entrenamiento de Modelos de Lenguaje con 4 Bits de Precisión",
 *     section "Características del Formato NVFP4"];
 *  - each block of 16 contiguous elements shares one E4M3 scale
 *    [same section; "FP4 All the Way: Formación totalmente cuantificada de
 *     LLM", section "Describir"];
 *  - scaling is multi-level ["I ricercatori di Nvidia sbloccano ...",
 *    section "Come funziona NVFP4?"]: here a binary32 tensor scale over the
 *    block scales;
 *  - the training recipe adds 2-D block scaling for weights, random Hadamard
 *    transforms and stochastic rounding of gradients ["Entrenamiento ...",
 *    section "Metodología de Entrenamiento"]; round-to-nearest in the
 *    forward pass, stochastic rounding in backward and update ["FP4 All the
 *    Way", section "Describir"].
 *
 * Arithmetic (readings where the pages are silent):
 *  - amax = max |x| over the tensor (over the transformed values for the
 *    Hadamard variant); s_enc = 2688 / amax (binary32, saturated to FLT_MAX),
 *    g = amax / 2688 is the stored decode scale (0 when amax == 0);
 *  - block scale byte = E4M3(rn(rn(bamax / 6) * s_enc)), nearest-even,
 *    saturating at 448;
 *  - f = rn(s_enc / E4M3value(byte)); v = rn(x * f); E2M1 code by nearest-even
 *    (NVFP4_ROUND_RN) or stochastic rounding (NVFP4_ROUND_SR): rounded up iff
 *    the fraction between the grid neighbours, kept to 16 bits, plus a 16-bit
 *    random value carries; the block's 16 values come from the four words of
 *    Philox4x32-10 (key = seed, counter = (block index, 0, 0)), elements
 *    4m..4m+3 from word m with bytes b0..b3 as (b2 b0), (rev b0, rev b2),
 *    (b3 b1), (rev b1, rev b3), rev = bit reversal; |v| above 6 saturates;
 *    the sign bit is kept;
 *  - decoded value of element (r, c) = E2M1(code) * E4M3(scale(r, c/16)) * g.
 *
 * Layouts:
 *  - bf16 inputs are row-major with a leading dimension `ld` in elements;
 *  - codes are packed two per byte, element 2i in the low nibble, rows dense
 *    (row stride = cols / 2 bytes);
 *  - scale bytes use the 128 x 4 atom layout block-scaled tensor-core matmuls
 *    read: byte of (row r, block kb) at
 *      ((r / 128) * Cp + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4,
 *    Cp = ceil(kblocks / 4); rows are padded to 128 and blocks to 4, padding
 *    is written as 0 by the quantizers.  Size: nvfp4_sf_bytes(rows, cols).
 *
 * Conventions for every call:
 *  - all data pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing and keeps no state between calls;
 *  - calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream); argument, shape and alignment errors are returned
 *    before anything is launched;
 *  - `ws` is a caller-owned device workspace of nvfp4_workspace_bytes()
 *    bytes, zeroed once with nvfp4_workspace_init before first use; every
 *    call leaves it ready for the next call on the same stream.  Calls that
 *    may run concurrently need distinct workspaces.  Errors found on the
 *    device (non-finite input, a wait that ran out) are recorded in `ws`
 *    and read with nvfp4_device_status;
 *  - pointers must be 16-byte aligned and `ld` a multiple of 8 elements.
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_ARG = 1,         /* null pointer or bad enum value */
    NVFP4_ERR_SHAPE = 2,       /* shape outside what the call supports */
    NVFP4_ERR_ALIGN = 3,       /* pointer or leading dimension misaligned */
    NVFP4_ERR_NONFINITE = 4,   /* input holds Inf or NaN (device-detected) */
    NVFP4_ERR_TIMEOUT = 5,     /* a bounded device wait ran out (device-detected) */
    NVFP4_ERR_CUDA = 6,        /* a CUDA runtime or driver call failed */
    NVFP4_ERR_UNSUPPORTED = 7  /* device is not sm_103 (the library carries sm_103a code only) */
} nvfp4_status;

typedef enum { NVFP4_ROUND_RN = 0, NVFP4_ROUND_SR = 1 } nvfp4_round;
typedef enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_F32 = 1 } nvfp4_out_dtype;

typedef void* nvfp4_stream_t; /* cudaStream_t */

/* Bytes of the swizzled scale buffer for a rows x cols matrix (cols % 16 == 0). */
size_t nvfp4_sf_bytes(int64_t rows, int64_t cols);

/* Bytes of the device workspace (independent of the shapes given). */
size_t nvfp4_workspace_bytes(int64_t rows, int64_t cols);

/* Zero a workspace on `stream` (needed once, and after any device error). */
nvfp4_status nvfp4_workspace_init(void* ws, nvfp4_stream_t stream);

/*
 * 1x16 quantization along rows [16 contiguous elements share an E4M3 scale:
 * "Entrenamiento ...", "Características del Formato NVFP4"; RN forward / SR
 * backward: "FP4 All the Way", "Describir"].
 *   x      bf16 [rows, cols], leading dimension ld (elements); cols % 16 == 0
 *   mode   NVFP4_ROUND_RN or NVFP4_ROUND_SR; sr_seed keys the SR generator
 *          (block index = row * cols/16 + col/16)
 *   q      out: uint8 [rows, cols/2] packed codes
 *   sf     out: nvfp4_sf_bytes(rows, cols) swizzled scale bytes
 *   g_dec  out: one float, the tensor decode scale (device memory)
 * One fused kernel: per-tensor amax, grid-wide barrier, block scales, codes.
 */
nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld,
                            nvfp4_round mode, uint64_t sr_seed,
                            uint8_t* q, uint8_t* sf, float* g_dec,
                            void* ws, nvfp4_stream_t stream);

/*
 * 2-D 16x16 block quantization for weights ["Entrenamiento ...",
 * "Metodología de Entrenamiento": two-dimensional block scaling for weights].
 * One E4M3 scale per 16x16 tile, stored in each of the tile's 16 rows;
 * round-to-nearest.  rows % 16 == 0, cols % 16 == 0.
 *   q, sf   out: [rows, cols/2] codes and their scales (as nvfp4_quantize)
 *   qT, sfT out (both NULL or both set): the transpose, [cols, rows/2] codes
 *           and nvfp4_sf_bytes(cols, rows) scales — the K-major operand of
 *           the gradient-wrt-input matmul.
 */
nvfp4_status nvfp4_quantize_2d(const void* w, int64_t rows, int64_t cols, int64_t ld,
                               uint8_t* q, uint8_t* sf, uint8_t* qT, uint8_t* sfT,
                               float* g_dec, void* ws, nvfp4_stream_t stream);

/*
 * Random Hadamard transform + quantization, written transposed, for the
 * weight-gradient operands ["Entrenamiento ...", "Metodología de
 * Entrenamiento": random Hadamard transforms; stochastic rounding on
 * gradients].  For every channel c and 16-token chunk v of x [T, C]:
 * y = (1/4) H16 D v, D = diag(±1) from rht_seed (the same for all chunks and
 * for both operands of one weight-gradient matmul), butterflies with strides
 * 1, 2, 4, 8.  amax runs over the transformed values.  T % 16 == 0.
 *   qT  out: uint8 [C, T/2] codes, tokens contiguous (block index for SR =
 *       c * T/16 + t/16)
 *   sfT out: nvfp4_sf_bytes(C, T) scales
 */
nvfp4_status nvfp4_rht_quantize(const void* x, int64_t T, int64_t C, int64_t ld,
                                uint64_t rht_seed, nvfp4_round mode, uint64_t sr_seed,
                                uint8_t* qT, uint8_t* sfT, float* g_dec,
                                void* ws, nvfp4_stream_t stream);

/*
 * Both quantized forms of one activation or gradient x [T, C] from a single
 * read of x: the 1x16 row form (q, sf, g_dec; exactly what nvfp4_quantize
 * writes with mode / sr_seed) for the forward or data-gradient matmul, and
 * the Hadamard-transformed transposed form (qT, sfT, g_dec_t; exactly what
 * nvfp4_rht_quantize writes with rht_seed / mode_t / sr_seed_t) for the
 * weight-gradient matmul ["Entrenamiento ...", "Metodología de
 * Entrenamiento": each matmul's operands are quantized along its reduction
 * dimension; random Hadamard transforms on Wgrad inputs].  Each form has its
 * own tensor amax and decode scale.  T % 16 == 0, C % 16 == 0.  All outputs
 * are device buffers owned by the caller; the errors are those of the two
 * single-form calls.
 */
nvfp4_status nvfp4_quantize_dual(const void* x, int64_t T, int64_t C, int64_t ld,
                                 nvfp4_round mode, uint64_t sr_seed,
                                 uint8_t* q, uint8_t* sf, float* g_dec,
                                 uint64_t rht_seed, nvfp4_round mode_t, uint64_t sr_seed_t,
                                 uint8_t* qT, uint8_t* sfT, float* g_dec_t,
                                 void* ws, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_dual with both tensor amaxes given: amax (2 floats of
 * DEVICE memory, 4-byte aligned) holds max |x| and the Hadamard form's max
 * |y| as nvfp4_gemm_amax writes them for its output.  The kernel skips its
 * reduction pass and the grid-wide barrier and reads x once.  Every output is
 * what nvfp4_quantize_dual writes when the given values are the true
 * maxima; a non-finite amax is reported as NVFP4_ERR_NONFINITE.
 */
nvfp4_status nvfp4_quantize_dual_from_amax(const void* x, int64_t T, int64_t C, int64_t ld,
                                           const float* amax,
                                           nvfp4_round mode, uint64_t sr_seed,
                                           uint8_t* q, uint8_t* sf, float* g_dec,
                                           uint64_t rht_seed, nvfp4_round mode_t, uint64_t sr_seed_t,
                                           uint8_t* qT, uint8_t* sfT, float* g_dec_t,
                                           void* ws, nvfp4_stream_t stream);

/*
 * Quantization-noise meter ["FP4 All the Way", "Describir": quantized
 * training loses efficiency once the gradient norm falls below about
 * sqrt(3) times the quantization noise].  For x [rows, cols] (bf16, leading
 * dimension ld) and its 1x16 form (q, sf, g_dec) as nvfp4_quantize, the row
 * outputs of nvfp4_quantize_2d or nvfp4_quantize_dual write it:
 *   sums[0] = sum over all elements of (Q(x) - x)^2,
 *             Q(x) = E2M1(code) * E4M3(scale) * g_dec,
 *   sums[1] = sum of x^2,
 * so ||x|| / ||Q(x) - x|| = sqrt(sums[1] / sums[0]) is compared with sqrt(3).
 * sums: 2 doubles of DEVICE memory (8-byte aligned), overwritten (the call
 * zeroes them on `stream` first).  Elements are differenced in binary32
 * (one fused multiply-add each), blocks summed in binary32 and totals kept in
 * binary64; the order of the totals is not fixed (relative differences of a
 * few 1e-7 between runs).  cols % 16 == 0.  Non-finite x gives non-finite
 * sums.  No workspace needed.
 */
nvfp4_status nvfp4_quant_noise(const void* x, int64_t rows, int64_t cols, int64_t ld,
                               const uint8_t* q, const uint8_t* sf, const float* g_dec,
                               double* sums, nvfp4_stream_t stream);

/*
 * Block-scaled NVFP4 matmul on the tcgen05 tensor cores [NVFP4 is supported
 * by Blackwell tensor cores: "Entrenamiento ...", "El Desafío de la
 * Precisión de 4 Bits"].
 *   D[m, n] = ga * gb * sum_k A(m, k) B(n, k), A and B decoded NVFP4 (codes
 *   times block scales), binary32 accumulation, output bf16 (round to
 *   nearest) or binary32.
 *   a, sfa  [M, K/2] codes + nvfp4_sf_bytes(M, K) scales (K contiguous)
 *   b, sfb  [N, K/2] codes + nvfp4_sf_bytes(N, K) scales (K contiguous)
 *   ga, gb  device floats (the quantizers' g_dec)
 *   d       out: [M, N] row-major, leading dimension ldd (elements); ldd
 *           times the element size a multiple of 16 bytes
 * Shapes: M, N, K > 0 and K % 32 == 0 (a code row must be a whole number of
 * 16-byte units for the tensor copies).  Ragged M, N and K are handled: the
 * last tiles are padded on chip and only rows < M, columns < N are written.
 * The padding bytes of sfa and sfb (past row M / N, past K/16 in the last
 * 4-block group) must not be NaN codes (0x7F, 0xFF); the quantizers write
 * zeros there.
 */
nvfp4_status nvfp4_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga,
                        const uint8_t* b, const uint8_t* sfb, const float* gb,
                        int64_t M, int64_t N, int64_t K,
                        void* d, int64_t ldd, nvfp4_out_dtype out_dtype,
                        void* ws, nvfp4_stream_t stream);

/*
 * nvfp4_gemm with bf16 output that also reduces the two tensor amaxes the
 * quantization of its output needs, so that nvfp4_quantize_dual_from_amax can
 * quantize D in one pass instead of reading it twice [multi-level scaling:
 * the tensor scale comes from the tensor's amax, "I ricercatori di Nvidia
 * ...", "Come funziona NVFP4?"; the Wgrad form is Hadamard-transformed along
 * tokens, "Entrenamiento ...", "Metodología de Entrenamiento"].  Rows of D
 * are tokens, columns channels.
 *   amax    out: 2 floats of DEVICE memory (4-byte aligned), written when the
 *           GEMM ends:
 *             amax[0] = max |D| over the bf16 output,
 *             amax[1] = max |y| over y = (1/4) H16 S v for every 16-row block
 *                       v of every column of D (S from rht_seed, as
 *                       nvfp4_rht_quantize; butterflies with strides 1, 2, 4,
 *                       8 in binary32),
 *           bit-identical to the amaxes nvfp4_quantize_dual computes from D
 *           with the same rht_seed.  A non-finite D gives a non-finite amax,
 *           which the quantizer reports.
 * Arguments otherwise as nvfp4_gemm with out_dtype = NVFP4_OUT_BF16.
 * M % 16 == 0 and N % 16 == 0 (the shapes the dual quantizer takes).  Runs on
 * the paired-SM kernel for every M.  The workspace carries the partial
 * maxima while the GEMM runs (the last CTA clears them): one call at a time
 * per workspace, as for every call.
 */
nvfp4_status nvfp4_gemm_amax(const uint8_t* a, const uint8_t* sfa, const float* ga,
                             const uint8_t* b, const uint8_t* sfb, const float* gb,
                             int64_t M, int64_t N, int64_t K,
                             void* d, int64_t ldd, uint64_t rht_seed, float* amax,
                             void* ws, nvfp4_stream_t stream);

/*
 * MXFP4, the comparison format ["I ricercatori di Nvidia sbloccano ...",
 * section "Come funziona NVFP4?": MXFP4 reached the same accuracy only with
 * markedly more training data].  The pages do not define it; this follows the
 * OCP Microscaling (MX) v1.0 specification: blocks of 32 contiguous
 * elements, E2M1 codes, one UE8M0 scale 2^e per block, no tensor scale.
 *   e = floor(log2(max |x| over the block)) - 2, clamped to [-127, 127]
 *       (max 0 or below the smallest normal binary32: e = -127);
 *   code = E2M1 round-to-nearest-even of x / 2^e, saturating at 6, sign kept;
 *   scale byte = e + 127; a block holding Inf/NaN gets 0xFF (UE8M0 NaN),
 *   zero codes, and NVFP4_ERR_NONFINITE is recorded in `ws`.
 *   x   bf16 [rows, cols], leading dimension ld; cols % 32 == 0
 *   q   out: uint8 [rows, cols/2] codes (element 2i in the low nibble)
 *   sf  out: nvfp4_sf_bytes(rows, cols) bytes: one 32-bit word per row per 64
 *       elements in the 128 x 4 atom layout, the two block scales in bytes 0
 *       and 1, bytes 2 and 3 zero; byte of (row r, block kb) at
 *       ((r/128) * Cp + kb/2) * 512 + (r%32) * 16 + ((r%128)/32) * 4 + kb%2,
 *       Cp = ceil(cols / 64); padding rows and bytes are written as 0.
 * One streaming pass (no tensor amax, no grid barrier).
 */
nvfp4_status nvfp4_mxfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                  uint8_t* q, uint8_t* sf, void* ws, nvfp4_stream_t stream);

/*
 * MXFP4 block-scaled matmul on the tcgen05 tensor cores (UE8M0 block-32
 * scales): D[m, n] = sum_k A(m, k) B(n, k), A and B decoded MXFP4, binary32
 * accumulation, output bf16 (nearest) or binary32.  Operands as
 * nvfp4_mxfp4_quantize writes them, K contiguous; shapes and output rules as
 * nvfp4_gemm (any M, N > 0, K % 32 == 0, only rows < M and columns < N
 * written).  Padding scale bytes must not be 0xFF.
 */
nvfp4_status nvfp4_mxfp4_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                              int64_t M, int64_t N, int64_t K, void* d, int64_t ldd,
                              nvfp4_out_dtype out_dtype, void* ws, nvfp4_stream_t stream);

/* Synchronise `stream` and return the sticky device status kept in `ws`
 * (NVFP4_OK if no device-side error was recorded). */
nvfp4_status nvfp4_device_status(void* ws, nvfp4_stream_t stream);

/* Static string for a status code. */
const char* nvfp4_status_str(nvfp4_status s);

/*
 * Diagnostic entry point: run the device's element encoders on n inputs —
 * E4M3 nearest-even saturating (e4m3_out, for x >= 0), E2M1 nearest-even
 * (e2m1_rn_out) and E2M1 stochastic with the 16-bit random value r[i]
 * (e2m1_sr_out: up iff the fraction between the grid neighbours, kept to 16
 * bits, plus r[i] carries) — the instructions the quantizers use.  r may be
 * NULL (all zero); any output may be NULL.  Device pointers.
 */
nvfp4_status nvfp4_encode_probe(const float* v, const uint16_t* r, int64_t n,
                                uint8_t* e4m3_out, uint8_t* e2m1_rn_out, uint8_t* e2m1_sr_out,
                                nvfp4_stream_t stream);

/*
 * nvfp4_quantize_noalloc — the 1x16 quantizer of nvfp4_quantize for callers
 * that cannot allocate device memory.  (The pages have no counterpart; this
 * is an interface convenience.)
 *
 * Who needs it: code that may not call cudaMalloc or any allocating routine —
 * a plugin running inside a host program that owns all device memory through
 * its own allocator, a deployment that reserves the whole device at start-up,
 * or a latency-critical path where an allocation could block or synchronise
 * the device.  nvfp4_quantize wants a caller-allocated workspace; this variant
 * keeps that scratch in a 256-byte static device array inside the library
 * instead, so the caller passes only the input and the outputs.
 *
 * Arguments, layouts and results are those of nvfp4_quantize (same kernel,
 * same bits).  Differences:
 *  - no workspace: the scratch is a file-scope device array of 256 bytes,
 *    held by every GPU that loads the library until the process exits; a
 *    shape whose workspace (nvfp4_workspace_bytes) would exceed it returns
 *    NVFP4_ERR_SHAPE;
 *  - nothing is allocated: no cudaMalloc/cudaFree, no allocating library call;
 *  - each call clears the scratch on `stream` before its launch; all calls
 *    share the one array, so calls that overlap on the GPU (e.g. on two
 *    streams at once) race — serialise them, e.g. on one stream;
 *  - every call looks up the array's device address (cudaGetSymbolAddress,
 *    which allocates nothing) with the calling thread's device current, so an
 *    address that moved after cudaDeviceReset or a module reload is never
 *    reused; while `stream` is capturing, the address looked up by the last
 *    call on that device outside a capture is used, so make the first call on
 *    each device before any stream capture begins;
 *  - device-detected errors are not kept anywhere the caller can query, and
 *    the next call's clear erases them: a non-finite input shows up as a
 *    non-finite *g_dec, but a bounded device wait that runs out (the grid
 *    barrier after 2 s, NVFP4_ERR_TIMEOUT under nvfp4_quantize) leaves finite,
 *    wrong codes, scales and *g_dec that nothing reports.  Callers that need
 *    to see those errors use nvfp4_quantize with a workspace and
 *    nvfp4_device_status.
 */
nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                    nvfp4_round mode, uint64_t sr_seed,
                                    uint8_t* q, uint8_t* sf, float* g_dec,
                                    nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H */
