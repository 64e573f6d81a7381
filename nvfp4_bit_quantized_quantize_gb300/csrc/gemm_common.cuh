// Pieces of the block-scaled GEMM kernel: arguments, instruction descriptor,
// epilogue store.
#pragma once

#include "device.cuh"

namespace nvfp4 {

struct GemmArgs {
    const uint8_t* sfa;
    const uint8_t* sfb;
    const float* ga;
    const float* gb;
    void* d;
    int64_t ldd;
    int32_t M, N, K;
    int32_t out_f32;
    // bf16 output only: when set, the epilogue also reduces max |D| and
    // max |RHT(D)| (see epilogue_amax) and the last epilogue warp of the grid
    // writes them here
    float* amax_out;
    uint32_t rht_signs;  // bit i: the sign diagonal flips token i of every 16-token block
};

// Instruction descriptor for kind::mxf4nvf4: E2M1 A and B (format 1),
// K-major both, N >> 3 at bit 17, scale type at bit 23 (0 = E4M3 for NVFP4's
// block-16 scales, 1 = UE8M0 for MXFP4's block-32 scales), M >> 4 at bit 24,
// scale-factor ids 0 (one 32-bit scale word per row per K = 64 step).
template <bool kMx>
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t m, uint32_t n)
{
    return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24) | (kMx ? (1u << 23) : 0u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

constexpr int kStoreBufBytes = 1024;  // per epilogue warp: 32 rows x 32 bytes

// Write this lane's 32-byte row (words base .. base + 7 of w) of a 32-row
// chunk of `width` columns into the warp's staging buffer (after the previous
// tensor store has read it), then either send the chunk with one TMA tensor
// store at (col, row0) or, for a chunk crossing the M or N edge, copy each
// row's elements inside M x N out with plain stores (so nothing outside
// M x N is touched whatever the tensor unit would do with a partial 16-byte
// unit).
template <int kN>
__device__ __forceinline__ void store_chunk(const uint32_t (&w)[kN], int base, int32_t col, int32_t width,
                                            int32_t row0, const GemmArgs& args, uint8_t* buf,
                                            const CUtensorMap* tma_d, int lane)
{
    if (elect_one())
        bulk_wait_read0();
    __syncwarp();
    uint8_t* row = buf + lane * 32;
    reinterpret_cast<uint4*>(row)[0] = make_uint4(w[base], w[base + 1], w[base + 2], w[base + 3]);
    reinterpret_cast<uint4*>(row)[1] = make_uint4(w[base + 4], w[base + 5], w[base + 6], w[base + 7]);
    if (col + width > args.N || row0 + 32 > args.M) {
        __syncwarp();
        const int32_t r = row0 + lane;
        const int es = 32 / width;  // element bytes
        if (r < args.M) {
            uint8_t* dst = static_cast<uint8_t*>(args.d) + ((int64_t)r * args.ldd + col) * es;
#pragma unroll 1
            for (int e = 0; e < width && col + e < args.N; ++e) {
                if (es == 2)
                    reinterpret_cast<uint16_t*>(dst)[e] = reinterpret_cast<const uint16_t*>(row)[e];
                else
                    reinterpret_cast<uint32_t*>(dst)[e] = reinterpret_cast<const uint32_t*>(row)[e];
            }
        }
        __syncwarp();
        return;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (elect_one()) {
        tma_store_2d(tma_d, buf, col, row0);
        bulk_commit_group();
    }
}

// Store this warp's 32 rows (row0 + lane) x 128 columns (c0 ..) held as bf16
// pairs in p (word j: columns c0 + 2j, c0 + 2j + 1, the first in the low
// half) as eight 16-column chunks.
__device__ __forceinline__ void epilogue_store_bf16(const uint32_t (&p)[64], int32_t row0, int32_t c0,
                                                   const GemmArgs& args, uint8_t* buf, const CUtensorMap* tma_d,
                                                   int lane)
{
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const int32_t col = c0 + ch * 16;
        if (col >= args.N)
            break;
        store_chunk(p, ch * 8, col, 16, row0, args, buf, tma_d, lane);
    }
}

// Store 32 rows x 32 columns (c0 ..) of binary32 accumulator values r times
// alpha as four 8-column chunks.
__device__ __forceinline__ void epilogue_store_f32(const uint32_t (&r)[32], float alpha, int32_t row0, int32_t c0,
                                                  const GemmArgs& args, uint8_t* buf, const CUtensorMap* tma_d,
                                                  int lane)
{
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 32; ++e)
        w[e] = __float_as_uint(__fmul_rn(__uint_as_float(r[e]), alpha));
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const int32_t col = c0 + ch * 8;
        if (col >= args.N)
            break;
        store_chunk(w, ch * 8, col, 8, row0, args, buf, tma_d, lane);
    }
}

// ---- wide chunks (binary32 output of the paired-SM kernel): 32 rows x 128
// bytes per tensor store, staged in a 4 KB buffer per warp in the store's
// 128-byte swizzle
// (16-byte unit u of row r at r * 128 + ((u ^ (r % 8)) * 16), so the eight
// rows of a quarter-warp's 16-byte writes cover all 32 banks).
constexpr int kWideBufBytes = 4096;

// Write this lane's 128-byte row (words w[base] .. w[base + 31]) of a chunk of
// `width` columns at (col, row0), after the previous store has read the
// buffer, then send it with one tensor store -- or, across the M or N edge,
// copy each row's elements inside M x N out with plain stores.
__device__ __forceinline__ void store_wide_chunk(const uint32_t* w, int32_t col, int32_t width, int32_t row0,
                                                 const GemmArgs& args, uint8_t* buf, const CUtensorMap* tma_d,
                                                 int lane)
{
    if (elect_one())
        bulk_wait_read0();
    __syncwarp();
    uint8_t* row = buf + lane * 128;
    const uint32_t r7 = (uint32_t)lane & 7u;
#pragma unroll
    for (uint32_t u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(row + ((u ^ r7) << 4)) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
    if (col + width > args.N || row0 + 32 > args.M) {
        __syncwarp();
        const int32_t r = row0 + lane;
        const int es = 128 / width;  // element bytes
        if (r < args.M) {
            uint8_t* dst = static_cast<uint8_t*>(args.d) + ((int64_t)r * args.ldd + col) * es;
#pragma unroll 1
            for (int e = 0; e < width && col + e < args.N; ++e) {
                const uint32_t off = (uint32_t)(e * es);
                const uint8_t* src = row + ((((off >> 4) ^ r7) << 4) | (off & 15u));
                if (es == 2)
                    reinterpret_cast<uint16_t*>(dst)[e] = *reinterpret_cast<const uint16_t*>(src);
                else
                    reinterpret_cast<uint32_t*>(dst)[e] = *reinterpret_cast<const uint32_t*>(src);
            }
        }
        __syncwarp();
        return;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (elect_one()) {
        tma_store_2d(tma_d, buf, col, row0);
        bulk_commit_group();
    }
}

// 32 rows x 32 binary32 columns (c0 ..) of accumulator values r times alpha
// as one chunk.
__device__ __forceinline__ void epilogue_store_f32_wide(const uint32_t (&r)[32], float alpha, int32_t row0,
                                                       int32_t c0, const GemmArgs& args, uint8_t* buf,
                                                       const CUtensorMap* tma_d, int lane)
{
    if (c0 >= args.N)
        return;
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 32; ++e)
        w[e] = __float_as_uint(__fmul_rn(__uint_as_float(r[e]), alpha));
    store_wide_chunk(w, c0, 32, row0, args, buf, tma_d, lane);
}

// ---- output maxima for the quantizers of D ----------------------------------
// The activation or gradient a GEMM writes is quantized next in both of its
// forms, each needing its tensor amax: max |D| over the bf16 output (the 1x16
// form) and max |y| over y = (1/4) H16 S v for every 16-row block v of each
// column (the Hadamard form along tokens: rows of D are tokens; S the sign
// diagonal of rht_signs).  The epilogue holds every output value once, so it
// reduces both there, in the arithmetic the quantizer's own reduction uses
// (bf16 values widened exactly, sign flips, butterflies of strides 1, 2, 4 in
// binary32, the stride-8 pair's larger magnitude as rn(|a| + |b|), the exact
// 1/4 last), which makes the maxima bit-identical to what a separate pass over
// D computes.  Elements outside M x N count as zeros.

// Per epilogue warp: 32 rows x 16 words (32 columns) of bf16 pairs, row
// stride 17 words, so both the row-wise writes and the column-wise reads of
// 16 rows fall in 32 different banks.
constexpr int kRhtStride = 17;
constexpr int kRhtBufBytes = 32 * kRhtStride * 4;

// Fold 32-column chunk ch (words 16 ch .. 16 ch + 15 of p: columns c0 + 32 ch
// ..) of this warp's 32 rows (row0 + lane) into the lane's running maxima:
// rmax, a bf16x2 |.| accumulator over D, and tmax, the largest stride-8
// magnitude rn(|a| + |b|) of the transformed blocks (binary32,
// NaN-propagating).  The Hadamard blocks are rows 16g .. 16g + 15 of the warp
// (row0 is a multiple of 32); the chunk goes through rbuf so that lane (g, u)
// gets the 16 tokens of column pair u.
__device__ __forceinline__ void epilogue_amax_chunk(const uint32_t (&p)[64], int ch, int32_t row0, int32_t c0,
                                                    const GemmArgs& args, uint32_t* rbuf, int lane, uint32_t& rmax,
                                                    float& tmax)
{
    const int32_t ncols = args.N - c0 - ch * 32;  // > 0
    const bool row_in = row0 + lane < args.M;
    const bool whole = ncols >= 32 && row0 + 32 <= args.M;
    const uint32_t flip = ((args.rht_signs >> (lane & 15)) & 1u) ? 0x80008000u : 0u;
    __syncwarp();  // the previous chunk's reads are done
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        uint32_t w = p[ch * 16 + j];
        if (!whole)
            w &= (!row_in || 2 * j >= ncols) ? 0u : (2 * j + 1 >= ncols ? 0xFFFFu : 0xFFFFFFFFu);
        rmax = habs_max2(rmax, w);
        rbuf[lane * kRhtStride + j] = w ^ flip;
    }
    __syncwarp();
    const uint32_t* col = rbuf + (lane >> 4) * 16 * kRhtStride + (lane & 15);
    uint64_t P[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t w = col[i * kRhtStride];
        P[i] = f2_pack(bf16lo(w), bf16hi(w));
    }
#pragma unroll
    for (int hs = 1; hs < 8; hs <<= 1) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k & hs)
                continue;
            const uint64_t a = P[k], b = P[k + hs];
            P[k] = f2_add(a, b);
            P[k + hs] = f2_sub(a, b);
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float a0, a1, b0, b1;
        f2_unpack(P[k], a0, a1);
        f2_unpack(P[k + 8], b0, b1);
        asm("max.NaN.f32 %0, %1, %2;" : "=f"(tmax) : "f"(tmax), "f"(__fadd_rn(fabsf(a0), fabsf(b0))));
        asm("max.NaN.f32 %0, %1, %2;" : "=f"(tmax) : "f"(tmax), "f"(__fadd_rn(fabsf(a1), fabsf(b1))));
    }
}

// epilogue_store_bf16 with the output maxima: each 32-column chunk is folded
// in right after its two stores, so the stored words die as the loop goes.
__device__ __forceinline__ void epilogue_store_bf16_amax(const uint32_t (&p)[64], int32_t row0, int32_t c0,
                                                        const GemmArgs& args, uint8_t* buf, uint32_t* rbuf,
                                                        const CUtensorMap* tma_d, int lane, uint32_t& rmax,
                                                        float& tmax)
{
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const int32_t col = c0 + ch * 32;
        if (col >= args.N)
            break;
        store_chunk(p, ch * 16, col, 16, row0, args, buf, tma_d, lane);
        if (col + 16 < args.N)
            store_chunk(p, ch * 16 + 8, col + 16, 16, row0, args, buf, tma_d, lane);
        epilogue_amax_chunk(p, ch, row0, c0, args, rbuf, lane, rmax, tmax);
    }
}

// After its last tile: the warp's maxima into the workspace; the grid's last
// epilogue warp (of `warps`) reads the totals, writes them to args.amax_out
// as floats (max |D|, max |y|) and clears the workspace for the next call.
__device__ __forceinline__ void epilogue_amax_finish(uint32_t rmax, float tmax, const GemmArgs& args,
                                                     Workspace* ws, uint32_t warps, int lane)
{
    uint32_t rb = __float_as_uint(hmax_to_float(rmax));
    uint32_t tb = __float_as_uint(__fmul_rn(tmax, 0.25f));  // exact, and monotone
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        rb = max(rb, __shfl_xor_sync(0xFFFFFFFFu, rb, off));
        tb = max(tb, __shfl_xor_sync(0xFFFFFFFFu, tb, off));
    }
    if (lane != 0)
        return;
    atomicMax(&ws->gemm_amax[0], rb);
    atomicMax(&ws->gemm_amax[1], tb);
    __threadfence();
    if (atomicAdd(&ws->gemm_done, 1u) == warps - 1) {
        __threadfence();
        const uint32_t a0 = atomicMax(&ws->gemm_amax[0], 0u);
        const uint32_t a1 = atomicMax(&ws->gemm_amax[1], 0u);
        args.amax_out[0] = __uint_as_float(a0);
        args.amax_out[1] = __uint_as_float(a1);
        ws->gemm_amax[0] = 0u;
        ws->gemm_amax[1] = 0u;
        ws->gemm_done = 0u;
        __threadfence();
    }
}

}  // namespace nvfp4
