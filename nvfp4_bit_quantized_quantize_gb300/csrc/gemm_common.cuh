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
    if (lane == 0)
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
    if (lane == 0) {
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
    if (lane == 0)
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
    if (lane == 0) {
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

}  // namespace nvfp4
