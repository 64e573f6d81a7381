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

// A 32-row x `width`-column output chunk that crosses the M or N edge is
// written with plain stores instead of a tensor store, so that nothing outside
// M x N is touched whatever the tensor unit does with a partial 16-byte unit.
__device__ __forceinline__ bool edge_chunk(int32_t col, int32_t width, int32_t row0, const GemmArgs& a)
{
    return col + width > a.N || row0 + 32 > a.M;
}

constexpr int kStoreBufBytes = 1024;  // per epilogue warp: 32 rows x 32 bytes

// Send one 32-row x 32-byte chunk (w: this lane's row) through the warp's
// staging buffer and a TMA tensor store at (col, row0).
__device__ __forceinline__ void store_chunk(const uint32_t (&w)[8], int32_t col, int32_t row0, uint8_t* buf,
                                            const CUtensorMap* tma_d, int lane)
{
    if (lane == 0)
        bulk_wait_read0();
    __syncwarp();
    reinterpret_cast<uint4*>(buf + lane * 32)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(buf + lane * 32)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tma_d, buf, col, row0);
        bulk_commit_group();
    }
}

// Store this warp's 32 rows (row0 + lane) x 128 columns (c0 ..) held as bf16
// pairs in p (word j: columns c0 + 2j, c0 + 2j + 1, the first in the low
// half): 16-column chunks leave through TMA tensor stores; chunks on the M/N
// edge take plain stores of the valid elements.
__device__ __forceinline__ void epilogue_store_bf16(const uint32_t (&p)[64], int32_t row0, int32_t c0,
                                                   const GemmArgs& args, uint8_t* buf, const CUtensorMap* tma_d,
                                                   int lane)
{
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const int32_t col = c0 + ch * 16;
        if (col >= args.N)
            break;
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            w[e] = p[ch * 8 + e];
        if (edge_chunk(col, 16, row0, args)) {
            const int32_t row = row0 + lane;
            if (row < args.M) {
                uint16_t* dst = static_cast<uint16_t*>(args.d) + (int64_t)row * args.ldd + col;
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (col + e < args.N)
                        dst[e] = (uint16_t)(w[e >> 1] >> (16 * (e & 1)));
            }
            continue;
        }
        store_chunk(w, col, row0, buf, tma_d, lane);
    }
}

// Store 32 rows x 32 columns (c0 ..) of binary32 accumulator values r times
// alpha, in 8-column chunks, as above.
__device__ __forceinline__ void epilogue_store_f32(const uint32_t (&r)[32], float alpha, int32_t row0, int32_t c0,
                                                  const GemmArgs& args, uint8_t* buf, const CUtensorMap* tma_d,
                                                  int lane)
{
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const int32_t col = c0 + ch * 8;
        if (col >= args.N)
            break;
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            w[e] = __float_as_uint(__fmul_rn(__uint_as_float(r[ch * 8 + e]), alpha));
        if (edge_chunk(col, 8, row0, args)) {
            const int32_t row = row0 + lane;
            if (row < args.M) {
                float* dst = static_cast<float*>(args.d) + (int64_t)row * args.ldd + col;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (col + e < args.N)
                        dst[e] = __uint_as_float(w[e]);
            }
            continue;
        }
        store_chunk(w, col, row0, buf, tma_d, lane);
    }
}

}  // namespace nvfp4
