// Quantization-noise meter ("FP4 All the Way: Formación totalmente
// cuantificada de LLM", section "Describir": quantized training loses
// efficiency once the gradient norm drops below about sqrt(3) times the
// quantization noise).
//
// For a bf16 tensor x [rows, cols] and its 1x16 NVFP4 form (codes q, scales
// sf, decode scale g), one pass over the three accumulates
//   sums[0] = sum (Q(x) - x)^2,  Q(x) = E2M1(code) * E4M3(scale) * g,
//   sums[1] = sum x^2,
// so that the caller compares ||x|| with sqrt(3) ||Q(x) - x||.
//
// Memory-bound: 2 + 0.5 + 1/16 bytes read per element.  One warp walks one
// row at a time, each lane one 16-element block per step (the warp reads 1 KB
// of x and 256 bytes of codes contiguously); per block the differences are
// formed with one fused multiply-add each, summed in binary32 and added to
// binary64 per-thread totals, which meet in shared memory and then in two
// binary64 atomics per CTA.
#include "device.cuh"

namespace nvfp4 {
namespace {

constexpr int kNoiseThreads = 256;
constexpr int kNoiseCtasPerSm = 8;

// Two E2M1 codes (one byte, element 2i in the low nibble) to two floats.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte)
{
    uint32_t h2;
    asm("{\n.reg .b8 t;\ncvt.u8.u32 t, %1;\ncvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(h2) : "r"(byte));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

struct NoiseArgs {
    const uint8_t* x;  // bf16 rows, stride ld elements
    const uint8_t* q;
    const uint8_t* sf;
    const float* g_dec;
    double* sums;
    int64_t rows;
    int64_t ld;
    uint32_t kblocks;  // cols / 16
    uint32_t cp;       // 4-block groups per row in the scale layout
};

__device__ __forceinline__ void block_noise(const NoiseArgs& a, int64_t r, uint32_t kc, float g, double& se,
                                            double& sx)
{
    const uint4* xp = reinterpret_cast<const uint4*>(a.x + (r * a.ld + (int64_t)kc * 16) * 2);
    const uint4 x0 = __ldcs(xp), x1 = __ldcs(xp + 1);
    const uint2 cq = __ldcs(reinterpret_cast<const uint2*>(a.q + r * (int64_t)a.kblocks * 8 + (int64_t)kc * 8));
    const uint32_t rr = (uint32_t)(r & 127);
    const uint8_t sb = a.sf[((r >> 7) * a.cp + (kc >> 2)) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (kc & 3)];
    const float s = __fmul_rn(e4m3_value(sb), g);
    const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const uint32_t qw[2] = {cq.x, cq.y};
    float e = 0.0f, xx = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 c = e2m1x2_to_float2((qw[j >> 2] >> (8 * (j & 3))) & 0xFFu);
        const float v0 = bf16lo(xw[j]), v1 = bf16hi(xw[j]);
        const float d0 = __fmaf_rn(c.x, s, -v0), d1 = __fmaf_rn(c.y, s, -v1);
        e = __fmaf_rn(d0, d0, e);
        e = __fmaf_rn(d1, d1, e);
        xx = __fmaf_rn(v0, v0, xx);
        xx = __fmaf_rn(v1, v1, xx);
    }
    se += (double)e;
    sx += (double)xx;
}

__global__ void __launch_bounds__(kNoiseThreads) noise_meter_kernel(const NoiseArgs a)
{
    __shared__ double part[2][kNoiseThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gwarp = (int64_t)blockIdx.x * (kNoiseThreads / 32) + warp;
    const int64_t nwarps = (int64_t)gridDim.x * (kNoiseThreads / 32);
    const float g = *a.g_dec;
    double se = 0.0, sx = 0.0;
    for (int64_t r = gwarp; r < a.rows; r += nwarps) {
        uint32_t kc = (uint32_t)lane;
        for (; kc + 32 < a.kblocks; kc += 64) {  // two blocks in flight per lane
            block_noise(a, r, kc, g, se, sx);
            block_noise(a, r, kc + 32, g, se, sx);
        }
        if (kc < a.kblocks)
            block_noise(a, r, kc, g, se, sx);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        se += __shfl_xor_sync(0xFFFFFFFFu, se, off);
        sx += __shfl_xor_sync(0xFFFFFFFFu, sx, off);
    }
    if (lane == 0) {
        part[0][warp] = se;
        part[1][warp] = sx;
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        double t = 0.0;
        for (int w = 0; w < kNoiseThreads / 32; ++w)
            t += part[threadIdx.x][w];
        atomicAdd(&a.sums[threadIdx.x], t);
    }
}

}  // namespace

nvfp4_status launch_quant_noise(const void* x, int64_t rows, int64_t cols, int64_t ld, const uint8_t* q,
                                const uint8_t* sf, const float* g_dec, double* sums, cudaStream_t stream)
{
    if (cudaMemsetAsync(sums, 0, 2 * sizeof(double), stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    NoiseArgs a;
    a.x = static_cast<const uint8_t*>(x);
    a.q = q;
    a.sf = sf;
    a.g_dec = g_dec;
    a.sums = sums;
    a.rows = rows;
    a.ld = ld;
    a.kblocks = (uint32_t)(cols / 16);
    a.cp = (a.kblocks + 3) / 4;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, noise_meter_kernel, kNoiseThreads, 0) != cudaSuccess ||
        occ < 1)
        return NVFP4_ERR_CUDA;
    const int64_t warps_needed = rows;
    int64_t grid = (int64_t)device_sm_count() * (occ < kNoiseCtasPerSm ? occ : kNoiseCtasPerSm);
    const int64_t need = (warps_needed + kNoiseThreads / 32 - 1) / (kNoiseThreads / 32);
    if (need < grid)
        grid = need;
    noise_meter_kernel<<<(unsigned)grid, kNoiseThreads, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
