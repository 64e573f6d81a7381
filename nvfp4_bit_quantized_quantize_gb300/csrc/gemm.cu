// Block-scaled NVFP4 GEMM on the sm_103a tensor cores ("Entrenamiento ...",
// "El Desafío de la Precisión de 4 Bits": NVFP4 runs on Blackwell tensor
// cores).
//
//   D[m, n] = ga * gb * sum_k A(m, k) * B(n, k)
//
// A [M, K] and B [N, K] are packed E2M1 codes (K contiguous) with one E4M3
// scale per 16 elements in the 128 x 4 atom layout.  Each CTA owns a
// persistent sequence of 128 x 256 output tiles:
//   warp 0  TMA producer: A/B tiles (128-byte swizzle) and the scale atoms
//           (bulk copies) into a 4-stage shared-memory ring;
//   warp 1  allocates tensor memory, moves the scale atoms into it
//           (tcgen05.cp) and issues tcgen05.mma.kind::mxf4nvf4 (K = 64 per
//           instruction, binary32 accumulator in tensor memory);
//   warps 2-5 epilogue: tcgen05.ld of the accumulator, times ga*gb, round to
//           bf16 (or keep binary32), store.
// Every wait is bounded; a wait that runs out records NVFP4_ERR_TIMEOUT and
// all roles wind down, drain their asynchronous work, and free tensor memory.
#include "device.cuh"

namespace nvfp4 {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 256;                       // elements per stage (128 bytes of codes per row)
constexpr int kStages = 4;
constexpr int kABytes = BM * BK / 2;          // 16 KB
constexpr int kBBytes = BN * BK / 2;          // 32 KB
constexpr int kSfaBytes = (BM / 128) * (BK / 64) * 512;  // 2 KB
constexpr int kSfbBytes = (BN / 128) * (BK / 64) * 512;  // 4 KB
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = BN;             // fp32 accumulator: 128 lanes x 256 columns
constexpr uint32_t kSfColsPerStage = 16 + 32; // SFA 4 steps x 4 cols, SFB 4 steps x 8 cols

static_assert(kStageBytes % 1024 == 0, "stage alignment");
static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");

struct GemmCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + sizeof(GemmCtl);

// Instruction descriptor for kind::mxf4nvf4: E2M1 A and B (format 1),
// K-major both, N >> 3 at bit 17, E4M3 scales (bit 23 = 0), M >> 4 at bit 24,
// scale-factor ids 0 (four scales per row per K = 64 step).
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct GemmArgs {
    const uint8_t* sfa;
    const uint8_t* sfb;
    const float* ga;
    const float* gb;
    void* d;
    int64_t M, N, K, ldd;
    int out_f32;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
    nvf4_gemm_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                     const GemmArgs args, Workspace* ws)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GemmCtl* ctl = reinterpret_cast<GemmCtl*>(smem + (size_t)kStages * kStageBytes);
    volatile int* abort = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_m = args.M / BM;
    const int64_t tiles_n = (args.N + BN - 1) / BN;
    const int64_t ntiles = tiles_m * tiles_n;
    const int64_t kstages = (args.K + BK - 1) / BK;
    const int64_t cp = (args.K / 16 + 3) / 4;   // scale atoms along K

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->tmem_full, 1);
        mbar_init(&ctl->tmem_empty, 4);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer ----
        tma_prefetch_desc(&tma_a);
        tma_prefetch_desc(&tma_b);
        int64_t it = 0;
        for (int64_t t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
            const int64_t tm = t % tiles_m, tn = t / tiles_m;
            const int64_t n0 = tn * BN;
            const int nrt = (args.N - n0) >= 256 ? 2 : 1;   // 128-row scale tiles present in B
            for (int64_t ks = 0; ks < kstages; ++ks, ++it) {
                const int s = (int)(it % kStages);
                if (it >= kStages && !mbar_wait(&ctl->empty[s], (uint32_t)(((it / kStages) - 1) & 1), ws, abort))
                    goto producer_done;
                uint8_t* st = smem + (size_t)s * kStageBytes;
                const int64_t groups_left = cp - ks * 4;
                const uint32_t gk = (uint32_t)(groups_left < 4 ? groups_left : 4);
                const uint32_t bytes = kABytes + kBBytes + gk * 512u * (1u + (uint32_t)nrt);
                mbar_expect_tx(&ctl->full[s], bytes);
                tma_load_2d(st, &tma_a, &ctl->full[s], (int32_t)(ks * 128), (int32_t)(tm * BM));
                tma_load_2d(st + kABytes, &tma_b, &ctl->full[s], (int32_t)(ks * 128), (int32_t)n0);
                bulk_load(st + kABytes + kBBytes, args.sfa + (tm * cp + ks * 4) * 512, gk * 512u, &ctl->full[s]);
                for (int h = 0; h < nrt; ++h)
                    bulk_load(st + kABytes + kBBytes + kSfaBytes + h * 2048,
                              args.sfb + ((2 * tn + h) * cp + ks * 4) * 512, gk * 512u, &ctl->full[s]);
            }
        }
    producer_done:
        for (int64_t i = it > kStages ? it - kStages : 0; i < it; ++i)
            mbar_wait(&ctl->full[i % kStages], (uint32_t)((i / kStages) & 1), ws, nullptr);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------ MMA issuer ----
        int64_t it = 0, titer = 0;
        for (int64_t t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x, ++titer) {
            if (titer > 0 && !mbar_wait(&ctl->tmem_empty, (uint32_t)((titer - 1) & 1), ws, abort))
                break;
            tc_fence_after();
            for (int64_t ks = 0; ks < kstages; ++ks, ++it) {
                const int s = (int)(it % kStages);
                if (!mbar_wait(&ctl->full[s], (uint32_t)((it / kStages) & 1), ws, abort))
                    goto mma_done;
                tc_fence_after();
                const uint32_t st = smem_u32(smem + (size_t)s * kStageBytes);
                const int64_t k_left = args.K - ks * BK;
                const int kk = (int)(k_left >= BK ? 4 : k_left / 64);
                const uint32_t sf_col = kAccCols + (uint32_t)s * kSfColsPerStage;
                for (int j = 0; j < kk; ++j) {
                    const uint32_t sfa_s = st + kABytes + kBBytes + j * 512;
                    const uint32_t sfb_s = st + kABytes + kBBytes + kSfaBytes + j * 512;
                    tmem_cp_32x128b_x4(tmem + sf_col + 4 * j, smem_desc(sfa_s, 0, 128, kSwizzleNone));
                    tmem_cp_32x128b_x4(tmem + sf_col + 16 + 8 * j, smem_desc(sfb_s, 0, 128, kSwizzleNone));
                    tmem_cp_32x128b_x4(tmem + sf_col + 16 + 8 * j + 4, smem_desc(sfb_s + 2048, 0, 128, kSwizzleNone));
                }
                for (int j = 0; j < kk; ++j) {
                    const uint64_t ad = smem_desc(st + 32 * j, 16, 1024, kSwizzle128B);
                    const uint64_t bd = smem_desc(st + kABytes + 32 * j, 16, 1024, kSwizzle128B);
                    mma_nvf4(tmem, ad, bd, kIdesc, tmem + sf_col + 4 * j, tmem + sf_col + 16 + 8 * j,
                             (ks > 0 || j > 0) ? 1u : 0u);
                }
                tc_commit(&ctl->empty[s]);
            }
            tc_commit(&ctl->tmem_full);
        }
    mma_done:
        // all tensor-core work issued by this thread completes before teardown
        tc_commit(&ctl->drain);
        mbar_wait(&ctl->drain, 0, ws, nullptr);
    } else if (warp >= 2) {
        // -------------------------------------------------------- epilogue ----
        const int q = warp & 3;                      // tensor-memory lane quarter
        const float alpha = __fmul_rn(*args.ga, *args.gb);
        int64_t titer = 0;
        for (int64_t t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x, ++titer) {
            const int64_t tm = t % tiles_m, tn = t / tiles_m;
            if (!mbar_wait(&ctl->tmem_full, (uint32_t)(titer & 1), ws, abort))
                break;
            tc_fence_after();
            const int64_t row = tm * BM + q * 32 + lane;
            const int64_t n0 = tn * BN;
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
            if (args.out_f32) {
                float* drow = reinterpret_cast<float*>(args.d) + row * args.ldd + n0;
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, r);
                    tmem_ld_wait();
                    if (n0 + c * 32 < args.N) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            reinterpret_cast<float4*>(drow + c * 32)[v] =
                                make_float4(__fmul_rn(__uint_as_float(r[4 * v]), alpha),
                                            __fmul_rn(__uint_as_float(r[4 * v + 1]), alpha),
                                            __fmul_rn(__uint_as_float(r[4 * v + 2]), alpha),
                                            __fmul_rn(__uint_as_float(r[4 * v + 3]), alpha));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ctl->tmem_empty);
            } else {
                uint32_t packed[BN / 2];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int v = 0; v < 16; ++v)
                        packed[c * 16 + v] = pack_bf16x2(__fmul_rn(__uint_as_float(r[2 * v]), alpha),
                                                         __fmul_rn(__uint_as_float(r[2 * v + 1]), alpha));
                }
                // accumulator is free once every load has landed in registers
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ctl->tmem_empty);
                __nv_bfloat16* drow = reinterpret_cast<__nv_bfloat16*>(args.d) + row * args.ldd + n0;
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    if (n0 + c * 32 < args.N) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            reinterpret_cast<uint4*>(drow + c * 32)[v] =
                                make_uint4(packed[c * 16 + 4 * v], packed[c * 16 + 4 * v + 1],
                                           packed[c * 16 + 4 * v + 2], packed[c * 16 + 4 * v + 3]);
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

nvfp4_status launch_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                         const uint8_t* sfb, const float* gb, int64_t M, int64_t N, int64_t K, void* d,
                         int64_t ldd, nvfp4_out_dtype dt, Workspace* ws, cudaStream_t stream)
{
    CUtensorMap ma, mb;
    if (!encode_tensor_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(a), (uint64_t)(K / 2),
                              (uint64_t)M, (uint64_t)(K / 2), 128u, (uint32_t)BM, CU_TENSOR_MAP_SWIZZLE_128B))
        return NVFP4_ERR_CUDA;
    if (!encode_tensor_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(b), (uint64_t)(K / 2),
                              (uint64_t)N, (uint64_t)(K / 2), 128u, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return NVFP4_ERR_CUDA;

    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(nvf4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess)
            return NVFP4_ERR_CUDA;
        attr_set[dev] = true;
    }
    GemmArgs args{sfa, sfb, ga, gb, d, M, N, K, ldd, dt == NVFP4_OUT_F32 ? 1 : 0};
    const int64_t ntiles = (M / BM) * ((N + BN - 1) / BN);
    const int sms = device_sm_count();
    const int grid = (int)(ntiles < sms ? ntiles : sms);
    nvf4_gemm_kernel<<<grid, kThreads, kSmemBytes, stream>>>(ma, mb, args, ws);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
