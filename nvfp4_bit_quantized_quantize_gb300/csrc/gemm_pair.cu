// Block-scaled NVFP4 / MXFP4 GEMM on paired SMs (tcgen05 cta_group::2).
//
//   D[m, n] = ga * gb * sum_k A(m, k) * B(n, k)     (MXFP4: no ga * gb)
//
// A cluster of two CTAs on two SMs computes one 256 x 256 output tile with
// one M = 256 MMA per K = 64 step, issued by a single thread of the even CTA:
// each CTA stages its own 128 rows of A and its own 128 rows of B, so a CTA
// brings in half the B operand the one-SM kernel needs for the same work (the
// SM's L2 -> shared-memory traffic, not the tensor pipe, limits that kernel).
// Each CTA's tensor memory holds the accumulator of its 128 rows (256
// columns) and, per K step, its own rows' A scales and all 256 B scales.
//
//   warp 0    TMA producer (both CTAs): A and B boxes (128 rows x 128 bytes,
//             128-byte swizzle) and the scale atoms (3-D tensor boxes of
//             4 atoms; small non-tensor bulk copies here stalled the tensor
//             pipe) into a 5-stage ring;
//   warp 1    even CTA: tensor-memory allocation (with the odd CTA), scale
//             copies (tcgen05.cp.cta_group::2) and the MMAs; odd CTA: tells
//             the even CTA when each of its stages has landed;
//   warps 2-9 epilogue (both CTAs), two per tensor-memory lane quarter.
//
// Stage release and accumulator-ready signals go to both CTAs through
// multicast tcgen05.commit; the odd CTA's stage-landed and accumulator-drained
// signals reach the even CTA through relaxed remote mbarrier arrives (what
// they report finished before the arrive: the stage's TMA transfers, whose
// completion the odd CTA observed, and its tcgen05.ld of the accumulator,
// waited for with tcgen05.wait::ld), so no thread pays a cluster-scope fence
// in the steady state.  Every wait is
// bounded (a wait that runs out records NVFP4_ERR_TIMEOUT and the roles wind
// down); a cluster barrier keeps both CTAs (whose shared and tensor memory the
// MMAs touch) alive until all tensor-core work has finished.
#include "gemm_common.cuh"

namespace nvfp4 {
namespace {

constexpr int PM = 256;                 // pair tile rows (128 per CTA)
constexpr int PN = 256;                 // pair tile columns
constexpr int PK = 256;                 // elements of K per stage
constexpr int kPairStages = 5;
constexpr int kPA = 128 * PK / 2;       // 16 KB: this CTA's 128 rows of A
constexpr int kPB = 128 * PK / 2;       // 16 KB: this CTA's 128 rows of B
constexpr int kPSfa = (PK / 64) * 512;  // 2 KB: 4 atoms of this CTA's A rows
constexpr int kPSfb = 2 * (PK / 64) * 512;  // 4 KB: 4 atoms for each 128-row half of B
constexpr int kPStage = kPA + kPB + kPSfa + kPSfb;
constexpr int kPEpiWarps = 8;
constexpr int kPThreads = (2 + kPEpiWarps) * 32;
constexpr uint32_t kPTmemCols = 512;
constexpr uint32_t kPAccCols = PN;
constexpr uint32_t kPSfCols = 16 + 32;  // per stage: SFA 4 steps x 4 columns, SFB 4 steps x 8 columns
constexpr uint32_t kPSfSlots = 4;       // scale slots in tensor memory (a ring of their own)
constexpr uint32_t kPSfStride = 64;     // on 64-column boundaries

static_assert(kPStage % 1024 == 0, "stage alignment");
static_assert(kPSfCols <= kPSfStride, "scale slot");
static_assert(kPAccCols + kPSfSlots * kPSfStride <= kPTmemCols, "tensor memory budget");

struct PairCtl {
    uint64_t full[kPairStages];       // this CTA's stage landed (local TMA)
    uint64_t peer_full[kPairStages];  // even CTA: the odd CTA's stage landed
    uint64_t empty[kPairStages];      // stage free (multicast commit)
    uint64_t tmem_full;               // accumulator ready (multicast commit)
    uint64_t tmem_empty;              // even CTA: both CTAs drained (16 warps)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kPSmemBytes =
    1024 + (size_t)kPairStages * kPStage + kPEpiWarps * kStoreBufBytes + sizeof(PairCtl);

template <bool kMx>
__device__ __forceinline__ void pair_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t sfa, uint32_t sfb,
                                         uint32_t acc)
{
    if constexpr (kMx)
        mma_mxf4_pair(d, adesc, bdesc, mma_idesc<true>(PM, PN), sfa, sfb, acc);
    else
        mma_nvf4_pair(d, adesc, bdesc, mma_idesc<false>(PM, PN), sfa, sfb, acc);
}

template <bool kMx>
__global__ void __launch_bounds__(kPThreads, 1)
    nvf4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                          const __grid_constant__ CUtensorMap tma_sfa, const __grid_constant__ CUtensorMap tma_sfb,
                          const __grid_constant__ CUtensorMap tma_d, const GemmArgs args, Workspace* ws)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* store_buf = smem + (size_t)kPairStages * kPStage;
    PairCtl* ctl = reinterpret_cast<PairCtl*>(store_buf + kPEpiWarps * kStoreBufBytes);
    volatile int* abort = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
    const uint32_t cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const uint32_t tiles_m = ((uint32_t)args.M + PM - 1) / PM;
    const uint32_t tiles_n = ((uint32_t)args.N + PN - 1) / PN;
    const uint32_t ntiles = tiles_m * tiles_n;
    const uint32_t kstages = ((uint32_t)args.K + PK - 1) / PK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->peer_full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->tmem_full, 1);
        mbar_init(&ctl->tmem_empty, 2 * kPEpiWarps);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&ctl->tmem_base, kPTmemCols);
        tc_fence_before();
    }
    __syncthreads();
    // both CTAs' barriers are initialised before any remote arrive
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer ----
        tma_prefetch_desc(&tma_a);
        tma_prefetch_desc(&tma_b);
        tma_prefetch_desc(&tma_sfa);
        tma_prefetch_desc(&tma_sfb);
        uint32_t s = 0, phase = 0, issued = 0;
        for (uint32_t t = cluster; t < ntiles && !*abort; t += nclusters) {
            const uint32_t tm = t % tiles_m, tn = t / tiles_m;
            const uint32_t arow = tm * 2 + rank;  // this CTA's 128-row tile of A
            for (uint32_t ks = 0; ks < kstages; ++ks) {
                if (issued >= kPairStages && !mbar_wait(&ctl->empty[s], phase ^ 1, ws, abort))
                    goto producer_done;
                uint8_t* st = smem + (size_t)s * kPStage;
                // boxes past M, N or K read as zeros and still count in full
                mbar_expect_tx(&ctl->full[s], kPStage);
                tma_load_2d(st, &tma_a, &ctl->full[s], (int32_t)(ks * 128), (int32_t)(arow * 128));
                tma_load_2d(st + kPA, &tma_b, &ctl->full[s], (int32_t)(ks * 128), (int32_t)((2 * tn + rank) * 128));
                // scale atoms: this CTA's A rows; both 128-row halves of the B tile
                tma_load_3d(st + kPA + kPB, &tma_sfa, &ctl->full[s], 0, (int32_t)(ks * 4), (int32_t)arow);
                tma_load_3d(st + kPA + kPB + kPSfa, &tma_sfb, &ctl->full[s], 0, (int32_t)(ks * 4), (int32_t)(2 * tn));
                ++issued;
                if (++s == kPairStages) {
                    s = 0;
                    phase ^= 1;
                }
            }
        }
    producer_done:
        // never leave with copies in flight
        {
            const uint32_t n = issued < kPairStages ? issued : kPairStages;
            for (uint32_t i = 0; i < n; ++i) {
                s = (s == 0) ? kPairStages - 1 : s - 1;
                if (s == kPairStages - 1)
                    phase ^= 1;
                mbar_wait(&ctl->full[s], phase, ws, nullptr);
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 1) {
        // ------------------------------ odd CTA: forward "stage landed" ----
        uint32_t s = 0, phase = 0;
        for (uint32_t t = cluster; t < ntiles && !*abort; t += nclusters) {
            for (uint32_t ks = 0; ks < kstages; ++ks) {
                if (!mbar_wait(&ctl->full[s], phase, ws, abort))
                    goto relay_done;
                mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&ctl->peer_full[s]), 0));
                if (++s == kPairStages) {
                    s = 0;
                    phase ^= 1;
                }
            }
        }
    relay_done:;
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ------------------------------------------------------ MMA issuer ----
        const uint32_t base = smem_u32(smem);
        const uint64_t a_desc = smem_desc(base, 16, 1024, kSwizzle128B);
        const uint64_t b_desc = smem_desc(base + kPA, 16, 1024, kSwizzle128B);
        const uint64_t sfa_desc = smem_desc(base + kPA + kPB, 0, 128, kSwizzleNone);
        const uint64_t sfb_desc = smem_desc(base + kPA + kPB + kPSfa, 0, 128, kSwizzleNone);
        constexpr uint32_t kStageDesc = kPStage >> 4;
        constexpr uint16_t kBoth = 0x3;
        uint32_t s = 0, phase = 0, titer = 0, slot = 0;
        for (uint32_t t = cluster; t < ntiles && !*abort; t += nclusters, ++titer) {
            if (titer > 0 && !mbar_wait(&ctl->tmem_empty, (titer - 1) & 1, ws, abort))
                break;
            tc_fence_after();
            for (uint32_t ks = 0; ks < kstages; ++ks) {
                if (!mbar_wait(&ctl->full[s], phase, ws, abort) ||
                    !mbar_wait(&ctl->peer_full[s], phase, ws, abort))
                    goto mma_done;
                tc_fence_after();
                const uint64_t off = (uint64_t)(s * kStageDesc);
                const uint32_t sfa_t = tmem + kPAccCols + slot * kPSfStride;
                slot = slot + 1 == kPSfSlots ? 0 : slot + 1;
                const uint32_t sfb_t = sfa_t + 16;
                const uint32_t k_left = (uint32_t)args.K - ks * PK;
                const uint32_t kk = k_left >= PK ? 4u : (k_left + 63) / 64;
                if (kk == 4) {
#pragma unroll
                    for (uint32_t j = 0; j < 4; ++j) {
                        tmem_cp_32x128b_x4_pair(sfa_t + 4 * j, sfa_desc + off + 32 * j);
                        tmem_cp_32x128b_x4_pair(sfb_t + 8 * j, sfb_desc + off + 32 * j);
                        tmem_cp_32x128b_x4_pair(sfb_t + 8 * j + 4, sfb_desc + off + 128 + 32 * j);
                    }
#pragma unroll
                    for (uint32_t j = 0; j < 4; ++j)
                        pair_mma<kMx>(tmem, a_desc + off + 2 * j, b_desc + off + 2 * j, sfa_t + 4 * j, sfb_t + 8 * j,
                                      (ks | j) != 0 ? 1u : 0u);
                } else {
                    // last stage: the final K = 64 step possibly half filled
                    // (codes past K read as zeros, their scales are padding)
                    for (uint32_t j = 0; j < kk; ++j) {
                        tmem_cp_32x128b_x4_pair(sfa_t + 4 * j, sfa_desc + off + 32 * j);
                        tmem_cp_32x128b_x4_pair(sfb_t + 8 * j, sfb_desc + off + 32 * j);
                        tmem_cp_32x128b_x4_pair(sfb_t + 8 * j + 4, sfb_desc + off + 128 + 32 * j);
                    }
                    for (uint32_t j = 0; j < kk; ++j)
                        pair_mma<kMx>(tmem, a_desc + off + 2 * j, b_desc + off + 2 * j, sfa_t + 4 * j, sfb_t + 8 * j,
                                      (ks | j) != 0 ? 1u : 0u);
                }
                tc_commit_pair_multicast(&ctl->empty[s], kBoth);
                if (++s == kPairStages) {
                    s = 0;
                    phase ^= 1;
                }
            }
            tc_commit_pair_multicast(&ctl->tmem_full, kBoth);
        }
    mma_done:
        // all tensor-core work issued by this thread completes before teardown
        tc_commit_pair(&ctl->drain);
        mbar_wait(&ctl->drain, 0, ws, nullptr);
    } else if (warp >= 2) {
        // -------------------------------------------------------- epilogue ----
        const uint32_t q = warp & 3;            // tensor-memory lane quarter of this warp
        const uint32_t half = (warp - 2) >> 2;  // columns 128*half .. +127
        const float alpha = kMx ? 1.0f : __fmul_rn(*args.ga, *args.gb);
        const uint32_t empty_addr = mapa_shared(smem_u32(&ctl->tmem_empty), 0);
        uint32_t titer = 0;
        for (uint32_t t = cluster; t < ntiles && !*abort; t += nclusters, ++titer) {
            const uint32_t tm = t % tiles_m, tn = t / tiles_m;
            if (!mbar_wait(&ctl->tmem_full, titer & 1, ws, abort))
                break;
            tc_fence_after();
            const int32_t c0 = (int32_t)(tn * PN + half * 128);
            const uint32_t taddr = tmem + ((q * 32) << 16) + half * 128;
            uint32_t r[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld_32x32b_x32(taddr + c * 32, r[c]);
            tmem_ld_wait();
            // this CTA's accumulator is free once every load has landed
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster_relaxed(empty_addr);
            if (c0 >= args.N)
                continue;
            const int32_t row0 = (int32_t)(tm * PM + rank * 128 + q * 32);
            if (row0 >= args.M)
                continue;
            epilogue_store(r, alpha, row0, c0, args, store_buf + (warp - 2) * kStoreBufBytes, &tma_d, lane);
        }
        if (lane == 0)
            bulk_wait_all();
    }

    __syncthreads();
    // the even CTA's MMAs read this CTA's shared memory and write its tensor
    // memory: neither CTA frees anything before both are done
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, kPTmemCols);
    }
}

}  // namespace

nvfp4_status launch_gemm_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md,
                              const GemmArgs& args, bool mx, Workspace* ws, cudaStream_t stream)
{
    CUtensorMap msfa, msfb;
    if (!encode_sf_atom_map(&msfa, args.sfa, args.M, args.K, 1) ||
        !encode_sf_atom_map(&msfb, args.sfb, args.N, args.K, 2))
        return NVFP4_ERR_CUDA;
    static bool attr_set[2][64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    const void* kern = mx ? (const void*)nvf4_gemm_pair_kernel<true> : (const void*)nvf4_gemm_pair_kernel<false>;
    if (dev < 64 && !attr_set[mx][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmemBytes) !=
            cudaSuccess)
            return NVFP4_ERR_CUDA;
        attr_set[mx][dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int max_clusters = 0;
    cfg.gridDim = dim3(2, 1, 1);
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess || max_clusters < 1)
        return NVFP4_ERR_CUDA;
    const int64_t ntiles = ((int64_t)(args.M + PM - 1) / PM) * ((args.N + PN - 1) / PN);
    const int64_t clusters = ntiles < max_clusters ? ntiles : max_clusters;
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    cudaError_t e = mx ? cudaLaunchKernelEx(&cfg, nvf4_gemm_pair_kernel<true>, ma, mb, msfa, msfb, md, args, ws)
                       : cudaLaunchKernelEx(&cfg, nvf4_gemm_pair_kernel<false>, ma, mb, msfa, msfb, md, args, ws);
    return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
