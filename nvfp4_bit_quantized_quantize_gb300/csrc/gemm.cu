// Block-scaled NVFP4 GEMM on the sm_103a tensor cores ("Entrenamiento ...",
// "El Desafío de la Precisión de 4 Bits": NVFP4 runs on Blackwell tensor
// cores).
//
//   D[m, n] = ga * gb * sum_k A(m, k) * B(n, k)
//
// A [M, K] and B [N, K] are packed E2M1 codes (K contiguous) with one E4M3
// scale per 16 elements in the 128 x 4 atom layout.  Ragged M, N and K are
// padded on chip: tensor loads past the edges read zeros, the scale buffers'
// padding (zero, as the quantizers write it) covers the last atoms, and
// output chunks that cross M or N are written with plain stores of the
// elements inside M x N.
//
// Two kernels: the paired-SM kernel at the end of this file (256 x 256 tiles
// on two SMs, tcgen05 cta_group::2) runs every matrix of more than 128 rows
// and every call that wants the output maxima; the one-SM kernel here
// (128 x 256 tiles) runs the rest.  In the one-SM kernel each CTA owns a
// persistent sequence of 128 x 256 output tiles:
//   warp 0  TMA producer: A/B tiles (128-byte swizzle) and the scale atoms
//           (3-D tensor boxes of 4 atoms) into a 4-stage shared-memory ring;
//   warp 1  allocates tensor memory and issues tcgen05.mma.kind::mxf4nvf4
//           (K = 64 per instruction, binary32 accumulator in tensor memory);
//   warps 2-9 epilogue, two per tensor-memory lane quarter (128 columns
//           each): the accumulator read in two rounds of two tcgen05.ld and
//           one wait, times ga*gb and rounded to bf16 pairs, the accumulator
//           released, then 32-row chunks staged in a 1 KB shared buffer per
//           warp leave through TMA bulk tensor stores (per-thread 16-byte
//           global stores measured a third slower); binary32 output goes out
//           in four rounds of one load, each stored before the next;
//   warps 10-13 one per tensor-memory lane quarter: write each stage's scale
//           atoms from shared memory into that quarter's lanes with
//           tcgen05.st (every quarter holds the four 32-row groups of an atom,
//           the layout the MMA reads), wait for the stores and signal the
//           MMA warp.  (Issued by the MMA thread's single lane, a tcgen05.cp
//           of the atoms cost the tensor pipe ~56 cycles per copy, three per
//           MMA; the paired kernel issues its copies under elect.sync, where
//           they cost next to nothing.  This kernel runs only matrices of at
//           most 128 rows and keeps the store path.)
// The MMA warp's issue loop is kept lean: every descriptor is a precomputed
// base plus a constant offset, the four K = 64 steps of a stage are unrolled.
// Every wait is bounded; a wait that runs out records NVFP4_ERR_TIMEOUT and
// all roles wind down, drain their asynchronous work, and free tensor memory.
#include "gemm_common.cuh"

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
constexpr int kEpilogueWarps = 8;
constexpr int kScaleWarps = 4;
constexpr int kFirstScaleWarp = 2 + kEpilogueWarps;
constexpr int kThreads = (2 + kEpilogueWarps + kScaleWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = BN;             // fp32 accumulator: 128 lanes x 256 columns
constexpr uint32_t kSfColsPerStage = 16 + 32; // SFA 4 steps x 4 cols, SFB 4 steps x 8 cols
constexpr uint32_t kSfSlotStride = 64;        // scale slots on 64-column boundaries

static_assert(kStageBytes % 1024 == 0, "stage alignment");
static_assert(kSfColsPerStage <= kSfSlotStride, "scale slot");
static_assert(kAccCols + kStages * kSfSlotStride <= kTmemCols, "tensor memory budget");

struct GemmCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t sf_ready[kStages];  // scale atoms of the stage are in tensor memory
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kEpilogueWarps * kStoreBufBytes + sizeof(GemmCtl);

constexpr uint32_t kIdescNvf4 = mma_idesc<false>(BM, BN);
constexpr uint32_t kIdescMxf4 = mma_idesc<true>(BM, BN);

template <bool kMx>
__device__ __forceinline__ void mma_step(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t sfa, uint32_t sfb,
                                         uint32_t acc)
{
    if constexpr (kMx)
        mma_mxf4(d, adesc, bdesc, kIdescMxf4, sfa, sfb, acc);
    else
        mma_nvf4(d, adesc, bdesc, kIdescNvf4, sfa, sfb, acc);
}

// kMx = false: NVFP4 (E4M3 block-16 scales, D scaled by ga * gb);
// kMx = true: MXFP4 (UE8M0 block-32 scales, no tensor scale).  The scale
// buffers have the same shape in both: one 32-bit word per row per K = 64.
template <bool kMx>
__global__ void __launch_bounds__(kThreads, 1)
    nvf4_gemm_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                     const __grid_constant__ CUtensorMap tma_sfa, const __grid_constant__ CUtensorMap tma_sfb,
                     const __grid_constant__ CUtensorMap tma_d, const GemmArgs args, Workspace* ws)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* store_buf = smem + (size_t)kStages * kStageBytes;
    GemmCtl* ctl = reinterpret_cast<GemmCtl*>(store_buf + kEpilogueWarps * kStoreBufBytes);
    volatile int* abort = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tiles_m = ((uint32_t)args.M + BM - 1) / BM;
    const uint32_t tiles_n = ((uint32_t)args.N + BN - 1) / BN;
    const uint32_t ntiles = tiles_m * tiles_n;
    const uint32_t kstages = ((uint32_t)args.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
            mbar_init(&ctl->sf_ready[s], kScaleWarps);
        }
        mbar_init(&ctl->tmem_full, 1);
        mbar_init(&ctl->tmem_empty, kEpilogueWarps);
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
        tma_prefetch_desc(&tma_sfa);
        tma_prefetch_desc(&tma_sfb);
        uint32_t s = 0, phase = 0, issued = 0;
        for (uint32_t t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x) {
            const uint32_t tm = t % tiles_m, tn = t / tiles_m;
            const int32_t m0 = (int32_t)(tm * BM), n0 = (int32_t)(tn * BN);
            for (uint32_t ks = 0; ks < kstages; ++ks) {
                if (issued >= kStages && !mbar_wait(&ctl->empty[s], phase ^ 1, ws, abort))
                    goto producer_done;
                uint8_t* st = smem + (size_t)s * kStageBytes;
                // boxes past M, N or K read as zeros and still count in full
                mbar_expect_tx(&ctl->full[s], kStageBytes);
                tma_load_2d(st, &tma_a, &ctl->full[s], (int32_t)(ks * 128), m0);
                tma_load_2d(st + kABytes, &tma_b, &ctl->full[s], (int32_t)(ks * 128), n0);
                tma_load_3d(st + kABytes + kBBytes, &tma_sfa, &ctl->full[s], 0, (int32_t)(ks * 4), (int32_t)tm);
                tma_load_3d(st + kABytes + kBBytes + kSfaBytes, &tma_sfb, &ctl->full[s], 0, (int32_t)(ks * 4),
                            (int32_t)(2 * tn));
                ++issued;
                if (++s == kStages) {
                    s = 0;
                    phase ^= 1;
                }
            }
        }
    producer_done:
        // never leave with copies in flight: wait for the last kStages loads
        {
            const uint32_t n = issued < kStages ? issued : kStages;
            for (uint32_t i = 0; i < n; ++i) {
                s = (s == 0) ? kStages - 1 : s - 1;
                if (s == kStages - 1)
                    phase ^= 1;
                mbar_wait(&ctl->full[s], phase, ws, nullptr);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------ MMA issuer ----
        const uint32_t base = smem_u32(smem);
        const uint64_t a_desc = smem_desc(base, 16, 1024, kSwizzle128B);
        const uint64_t b_desc = smem_desc(base + kABytes, 16, 1024, kSwizzle128B);
        constexpr uint32_t kStageDesc = kStageBytes >> 4;  // stage stride in descriptor units
        uint32_t s = 0, phase = 0, titer = 0;
        for (uint32_t t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x, ++titer) {
            if (titer > 0 && !mbar_wait(&ctl->tmem_empty, (titer - 1) & 1, ws, abort))
                break;
            tc_fence_after();
            for (uint32_t ks = 0; ks < kstages; ++ks) {
                // the scale warps saw the stage's loads complete before they signalled
                if (!mbar_wait(&ctl->sf_ready[s], phase, ws, abort))
                    goto mma_done;
                tc_fence_after();
                const uint64_t off = (uint64_t)(s * kStageDesc);
                const uint32_t sfa_t = tmem + kAccCols + s * kSfSlotStride;
                const uint32_t sfb_t = sfa_t + 16;
                const uint32_t k_left = (uint32_t)args.K - ks * BK;
                if (k_left >= BK) {
#pragma unroll
                    for (uint32_t j = 0; j < 4; ++j)
                        mma_step<kMx>(tmem, a_desc + off + 2 * j, b_desc + off + 2 * j, sfa_t + 4 * j,
                                      sfb_t + 8 * j, (ks | j) != 0 ? 1u : 0u);
                } else {
                    // last stage: K = 64 steps, the final one possibly half
                    // filled (codes past K read as zeros, their scales are the
                    // zero padding of the last atom)
                    const uint32_t kk = (k_left + 63) / 64;
                    for (uint32_t j = 0; j < kk; ++j)
                        mma_step<kMx>(tmem, a_desc + off + 2 * j, b_desc + off + 2 * j, sfa_t + 4 * j,
                                      sfb_t + 8 * j, (ks | j) != 0 ? 1u : 0u);
                }
                tc_commit(&ctl->empty[s]);
                if (++s == kStages) {
                    s = 0;
                    phase ^= 1;
                }
            }
            tc_commit(&ctl->tmem_full);
        }
    mma_done:
        // all tensor-core work issued by this thread completes before teardown
        tc_commit(&ctl->drain);
        mbar_wait(&ctl->drain, 0, ws, nullptr);
    } else if (warp >= 2 && warp < kFirstScaleWarp) {
        // -------------------------------------------------------- epilogue ----
        const uint32_t q = warp & 3;             // tensor-memory lane quarter of this warp
        const uint32_t half = (warp - 2) >> 2;   // columns 128*half .. +127
        const float alpha = kMx ? 1.0f : __fmul_rn(*args.ga, *args.gb);
        uint32_t titer = 0;
        for (uint32_t t = blockIdx.x; t < ntiles && !*abort; t += gridDim.x, ++titer) {
            const uint32_t tm = t % tiles_m, tn = t / tiles_m;
            if (!mbar_wait(&ctl->tmem_full, titer & 1, ws, abort))
                break;
            tc_fence_after();
            const int32_t c0 = (int32_t)(tn * BN + half * 128);
            const int32_t row0 = (int32_t)(tm * BM + q * 32);
            const bool live = c0 < args.N && row0 < args.M;
            uint8_t* buf = store_buf + (warp - 2) * kStoreBufBytes;
            const uint32_t taddr = tmem + ((q * 32) << 16) + half * 128;
            if (args.out_f32) {
                // binary32 output: each 32-column round goes out before the next load
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + h * 32, r);
                    tmem_ld_wait();
                    if (live)
                        epilogue_store_f32(r, alpha, row0, c0 + h * 32, args, buf, &tma_d, lane);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ctl->tmem_empty);
            } else {
                // two rounds of two loads and one wait, packed to bf16 pairs
                uint32_t p[64];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t ra[32], rb[32];
                    tmem_ld_32x32b_x32(taddr + h * 64, ra);
                    tmem_ld_32x32b_x32(taddr + h * 64 + 32, rb);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        p[h * 32 + e] = pack_bf16x2(__fmul_rn(__uint_as_float(ra[2 * e]), alpha),
                                                    __fmul_rn(__uint_as_float(ra[2 * e + 1]), alpha));
                        p[h * 32 + 16 + e] = pack_bf16x2(__fmul_rn(__uint_as_float(rb[2 * e]), alpha),
                                                         __fmul_rn(__uint_as_float(rb[2 * e + 1]), alpha));
                    }
                }
                // the accumulator is free once every load has landed in registers
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ctl->tmem_empty);
                if (live)
                    epilogue_store_bf16(p, row0, c0, args, buf, &tma_d, lane);
            }
        }
        // (the lane that committed the stores: the elected one)
        if (elect_one())
            bulk_wait_all();
    } else if (warp >= kFirstScaleWarp) {
        // ----------------------------------------------------- scale warps ----
        // Stage layout: A's 4 atoms (steps 0..3), then B's row tile 0 steps
        // 0..3 and row tile 1 steps 0..3, 512 bytes each.  Lane i takes row i
        // (16 bytes) of every atom: tensor-memory columns slot + 4j .. + 3
        // for A's step j and slot + 16 + 8j .. + 7 for B's step j (tile 0,
        // then tile 1), in its quarter's lanes.
        const uint32_t q = warp & 3;
        const uint32_t lanes = (q * 32) << 16;
        uint32_t s = 0, phase = 0;
        for (uint32_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            for (uint32_t ks = 0; ks < kstages; ++ks) {
                int ok = 1;
                if (lane == 0)
                    ok = mbar_wait(&ctl->full[s], phase, ws, abort);
                if (!__shfl_sync(0xFFFFFFFFu, ok, 0))
                    goto scales_done;
                const uint8_t* sfa_s = smem + (size_t)s * kStageBytes + kABytes + kBBytes + lane * 16;
                const uint8_t* sfb_s = sfa_s + kSfaBytes;
                uint32_t v[48];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 a = *reinterpret_cast<const uint4*>(sfa_s + j * 512);
                    const uint4 b0 = *reinterpret_cast<const uint4*>(sfb_s + j * 512);
                    const uint4 b1 = *reinterpret_cast<const uint4*>(sfb_s + (4 + j) * 512);
                    v[4 * j] = a.x;
                    v[4 * j + 1] = a.y;
                    v[4 * j + 2] = a.z;
                    v[4 * j + 3] = a.w;
                    v[16 + 8 * j] = b0.x;
                    v[16 + 8 * j + 1] = b0.y;
                    v[16 + 8 * j + 2] = b0.z;
                    v[16 + 8 * j + 3] = b0.w;
                    v[16 + 8 * j + 4] = b1.x;
                    v[16 + 8 * j + 5] = b1.y;
                    v[16 + 8 * j + 6] = b1.z;
                    v[16 + 8 * j + 7] = b1.w;
                }
                const uint32_t slot = tmem + lanes + kAccCols + s * kSfSlotStride;
                tmem_st_32x32b_x16(slot, v);
                tmem_st_32x32b_x16(slot + 16, v + 16);
                tmem_st_32x32b_x16(slot + 32, v + 32);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ctl->sf_ready[s]);
                if (++s == kStages) {
                    s = 0;
                    phase ^= 1;
                }
            }
        }
    scales_done:;
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ============================================================ paired SMs ====
// The same GEMM on two SMs per output tile (tcgen05 cta_group::2): a cluster
// of two CTAs computes a 256 x 256 tile with one M = 256, N = 256, K = 64 MMA
// per step, issued by the even CTA.  Each CTA stages its own 128 rows of A,
// its own 128 rows of B (the tensor cores exchange the B halves), its A rows'
// scale atoms and the atoms of all 256 B rows, so each SM receives 38 KB per
// K = 256 stage instead of the one-SM kernel's 54 KB for the same work, and
// the freed shared memory holds a fifth stage.  Each CTA's tensor memory holds
// the accumulator of its 128 A rows (256 columns) and five scale slots, one
// per ring stage.
//   warp 0     TMA producer (both CTAs): this CTA's A and B boxes and scale
//              atoms of each stage; the bytes of both CTAs complete on the
//              even CTA's `full` barrier of the stage (the .cta_group::2 form
//              of the tensor copy), which expects both;
//   warp 1     tensor-memory allocation (collective over the pair); in the
//              even CTA, the MMA warp: per stage, once `full` says that both
//              CTAs' stage landed, one elected lane copies the scale atoms
//              into the stage's tensor-memory slot with tcgen05.cp (in both
//              CTAs) and issues the MMAs, three copies before each MMA, then
//              commits the stage free to both CTAs' producers;
//   warps 2-9  epilogue, as in the one-SM kernel.
// Every asynchronous instruction goes out from one elected lane of a warp
// that runs its loop together (lane 0 waits on the barriers): the producer's
// tensor copies, the MMA warp's scale copies, MMAs and commits, the
// epilogue's bulk stores.  Issued by one lane inside a divergent branch,
// every scale copy cost the tensor pipe ~40-56 cycles (the kernel ran at half
// speed) and the producer's copies went out measurably slower.  A stage's
// scale slot is rewritten only after the stage's next `full`, which the
// producer armed after the MMAs that read the slot had completed.
// Stage-free and accumulator-full signals reach both CTAs through the
// multicast form of tcgen05.commit; the odd CTA's drained-accumulator signals
// reach the even CTA by remote mbarrier arrives with the default (CTA-scope
// release) semantics: what they report was completed by an earlier wait of
// the arriving thread (tcgen05.wait::ld, then tcgen05.fence::before_thread_sync),
// and a cluster-scope release on these arrives halved the kernel's speed.
// Every wait is bounded.  The MMA warp's loops always run to their end (a
// wait that fails sets the abort flag, after which every later wait returns
// at once and the remaining MMAs read valid, stale operands), so no branch in
// the issuing loop depends on a wait.  A cluster barrier keeps both CTAs
// (whose shared and tensor memory the MMAs use) alive until all tensor-core
// work is done; after a failed wait, every CTA first gives the tensor copies
// it may have in flight time to land.

// One 128 x 4 scale atom (32 rows x 16 bytes of shared memory, every row
// holding the 4 scales of rows r, r + 32, r + 64, r + 96) into 4 columns of
// all four lane quarters of tensor memory, in both CTAs of the pair (each
// CTA's own shared memory into its own tensor memory): the layout the
// block-scaled MMA reads.
__device__ __forceinline__ void tmem_cp_pair_atom(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

constexpr int PM = 256;
constexpr int PN = 256;
constexpr int kPA = 128 * BK / 2;              // 16 KB: this CTA's 128 rows of A
constexpr int kPB = 128 * BK / 2;              // 16 KB: this CTA's 128 rows of B
constexpr int kPStage = kPA + kPB + kSfaBytes + kSfbBytes;
constexpr int kPStages = 5;                    // shared-memory ring (5 x 38 KB)
constexpr uint32_t kPSlotStride = 48;          // scale slot: A's 4 steps x 4 columns, B's 4 steps x 8
constexpr int kPThreads = (2 + kEpilogueWarps) * 32;  // producer, MMA, epilogue (no scale warps)

struct PairCtl {
    uint64_t full[kPStages];      // even CTA: both CTAs' stage landed (A, B, scale atoms)
    uint64_t empty[kPStages];     // the stage's MMAs are done (multicast commit)
    uint64_t tmem_full;
    uint64_t tmem_empty;          // even CTA: both CTAs drained the accumulator (16 arrivals)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kPSmemBytes = 1024 + (size_t)kPStages * kPStage + kEpilogueWarps * kWideBufBytes + sizeof(PairCtl);
static_assert(kPStage % 1024 == 0, "stage alignment");
static_assert(kAccCols + kPStages * kPSlotStride <= kTmemCols, "tensor memory budget");
static_assert(kPSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kStoreBufBytes + kRhtBufBytes <= kWideBufBytes, "epilogue buffer: bf16 chunk + Hadamard scratch");

constexpr uint32_t kIdescNvf4Pair = mma_idesc<false>(PM, PN);
constexpr uint32_t kIdescMxf4Pair = mma_idesc<true>(PM, PN);

template <bool kMx>
__device__ __forceinline__ void mma_step_pair(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t sfa, uint32_t sfb,
                                              uint32_t acc)
{
    if constexpr (kMx)
        mma_mxf4_pair(d, adesc, bdesc, kIdescMxf4Pair, sfa, sfb, acc);
    else
        mma_nvf4_pair(d, adesc, bdesc, kIdescNvf4Pair, sfa, sfb, acc);
}

template <bool kMx>
__global__ void __maxnreg__(128)
    nvf4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                          const __grid_constant__ CUtensorMap tma_sfa, const __grid_constant__ CUtensorMap tma_sfb,
                          const __grid_constant__ CUtensorMap tma_d, const GemmArgs args, Workspace* ws)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* store_buf = smem + (size_t)kPStages * kPStage;
    PairCtl* ctl = reinterpret_cast<PairCtl*>(store_buf + kEpilogueWarps * kWideBufBytes);
    volatile int* abort = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: the CTA that issues the MMAs
    const uint32_t cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const uint32_t tiles_m = ((uint32_t)args.M + PM - 1) / PM;
    const uint32_t tiles_n = ((uint32_t)args.N + PN - 1) / PN;
    const uint32_t ntiles = tiles_m * tiles_n;
    const uint32_t kstages = ((uint32_t)args.K + BK - 1) / BK;
    // this cluster's tiles are cluster, cluster + nclusters, ...; iteration i
    // of every role is K stage i % kstages of its (i / kstages)-th tile
    const uint32_t my_tiles = (ntiles - cluster + nclusters - 1) / nclusters;
    const uint32_t iters = my_tiles * kstages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->tmem_full, 1);
        mbar_init(&ctl->tmem_empty, 2 * kEpilogueWarps);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
        tc_fence_before();
    }
    __syncthreads();
    // both CTAs' barriers are initialised before any remote arrive
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer ----
        // The whole warp runs the loop: lane 0 waits, one elected lane issues
        // (a lone lane in a divergent branch issued the copies measurably
        // slower).
        if (elect_one()) {
            tma_prefetch_desc(&tma_a);
            tma_prefetch_desc(&tma_b);
            tma_prefetch_desc(&tma_sfa);
            tma_prefetch_desc(&tma_sfb);
        }
        __syncwarp();
        uint32_t ia = 0;  // stages issued
        for (; ia < iters; ++ia) {
            const uint32_t s = ia % kPStages;
            int ok = 1;
            if (lane == 0)
                ok = !*abort && (ia < kPStages || mbar_wait(&ctl->empty[s], ((ia / kPStages) - 1) & 1, ws, abort));
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0))
                break;
            const uint32_t t = cluster + (ia / kstages) * nclusters, ks = ia % kstages;
            const uint32_t tm = t % tiles_m, tn = t / tiles_m;
            const uint32_t arow = 2 * tm + rank;   // this CTA's 128-row tile of A
            uint8_t* st = smem + (size_t)s * kPStage;
            // boxes past M, N or K read as zeros and still count in full; both
            // CTAs' bytes complete on the even CTA's barrier, armed by the even
            // CTA for both (a byte count may arrive before the arming: the
            // phase completes only with its one arrival and a zero count)
            const uint32_t bar = mapa_shared(smem_u32(&ctl->full[s]), 0);
            if (elect_one()) {
                if (rank == 0)
                    mbar_expect_tx(&ctl->full[s], 2 * kPStage);
                tma_load_2d_pair(st, &tma_a, bar, (int32_t)(ks * 128), (int32_t)(arow * 128));
                tma_load_2d_pair(st + kPA, &tma_b, bar, (int32_t)(ks * 128), (int32_t)((2 * tn + rank) * 128));
                tma_load_3d_pair(st + kPA + kPB, &tma_sfa, bar, 0, (int32_t)(ks * 4), (int32_t)arow);
                tma_load_3d_pair(st + kPA + kPB + kSfaBytes, &tma_sfb, bar, 0, (int32_t)(ks * 4), (int32_t)(2 * tn));
            }
            __syncwarp();
        }
        // never leave with copies in flight: the even CTA's barriers count
        // both CTAs' copies of the stages it armed (after a failed wait the
        // settle below covers the rest)
        if (rank == 0 && lane == 0)
            for (uint32_t k = ia > kPStages ? ia - kPStages : 0; k < ia; ++k)
                mbar_wait(&ctl->full[k % kPStages], (k / kPStages) & 1, ws, abort);
        __syncwarp();
    } else if (warp == 1 && rank == 0) {
        // ------------------------------------------------------- MMA warp ----
        const uint32_t base = smem_u32(smem);
        const uint64_t a_desc = smem_desc(base, 16, 1024, kSwizzle128B);
        const uint64_t b_desc = smem_desc(base + kPA, 16, 1024, kSwizzle128B);
        // scale atoms: 512-byte blocks of 32 rows x 16 bytes, no swizzle
        const uint64_t sf_desc = smem_desc(base + kPA + kPB, 0, 128, 0);
        constexpr uint32_t kStageDesc = kPStage >> 4;  // stage stride in descriptor units
        constexpr uint32_t kSfbDesc = kSfaBytes >> 4;  // B's atoms after A's
        constexpr uint32_t kAtomDesc = 512 >> 4;
        constexpr uint16_t kBoth = 0x3;
        uint32_t i = 0;
        for (uint32_t n = 0; n < my_tiles; ++n) {
            if (n > 0) {
                if (lane == 0)
                    mbar_wait(&ctl->tmem_empty, (n - 1) & 1, ws, abort);
                __syncwarp();
            }
            tc_fence_after();
            for (uint32_t ks = 0; ks < kstages; ++ks, ++i) {
                const uint32_t s = i % kPStages;
                if (lane == 0)
                    mbar_wait(&ctl->full[s], (i / kPStages) & 1, ws, abort);
                __syncwarp();
                tc_fence_after();
                const uint64_t off = (uint64_t)(s * kStageDesc);
                const uint64_t sfa_src = sf_desc + off, sfb_src = sfa_src + kSfbDesc;
                const uint32_t sfa_t = tmem + kAccCols + s * kPSlotStride;
                const uint32_t sfb_t = sfa_t + 16;
                const uint32_t k_left = (uint32_t)args.K - ks * BK;
                const uint32_t kk = k_left >= BK ? 4u : (k_left + 63) / 64;
                if (elect_one()) {
                    // K step j: A's atom j into columns 4j, B's row tiles' atoms
                    // j (rows 0-127) and 4 + j (rows 128-255) into 8j and 8j + 4
                    if (kk == 4) {
#pragma unroll
                        for (uint32_t j = 0; j < 4; ++j) {
                            tmem_cp_pair_atom(sfa_t + 4 * j, sfa_src + kAtomDesc * j);
                            tmem_cp_pair_atom(sfb_t + 8 * j, sfb_src + kAtomDesc * j);
                            tmem_cp_pair_atom(sfb_t + 8 * j + 4, sfb_src + kAtomDesc * (4 + j));
                            mma_step_pair<kMx>(tmem, a_desc + off + 2 * j, b_desc + off + 2 * j, sfa_t + 4 * j,
                                               sfb_t + 8 * j, (ks | j) != 0 ? 1u : 0u);
                        }
                    } else {
                        for (uint32_t j = 0; j < kk; ++j) {
                            tmem_cp_pair_atom(sfa_t + 4 * j, sfa_src + kAtomDesc * j);
                            tmem_cp_pair_atom(sfb_t + 8 * j, sfb_src + kAtomDesc * j);
                            tmem_cp_pair_atom(sfb_t + 8 * j + 4, sfb_src + kAtomDesc * (4 + j));
                            mma_step_pair<kMx>(tmem, a_desc + off + 2 * j, b_desc + off + 2 * j, sfa_t + 4 * j,
                                               sfb_t + 8 * j, (ks | j) != 0 ? 1u : 0u);
                        }
                    }
                    tc_commit_pair_multicast(&ctl->empty[s], kBoth);
                }
                __syncwarp();
            }
            if (elect_one())
                tc_commit_pair_multicast(&ctl->tmem_full, kBoth);
            __syncwarp();
        }
        // all tensor-core work issued by this warp completes before teardown
        // (elect.sync picks the same lane as above: the commit covers it)
        if (elect_one()) {
            tc_commit_pair_multicast(&ctl->drain, 0x1);
            mbar_wait(&ctl->drain, 0, ws, nullptr);
        }
        __syncwarp();
    } else if (warp >= 2 && warp < kFirstScaleWarp) {
        // -------------------------------------------------------- epilogue ----
        const uint32_t q = warp & 3;             // tensor-memory lane quarter of this warp
        const uint32_t half = (warp - 2) >> 2;   // columns 128*half .. +127
        const float alpha = kMx ? 1.0f : __fmul_rn(*args.ga, *args.gb);
        const uint32_t empty_addr = mapa_shared(smem_u32(&ctl->tmem_empty), 0);
        const bool amax_on = !kMx && args.amax_out != nullptr;
        uint32_t* rbuf = reinterpret_cast<uint32_t*>(store_buf + (warp - 2) * kWideBufBytes + kStoreBufBytes);
        uint32_t rmax = 0;
        float tmax = 0.0f;
        for (uint32_t n = 0; n < my_tiles && !*abort; ++n) {
            const uint32_t t = cluster + n * nclusters;
            const uint32_t tm = t % tiles_m, tn = t / tiles_m;
            if (!mbar_wait(&ctl->tmem_full, n & 1, ws, abort))
                break;
            tc_fence_after();
            const int32_t c0 = (int32_t)(tn * PN + half * 128);
            const int32_t row0 = (int32_t)(tm * PM + rank * 128 + q * 32);
            const bool live = c0 < args.N && row0 < args.M;
            uint8_t* buf = store_buf + (warp - 2) * kWideBufBytes;
            const uint32_t taddr = tmem + ((q * 32) << 16) + half * 128;
            if (args.out_f32) {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + h * 32, r);
                    tmem_ld_wait();
                    if (live)
                        epilogue_store_f32_wide(r, alpha, row0, c0 + h * 32, args, buf, &tma_d, lane);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_remote(empty_addr);
            } else {
                uint32_t p[64];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t ra[32], rb[32];
                    tmem_ld_32x32b_x32(taddr + h * 64, ra);
                    tmem_ld_32x32b_x32(taddr + h * 64 + 32, rb);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        p[h * 32 + e] = pack_bf16x2(__fmul_rn(__uint_as_float(ra[2 * e]), alpha),
                                                    __fmul_rn(__uint_as_float(ra[2 * e + 1]), alpha));
                        p[h * 32 + 16 + e] = pack_bf16x2(__fmul_rn(__uint_as_float(rb[2 * e]), alpha),
                                                         __fmul_rn(__uint_as_float(rb[2 * e + 1]), alpha));
                    }
                }
                // this CTA's accumulator is free once every load has landed
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_remote(empty_addr);
                // (with the output maxima, folded in as the chunks leave)
                if (live && amax_on)
                    epilogue_store_bf16_amax(p, row0, c0, args, buf, rbuf, &tma_d, lane, rmax, tmax);
                else if (live)
                    epilogue_store_bf16(p, row0, c0, args, buf, &tma_d, lane);
            }
        }
        // every epilogue warp reports, even one that stopped early
        if (amax_on)
            epilogue_amax_finish(rmax, tmax, args, ws, gridDim.x * kEpilogueWarps, lane);
        // (the lane that committed the stores: the elected one)
        if (elect_one())
            bulk_wait_all();
    }

    __syncthreads();
    // after a failed wait (here or in the peer CTA) tensor copies of this CTA
    // may still be in flight, their barrier never to complete: give them time
    // to land before the CTA's shared memory is released
    if (threadIdx.x == 0 && (*abort || ld_shared_cluster_u32(mapa_shared(smem_u32(&ctl->abort), rank ^ 1u))))
        __nanosleep(50000);
    // the even CTA's MMAs read this CTA's shared memory and write its tensor
    // memory: neither CTA frees anything before both are done
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace

nvfp4_status launch_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                         const uint8_t* sfb, const float* gb, int64_t M, int64_t N, int64_t K, void* d,
                         int64_t ldd, nvfp4_out_dtype dt, bool mx, float* amax_out, uint32_t rht_signs,
                         Workspace* ws, cudaStream_t stream)
{
    // 256-row pair tiles; a matrix of at most 128 rows would leave one SM of
    // every pair without A rows, so it runs on the one-SM kernel -- unless
    // the output maxima are wanted, which only the paired kernel reduces
    // (rows past M read as zeros there, so any M is correct on it)
    const bool pair = M > 128 || amax_out != nullptr;
    CUtensorMap ma, mb;
    if (!encode_tensor_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(a), (uint64_t)(K / 2),
                              (uint64_t)M, (uint64_t)(K / 2), 128u, (uint32_t)BM, CU_TENSOR_MAP_SWIZZLE_128B))
        return NVFP4_ERR_CUDA;
    if (!encode_tensor_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(b), (uint64_t)(K / 2),
                              (uint64_t)N, (uint64_t)(K / 2), 128u, pair ? 128u : (uint32_t)BN,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return NVFP4_ERR_CUDA;

    // output chunks: 32 rows x 32 bytes, except binary32 output of the
    // paired-SM kernel: 32 rows x 128 bytes in the 128-byte swizzle (that
    // epilogue holds the accumulator while it stores, so fewer, larger
    // stores free it sooner; for bf16 the small chunks measured faster)
    CUtensorMap md;
    const bool f32 = dt == NVFP4_OUT_F32;
    const bool wide = pair && f32;
    if (!encode_tensor_map_2d(&md, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d,
                              (uint64_t)N, (uint64_t)M, (uint64_t)ldd * (f32 ? 4u : 2u),
                              (wide ? 128u : 32u) / (f32 ? 4u : 2u), 32u,
                              wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE))
        return NVFP4_ERR_CUDA;
    GemmArgs args{sfa, sfb, ga, gb, d, ldd, (int32_t)M, (int32_t)N, (int32_t)K, dt == NVFP4_OUT_F32 ? 1 : 0,
                  amax_out, rht_signs};
    CUtensorMap msfa, msfb;
    if (!encode_sf_atom_map(&msfa, sfa, M, K, 1) || !encode_sf_atom_map(&msfb, sfb, N, K, 2))
        return NVFP4_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return NVFP4_ERR_CUDA;

    if (pair) {
        static bool attr_set[2][64] = {};
        static int max_clusters[2][64] = {};
        const void* kern = mx ? (const void*)nvf4_gemm_pair_kernel<true> : (const void*)nvf4_gemm_pair_kernel<false>;
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
        if (!attr_set[mx][dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmemBytes) !=
                cudaSuccess)
                return NVFP4_ERR_CUDA;
            cfg.gridDim = dim3(2, 1, 1);
            int mc = 0;
            if (cudaOccupancyMaxActiveClusters(&mc, kern, &cfg) != cudaSuccess || mc < 1)
                return NVFP4_ERR_CUDA;
            max_clusters[mx][dev] = mc;
            attr_set[mx][dev] = true;
        }
        const int64_t ntiles = ((M + PM - 1) / PM) * ((N + PN - 1) / PN);
        const int64_t clusters = ntiles < max_clusters[mx][dev] ? ntiles : max_clusters[mx][dev];
        cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
        const cudaError_t e =
            mx ? cudaLaunchKernelEx(&cfg, nvf4_gemm_pair_kernel<true>, ma, mb, msfa, msfb, md, args, ws)
               : cudaLaunchKernelEx(&cfg, nvf4_gemm_pair_kernel<false>, ma, mb, msfa, msfb, md, args, ws);
        return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
    }

    static bool attr_set[2][64] = {};
    const void* kern = mx ? (const void*)nvf4_gemm_kernel<true> : (const void*)nvf4_gemm_kernel<false>;
    if (!attr_set[mx][dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        attr_set[mx][dev] = true;
    }
    const int64_t ntiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int sms = device_sm_count();
    const int grid = (int)(ntiles < sms ? ntiles : sms);
    if (mx)
        nvf4_gemm_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(ma, mb, msfa, msfb, md, args, ws);
    else
        nvf4_gemm_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(ma, mb, msfa, msfb, md, args, ws);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
