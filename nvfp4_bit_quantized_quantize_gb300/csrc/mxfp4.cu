// MXFP4 quantizer: the comparison format the pages set against NVFP4
// ("I ricercatori di Nvidia sbloccano ...", section "Come funziona NVFP4?":
// MXFP4 needed markedly more training data for the same accuracy).  The pages
// name the format but do not define it; this follows the OCP Microscaling
// (MX) v1.0 specification: blocks of 32 contiguous elements, E2M1 elements,
// one UE8M0 (power-of-two) shared scale per block, no tensor-level scale.
//
//   shared exponent  e = floor(log2(max |x| over the block)) - 2  (2 = the
//                    largest E2M1 exponent), clamped to [-127, 127];
//   element code     E2M1 round-to-nearest-even of x / 2^e, saturating at 6;
//   scale byte       e + 127.
//
// A block whose max is 0 or below the smallest normal binary32 gets e = -127
// (byte 0).  A block holding Inf or NaN gets the UE8M0 NaN byte 0xFF and zero
// codes, and NVFP4_ERR_NONFINITE is recorded in the workspace.
//
// Layout: codes as for NVFP4 ([rows, cols/2], element 2i in the low nibble);
// scale bytes in the 128-row x 4-word atoms the block-scaled MMA reads, one
// 32-bit word per row per 64 elements holding the two block scales in bytes 0
// and 1 (bytes 2 and 3 zero): byte of (row r, block kb) at
//   ((r / 128) * Cp + kb / 2) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 2,
// Cp = ceil(cols / 64).
//
// No tensor amax, so one streaming pass: one warp per row at a time, one
// 32-element block per lane per step (the warp reads 2 KB of bf16 and writes
// 512 bytes of codes contiguously); lanes 2i and 2i+1 meet in one scale word.
// Rows up to the next multiple of 128 are visited too, to write the zero
// scale words of the padding rows.
#include "device.cuh"

namespace nvfp4 {
namespace {

constexpr int kMxThreads = 256;

struct MxArgs {
    const uint8_t* x;
    uint8_t* q;
    uint8_t* sf;
    Workspace* ws;
    int64_t rows;
    int64_t rows_pad;  // rows rounded up to the 128-row scale tile (padding rows get zero scale words)
    int64_t ld;        // elements
    uint32_t kblocks;  // cols / 32
    uint32_t cp;       // 64-element steps per row, rounded up
};

__global__ void __launch_bounds__(kMxThreads) mxfp4_quantize_kernel(const MxArgs a)
{
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = (int64_t)blockIdx.x * (kMxThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kMxThreads / 32);
    bool bad = false;
    for (int64_t r = gwarp; r < a.rows_pad; r += nwarps) {
        const bool row_live = r < a.rows;
        const uint32_t rr = (uint32_t)(r & 127);
        uint8_t* sf_row = a.sf + (r >> 7) * (int64_t)a.cp * 512 + (rr & 31) * 16 + (rr >> 5) * 4;
        // every lane of the warp runs the same number of steps (for the shuffle)
        for (uint32_t base = 0; base < a.kblocks; base += 32) {
            const uint32_t kb = base + (uint32_t)lane;
            const bool live = row_live && kb < a.kblocks;
            uint32_t w[16];
            if (live) {
                const uint4* xp = reinterpret_cast<const uint4*>(a.x + (r * a.ld + (int64_t)kb * 32) * 2);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = __ldcs(xp + i);
                    w[4 * i] = v.x;
                    w[4 * i + 1] = v.y;
                    w[4 * i + 2] = v.z;
                    w[4 * i + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = 0u;
            }
            uint32_t acc = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                acc = habs_max2(acc, w[i]);
            const uint32_t amax_bits = __float_as_uint(hmax_to_float(acc));
            uint32_t sb;
            uint4 c0 = make_uint4(0, 0, 0, 0);
            if (amax_bits >= 0x7F800000u) {
                sb = 0xFFu;  // UE8M0 NaN: the block holds Inf or NaN
                bad = bad || live;
            } else {
                // floor(log2 amax) = exponent field - 127 for normal amax;
                // scale byte = max(field - 2, 0) (zero/subnormal max -> 0)
                const uint32_t field = amax_bits >> 23;
                sb = field > 2u ? field - 2u : 0u;
                // 1 / 2^(sb - 127) = 2^(127 - sb): exponent field 254 - sb
                const float inv = __uint_as_float((254u - sb) << 23);
                uint32_t packed[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t* x = &w[4 * i];
                    packed[i] = e2m1x8_rn(__fmul_rn(bf16lo(x[0]), inv), __fmul_rn(bf16hi(x[0]), inv),
                                          __fmul_rn(bf16lo(x[1]), inv), __fmul_rn(bf16hi(x[1]), inv),
                                          __fmul_rn(bf16lo(x[2]), inv), __fmul_rn(bf16hi(x[2]), inv),
                                          __fmul_rn(bf16lo(x[3]), inv), __fmul_rn(bf16hi(x[3]), inv));
                }
                c0 = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            }
            if (live)
                *reinterpret_cast<uint4*>(a.q + r * (int64_t)a.kblocks * 16 + (int64_t)kb * 16) = c0;
            // lanes 2i and 2i+1 hold the two blocks of one 64-element step
            const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, sb, 1);
            if ((lane & 1) == 0 && kb < a.kblocks) {
                const uint32_t word = sb | ((kb + 1 < a.kblocks ? hi : 0u) << 8);
                *reinterpret_cast<uint32_t*>(sf_row + (int64_t)(kb >> 1) * 512) = word;
            }
        }
    }
    if (bad)
        record_status(a.ws, NVFP4_ERR_NONFINITE);
}

}  // namespace

nvfp4_status launch_mxfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q, uint8_t* sf,
                                   Workspace* ws, cudaStream_t stream)
{
    MxArgs a;
    a.x = static_cast<const uint8_t*>(x);
    a.q = q;
    a.sf = sf;
    a.ws = ws;
    a.rows = rows;
    a.rows_pad = (rows + 127) / 128 * 128;
    a.ld = ld;
    a.kblocks = (uint32_t)(cols / 32);
    a.cp = (uint32_t)((cols + 63) / 64);
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, mxfp4_quantize_kernel, kMxThreads, 0) != cudaSuccess ||
        occ < 1)
        return NVFP4_ERR_CUDA;
    int64_t grid = (int64_t)device_sm_count() * occ;
    const int64_t need = (a.rows_pad + kMxThreads / 32 - 1) / (kMxThreads / 32);
    if (need < grid)
        grid = need;
    mxfp4_quantize_kernel<<<(unsigned)grid, kMxThreads, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
