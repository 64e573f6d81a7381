// C-ABI entry points: argument validation, then one launch on the caller's
// stream.  Nothing here allocates device memory.
#include <cstring>

#include "device.cuh"

using namespace nvfp4;

namespace nvfp4 {

int device_sm_count()
{
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    if (dev < 64 && cache[dev] > 0)
        return cache[dev];
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (dev < 64)
        cache[dev] = n;
    return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace {
// cuTensorMapEncodeTiled, resolved once through the runtime (no libcuda link).
EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || p == nullptr)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}
}  // namespace

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t dim0, uint64_t dim1,
                          uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return false;
    const cuuint64_t dims[2] = {dim0, dim1};
    const cuuint64_t strides[1] = {stride1_bytes};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t elem_strides[2] = {1, 1};
    return fn(map, dtype, 2, base, dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_sf_atom_map(CUtensorMap* map, const uint8_t* sf, int64_t rows, int64_t K, uint32_t row_tiles_per_box)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return false;
    // 512-byte atoms as 64 x 8-byte elements; the atoms of one 128-row tile
    // are contiguous along K; row tiles follow each other
    const cuuint64_t cp = (cuuint64_t)((K / 16 + 3) / 4);
    const cuuint64_t tiles = (cuuint64_t)((rows + 127) / 128);
    const cuuint64_t dims[3] = {64, cp, tiles};
    const cuuint64_t strides[2] = {512, cp * 512};
    const cuuint32_t box[3] = {64, 4, row_tiles_per_box};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t*>(sf), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ----------------------------------------------------------------- probe ----
namespace {
__global__ void encode_probe_kernel(const float* v, const uint16_t* r, int64_t n, uint8_t* e4m3, uint8_t* rn,
                                    uint8_t* sr)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float x = v[i];
        if (e4m3)
            e4m3[i] = (uint8_t)e4m3_rn_sat(x);
        if (rn)
            rn[i] = (uint8_t)(e2m1x2_rn(x, 0.0f) & 15u);
        if (sr)
            sr[i] = (uint8_t)e2m1_sr(x, r ? r[i] : 0u);
    }
}
}  // namespace

nvfp4_status launch_encode_probe(const float* v, const uint16_t* r, int64_t n, uint8_t* e4m3, uint8_t* rn,
                                 uint8_t* sr, cudaStream_t stream)
{
    if (n == 0)
        return NVFP4_OK;
    const int64_t blocks64 = (n + 255) / 256;
    const int blocks = (int)(blocks64 < 4096 ? blocks64 : 4096);
    encode_probe_kernel<<<blocks, 256, 0, stream>>>(v, r, n, e4m3, rn, sr);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

void philox_round_keys(uint64_t seed, uint32_t (&keys)[20])
{
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        keys[2 * r] = k0;
        keys[2 * r + 1] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}

void rht_pair_masks(uint32_t sign_bits, uint32_t (&mask)[16])
{
    for (int i = 0; i < 16; ++i)
        mask[i] = ((sign_bits >> i) & 1u) ? 0x80008000u : 0u;
}

// 128-row x 64-column tiles, 1x16 blocks along the rows.
QuantParams params_1x16(int64_t rows, int64_t cols, int mode, uint64_t sr_seed, uint8_t* q, uint8_t* sf,
                        float* g_dec)
{
    QuantParams p = {};
    p.rows = rows;
    p.cols = cols;
    p.tiles_c = (cols + 63) / 64;
    p.tiles_r = (rows + 127) / 128;
    p.ntiles = p.tiles_r * p.tiles_c;
    p.q = q;
    p.sf = sf;
    p.g_dec = g_dec;
    p.sr_seed = sr_seed;
    philox_round_keys(sr_seed, p.keys[0]);
    p.mode = mode;
    return p;
}

}  // namespace nvfp4

// ------------------------------------------------------------------ C ABI ----
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

nvfp4_status check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    // the library carries sm_103a code only
    return (major == 10 && minor == 3) ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The random sign diagonal of the 16-point Hadamard transform: bit i of word 0
// of Philox4x32-10 (key = rht_seed, counter = (0, 0, 1, 0)) flips the sign of
// input i.
uint32_t rht_sign_bits(uint64_t rht_seed)
{
    uint32_t c[4] = {0u, 0u, 1u, 0u};
    uint32_t k[2] = {(uint32_t)rht_seed, (uint32_t)(rht_seed >> 32)};
    for (int round = 0; round < 10; ++round) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k[0];
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k[1];
        c[0] = n0;
        c[1] = (uint32_t)p1;
        c[2] = n2;
        c[3] = (uint32_t)p0;
        k[0] += 0x9E3779B9u;
        k[1] += 0xBB67AE85u;
    }
    return c[0] & 0xFFFFu;
}

// Both forms of nvfp4_quantize_dual; amax (device, 2 floats) given or nullptr.
nvfp4_status quantize_dual(const void* x, int64_t T, int64_t C, int64_t ld, nvfp4_round mode, uint64_t sr_seed,
                           uint8_t* q, uint8_t* sf, float* g_dec, uint64_t rht_seed, nvfp4_round mode_t,
                           uint64_t sr_seed_t, uint8_t* qT, uint8_t* sfT, float* g_dec_t, const float* amax, void* ws,
                           nvfp4_stream_t stream)
{
    if (!x || !q || !sf || !g_dec || !qT || !sfT || !g_dec_t || !ws ||
        (mode != NVFP4_ROUND_RN && mode != NVFP4_ROUND_SR) || (mode_t != NVFP4_ROUND_RN && mode_t != NVFP4_ROUND_SR))
        return NVFP4_ERR_ARG;
    if (T <= 0 || C <= 0 || T % 16 != 0 || C % 16 != 0 || ld < C || T > (1ll << 31) || C > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sf) || !aligned16(qT) || !aligned16(sfT) || !aligned16(ws) ||
        ld % 8 != 0)
        return NVFP4_ERR_ALIGN;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    QuantParams p = {};
    p.rows = T;
    p.cols = C;
    p.tiles_c = cdiv(C, 256);  // 64-token x 256-channel tiles
    p.tiles_r = cdiv(T, 64);
    p.ntiles = p.tiles_r * p.tiles_c;
    p.q = q;
    p.sf = sf;
    p.g_dec = g_dec;
    p.sr_seed = sr_seed;
    p.mode = mode;
    p.q2 = qT;
    p.sf2 = sfT;
    p.g_dec2 = g_dec_t;
    p.sr_seed2 = sr_seed_t;
    p.mode2 = mode_t;
    p.amax_in = amax;
    philox_round_keys(sr_seed, p.keys[0]);
    philox_round_keys(sr_seed_t, p.keys[1]);
    p.rht_signs = rht_sign_bits(rht_seed);
    rht_pair_masks(p.rht_signs, p.rht_mask);
    return launch_quantize(QuantKind::kDual, x, ld, p, static_cast<Workspace*>(ws), (cudaStream_t)stream);
}

}  // namespace

extern "C" {

size_t nvfp4_sf_bytes(int64_t rows, int64_t cols)
{
    if (rows < 0 || cols < 0)
        return 0;
    return (size_t)(cdiv(rows, 128) * 128 * cdiv(cols / 16, 4) * 4);
}

size_t nvfp4_workspace_bytes(int64_t, int64_t) { return kWorkspaceBytes; }

nvfp4_status nvfp4_workspace_init(void* ws, nvfp4_stream_t stream)
{
    if (ws == nullptr)
        return NVFP4_ERR_ARG;
    return cudaMemsetAsync(ws, 0, kWorkspaceBytes, (cudaStream_t)stream) == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, nvfp4_round mode,
                            uint64_t sr_seed, uint8_t* q, uint8_t* sf, float* g_dec, void* ws,
                            nvfp4_stream_t stream)
{
    if (!x || !q || !sf || !g_dec || !ws || (mode != NVFP4_ROUND_RN && mode != NVFP4_ROUND_SR))
        return NVFP4_ERR_ARG;
    if (rows <= 0 || cols <= 0 || cols % 16 != 0 || ld < cols || rows > (1ll << 31) || cols > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sf) || !aligned16(ws) || ld % 8 != 0)
        return NVFP4_ERR_ALIGN;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    const QuantParams p = params_1x16(rows, cols, mode, sr_seed, q, sf, g_dec);
    return launch_quantize(QuantKind::k1x16, x, ld, p, static_cast<Workspace*>(ws), (cudaStream_t)stream);
}

nvfp4_status nvfp4_quantize_2d(const void* w, int64_t rows, int64_t cols, int64_t ld, uint8_t* q, uint8_t* sf,
                               uint8_t* qT, uint8_t* sfT, float* g_dec, void* ws, nvfp4_stream_t stream)
{
    if (!w || !q || !sf || !g_dec || !ws || ((qT == nullptr) != (sfT == nullptr)))
        return NVFP4_ERR_ARG;
    if (rows <= 0 || cols <= 0 || cols % 16 != 0 || rows % 16 != 0 || ld < cols || rows > (1ll << 31) ||
        cols > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(w) || !aligned16(q) || !aligned16(sf) || !aligned16(ws) || ld % 8 != 0 ||
        (qT && (!aligned16(qT) || !aligned16(sfT))))
        return NVFP4_ERR_ALIGN;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    QuantParams p = {};
    p.rows = rows;
    p.cols = cols;
    p.tiles_c = cdiv(cols, 64);
    p.tiles_r = cdiv(rows, 128);
    p.ntiles = p.tiles_r * p.tiles_c;
    p.q = q;
    p.sf = sf;
    p.qT = qT;
    p.sfT = sfT;
    p.g_dec = g_dec;
    p.mode = NVFP4_ROUND_RN;
    return launch_quantize(QuantKind::k2d, w, ld, p, static_cast<Workspace*>(ws), (cudaStream_t)stream);
}

nvfp4_status nvfp4_rht_quantize(const void* x, int64_t T, int64_t C, int64_t ld, uint64_t rht_seed,
                                nvfp4_round mode, uint64_t sr_seed, uint8_t* qT, uint8_t* sfT, float* g_dec,
                                void* ws, nvfp4_stream_t stream)
{
    if (!x || !qT || !sfT || !g_dec || !ws || (mode != NVFP4_ROUND_RN && mode != NVFP4_ROUND_SR))
        return NVFP4_ERR_ARG;
    if (T <= 0 || C <= 0 || T % 16 != 0 || ld < C || T > (1ll << 31) || C > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(qT) || !aligned16(sfT) || !aligned16(ws) || ld % 8 != 0)
        return NVFP4_ERR_ALIGN;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    QuantParams p = {};
    p.rows = T;
    p.cols = C;
    p.tiles_c = cdiv(C, 256);  // 64-token x 256-channel tiles
    p.tiles_r = cdiv(T, 64);
    p.ntiles = p.tiles_r * p.tiles_c;
    p.q = qT;
    p.sf = sfT;
    p.g_dec = g_dec;
    p.sr_seed = sr_seed;
    philox_round_keys(sr_seed, p.keys[0]);
    p.rht_signs = rht_sign_bits(rht_seed);
    rht_pair_masks(p.rht_signs, p.rht_mask);
    p.mode = mode;
    return launch_quantize(QuantKind::kRht, x, ld, p, static_cast<Workspace*>(ws), (cudaStream_t)stream);
}

nvfp4_status nvfp4_quantize_dual(const void* x, int64_t T, int64_t C, int64_t ld, nvfp4_round mode,
                                 uint64_t sr_seed, uint8_t* q, uint8_t* sf, float* g_dec, uint64_t rht_seed,
                                 nvfp4_round mode_t, uint64_t sr_seed_t, uint8_t* qT, uint8_t* sfT, float* g_dec_t,
                                 void* ws, nvfp4_stream_t stream)
{
    return quantize_dual(x, T, C, ld, mode, sr_seed, q, sf, g_dec, rht_seed, mode_t, sr_seed_t, qT, sfT, g_dec_t,
                         nullptr, ws, stream);
}

nvfp4_status nvfp4_quantize_dual_from_amax(const void* x, int64_t T, int64_t C, int64_t ld, const float* amax,
                                           nvfp4_round mode, uint64_t sr_seed, uint8_t* q, uint8_t* sf,
                                           float* g_dec, uint64_t rht_seed, nvfp4_round mode_t, uint64_t sr_seed_t,
                                           uint8_t* qT, uint8_t* sfT, float* g_dec_t, void* ws,
                                           nvfp4_stream_t stream)
{
    if (!amax)
        return NVFP4_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(amax) & 3)
        return NVFP4_ERR_ALIGN;
    return quantize_dual(x, T, C, ld, mode, sr_seed, q, sf, g_dec, rht_seed, mode_t, sr_seed_t, qT, sfT, g_dec_t,
                         amax, ws, stream);
}

nvfp4_status nvfp4_quant_noise(const void* x, int64_t rows, int64_t cols, int64_t ld, const uint8_t* q,
                               const uint8_t* sf, const float* g_dec, double* sums, nvfp4_stream_t stream)
{
    if (!x || !q || !sf || !g_dec || !sums)
        return NVFP4_ERR_ARG;
    if (rows <= 0 || cols <= 0 || cols % 16 != 0 || ld < cols || rows > (1ll << 31) || cols > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sf) || ld % 8 != 0 || (reinterpret_cast<uintptr_t>(sums) & 7) ||
        (reinterpret_cast<uintptr_t>(g_dec) & 3))
        return NVFP4_ERR_ALIGN;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    return launch_quant_noise(x, rows, cols, ld, q, sf, g_dec, sums, (cudaStream_t)stream);
}

nvfp4_status nvfp4_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                        const uint8_t* sfb, const float* gb, int64_t M, int64_t N, int64_t K, void* d, int64_t ldd,
                        nvfp4_out_dtype out_dtype, void* ws, nvfp4_stream_t stream)
{
    if (!a || !sfa || !ga || !b || !sfb || !gb || !d || !ws ||
        (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32))
        return NVFP4_ERR_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || K % 32 != 0 || ldd < N ||
        K / 2 >= (1ll << 32) || M > (1ll << 31) || N > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(d) || !aligned16(ws) ||
        (ldd * (out_dtype == NVFP4_OUT_F32 ? 4 : 2)) % 16 != 0 || (reinterpret_cast<uintptr_t>(ga) & 3) ||
        (reinterpret_cast<uintptr_t>(gb) & 3))
        return NVFP4_ERR_ALIGN;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    return launch_gemm(a, sfa, ga, b, sfb, gb, M, N, K, d, ldd, out_dtype, false, nullptr, 0u,
                       static_cast<Workspace*>(ws), (cudaStream_t)stream);
}

nvfp4_status nvfp4_gemm_amax(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                             const uint8_t* sfb, const float* gb, int64_t M, int64_t N, int64_t K, void* d,
                             int64_t ldd, uint64_t rht_seed, float* amax, void* ws, nvfp4_stream_t stream)
{
    if (!a || !sfa || !ga || !b || !sfb || !gb || !d || !ws || !amax)
        return NVFP4_ERR_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || K % 32 != 0 || M % 16 != 0 || N % 16 != 0 || ldd < N ||
        K / 2 >= (1ll << 32) || M > (1ll << 31) || N > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(d) || !aligned16(ws) ||
        (ldd * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(ga) & 3) || (reinterpret_cast<uintptr_t>(gb) & 3) ||
        (reinterpret_cast<uintptr_t>(amax) & 3))
        return NVFP4_ERR_ALIGN;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    return launch_gemm(a, sfa, ga, b, sfb, gb, M, N, K, d, ldd, NVFP4_OUT_BF16, false, amax,
                       rht_sign_bits(rht_seed), static_cast<Workspace*>(ws), (cudaStream_t)stream);
}

nvfp4_status nvfp4_mxfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q, uint8_t* sf,
                                  void* ws, nvfp4_stream_t stream)
{
    if (!x || !q || !sf || !ws)
        return NVFP4_ERR_ARG;
    if (rows <= 0 || cols <= 0 || cols % 32 != 0 || ld < cols || rows > (1ll << 31) || cols > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sf) || !aligned16(ws) || ld % 8 != 0)
        return NVFP4_ERR_ALIGN;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    return launch_mxfp4_quantize(x, rows, cols, ld, q, sf, static_cast<Workspace*>(ws), (cudaStream_t)stream);
}

nvfp4_status nvfp4_mxfp4_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb, int64_t M,
                              int64_t N, int64_t K, void* d, int64_t ldd, nvfp4_out_dtype out_dtype, void* ws,
                              nvfp4_stream_t stream)
{
    if (!a || !sfa || !b || !sfb || !d || !ws || (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32))
        return NVFP4_ERR_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || K % 32 != 0 || ldd < N || K / 2 >= (1ll << 32) || M > (1ll << 31) ||
        N > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(d) || !aligned16(ws) ||
        (ldd * (out_dtype == NVFP4_OUT_F32 ? 4 : 2)) % 16 != 0)
        return NVFP4_ERR_ALIGN;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    return launch_gemm(a, sfa, nullptr, b, sfb, nullptr, M, N, K, d, ldd, out_dtype, true, nullptr, 0u,
                       static_cast<Workspace*>(ws), (cudaStream_t)stream);
}

nvfp4_status nvfp4_device_status(void* ws, nvfp4_stream_t stream)
{
    if (ws == nullptr)
        return NVFP4_ERR_ARG;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return (nvfp4_status)v;
}

const char* nvfp4_status_str(nvfp4_status s)
{
    switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_ARG: return "invalid argument";
    case NVFP4_ERR_SHAPE: return "unsupported shape";
    case NVFP4_ERR_ALIGN: return "misaligned pointer or leading dimension";
    case NVFP4_ERR_NONFINITE: return "non-finite input";
    case NVFP4_ERR_TIMEOUT: return "device wait timed out";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_UNSUPPORTED: return "unsupported device";
    }
    return "unknown status";
}

nvfp4_status nvfp4_encode_probe(const float* v, const uint16_t* r, int64_t n, uint8_t* e4m3_out,
                                uint8_t* e2m1_rn_out, uint8_t* e2m1_sr_out, nvfp4_stream_t stream)
{
    if (!v || n < 0)
        return NVFP4_ERR_ARG;
    nvfp4_status st = check_device();
    if (st != NVFP4_OK)
        return st;
    return launch_encode_probe(v, r, n, e4m3_out, e2m1_rn_out, e2m1_sr_out, (cudaStream_t)stream);
}

}  // extern "C"
