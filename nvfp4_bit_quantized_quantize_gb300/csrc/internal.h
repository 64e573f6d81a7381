// Internal declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// Device workspace (caller-owned, zeroed once).  The quantizers' grid-wide
// barrier and amax live here; the last CTA of every call puts them back to 0.
struct Workspace {
    uint32_t status;      // sticky nvfp4_status recorded by the device (0 = OK)
    uint32_t amax_bits;   // max |x| over the tensor, as float bits (atomicMax)
    uint32_t arrived;     // CTAs that reached the grid barrier
    uint32_t departed;    // CTAs that finished
    uint32_t amax2_bits;  // second output's amax (dual quantizer: max |RHT(x)|)
    uint32_t gemm_amax[2];  // GEMM with output maxima: max |D| and max |RHT(D)| so far, as float bits
    uint32_t gemm_done;     // GEMM epilogue warps that added their maxima
    uint32_t pad[56];
};
static_assert(sizeof(Workspace) == 256, "workspace layout");

constexpr size_t kWorkspaceBytes = sizeof(Workspace);

// Quantizer launch parameters (one struct for the three variants).
struct QuantParams {
    int64_t rows, cols;     // logical matrix of the input (rows x cols, or T x C)
    int64_t ntiles;         // tiles in the whole tensor
    int64_t tiles_c;        // tiles along the contiguous axis
    int64_t tiles_r;        // tiles along the strided axis (ntiles / tiles_c)
    uint8_t* q;             // codes
    uint8_t* sf;            // scales
    uint8_t* qT;            // transposed codes (2-D variant) or nullptr
    uint8_t* sfT;           // transposed scales (2-D variant) or nullptr
    float* g_dec;           // tensor decode scale out
    uint64_t sr_seed;
    uint32_t rht_signs;     // 16 sign bits (Hadamard variant)
    uint32_t rht_mask[16];  // per token i of a 16-block: 0x80008000 where the sign diagonal flips it, else 0
    uint32_t keys[2][20];   // Philox4x32-10 round keys (k0, k1 of rounds 0..9) of sr_seed and of sr_seed2
    int mode;               // nvfp4_round
    // second output of the dual quantizer (Hadamard, token-major codes)
    uint8_t* q2;
    uint8_t* sf2;
    float* g_dec2;
    uint64_t sr_seed2;
    int mode2;
    // the tensor amaxes (both outputs' for the dual quantizer), already
    // reduced on the device by the producer of x; nullptr: reduce them here
    const float* amax_in;
};

enum class QuantKind { k1x16, k2d, kRht, kDual };

// Philox4x32-10 round keys of a seed: round r uses (seed lo + r 0x9E3779B9,
// seed hi + r 0xBB67AE85) (Salmon et al., SC'11), precomputed once per call.
void philox_round_keys(uint64_t seed, uint32_t (&keys)[20]);

// XOR masks of the random sign diagonal for bf16 pairs (both halves).
void rht_pair_masks(uint32_t sign_bits, uint32_t (&mask)[16]);

// Launch parameters of the 1x16 quantizer (nvfp4_quantize and its
// allocation-free variant build them here, so the two cannot drift apart).
QuantParams params_1x16(int64_t rows, int64_t cols, int mode, uint64_t sr_seed, uint8_t* q, uint8_t* sf,
                        float* g_dec);

// Host launchers (quantize.cu, gemm.cu, noise.cu, mxfp4.cu, probe.cu).  They assume the
// arguments were validated by the C-ABI layer.
nvfp4_status launch_quantize(QuantKind kind, const void* x, int64_t ld, const QuantParams& p, Workspace* ws,
                             cudaStream_t stream);

nvfp4_status launch_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                         const uint8_t* sfb, const float* gb, int64_t M, int64_t N, int64_t K, void* d,
                         int64_t ldd, nvfp4_out_dtype dt, bool mx, float* amax_out, uint32_t rht_signs,
                         Workspace* ws, cudaStream_t stream);

nvfp4_status launch_mxfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* q, uint8_t* sf,
                                   Workspace* ws, cudaStream_t stream);

nvfp4_status launch_quant_noise(const void* x, int64_t rows, int64_t cols, int64_t ld, const uint8_t* q,
                                const uint8_t* sf, const float* g_dec, double* sums, cudaStream_t stream);

nvfp4_status launch_encode_probe(const float* v, const uint16_t* r, int64_t n, uint8_t* e4m3, uint8_t* rn,
                                 uint8_t* sr, cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).  Returns false if unavailable.
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t dim0,
                          uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                          CUtensorMapSwizzle swizzle);

// Tensor map over a scale buffer in the 128 x 4 atom layout: a 3-D tensor of
// 512-byte atoms (64 x 8-byte elements) x atoms along K x 128-row tiles; a
// box is 4 atoms (one 256-element K stage) of `row_tiles_per_box` row tiles.
// Atoms past K or past the last row tile read as zeros.
bool encode_sf_atom_map(CUtensorMap* map, const uint8_t* sf, int64_t rows, int64_t K, uint32_t row_tiles_per_box);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace nvfp4
