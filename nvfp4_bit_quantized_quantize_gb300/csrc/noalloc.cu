// nvfp4_quantize_noalloc: the 1x16 quantizer for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or any allocating routine: a plugin
// loaded into a host program that owns every byte of device memory through
// its own allocator, a deployment whose device memory is reserved in full at
// start-up, or a latency-critical path where an allocation could block or
// synchronise the device.  nvfp4_quantize needs a caller-provided workspace
// for its grid-wide barrier and amax; this variant keeps that scratch in a
// file-scope device array instead, so the caller passes only inputs and
// outputs.
//
// The array belongs to every GPU that loads this library and stays resident
// until the process exits.  All calls share it, so two calls that overlap on
// the GPU (for example on two streams) race on it; calls on one stream run one
// after the other and are safe.  Each call clears the scratch on its stream
// before it launches the kernel.
#include <mutex>

#include "device.cuh"

using namespace nvfp4;

namespace {

// Scratch capacity: one quantizer workspace.  Every shape the 1x16 quantizer
// supports needs exactly this much today; a shape needing more is rejected.
constexpr size_t kNoAllocScratchBytes = 256;
static_assert(kNoAllocScratchBytes >= sizeof(Workspace), "scratch holds one workspace");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch for the current device.  In host code
// the symbol is only a host-side stand-in; cudaGetSymbolAddress, with the
// device current, yields the device address.  It is looked up on every call
// that is not being captured (it allocates nothing and costs little), so an
// address that changed after cudaDeviceReset or a module reload is never
// reused; a call on a capturing stream takes the address the last uncaptured
// call on that device found.
std::mutex g_setup_mutex;
void* g_scratch_ptr[64] = {};

nvfp4_status scratch_for_current_device(cudaStream_t stream, void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return NVFP4_ERR_CUDA;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        (void)cudaGetLastError();  // an unqueryable stream is treated as not capturing
        cs = cudaStreamCaptureStatusNone;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (cs == cudaStreamCaptureStatusNone || g_scratch_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return NVFP4_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return NVFP4_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                               nvfp4_round mode, uint64_t sr_seed, uint8_t* q, uint8_t* sf,
                                               float* g_dec, nvfp4_stream_t stream)
{
    if (!x || !q || !sf || !g_dec || (mode != NVFP4_ROUND_RN && mode != NVFP4_ROUND_SR))
        return NVFP4_ERR_ARG;
    if (rows <= 0 || cols <= 0 || cols % 16 != 0 || ld < cols || rows > (1ll << 31) || cols > (1ll << 31))
        return NVFP4_ERR_SHAPE;
    if (nvfp4_workspace_bytes(rows, cols) > kNoAllocScratchBytes)
        return NVFP4_ERR_SHAPE;  // would need more scratch than the static array holds
    if (!aligned16(x) || !aligned16(q) || !aligned16(sf) || ld % 8 != 0)
        return NVFP4_ERR_ALIGN;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (!(major == 10 && minor == 3))
        return NVFP4_ERR_UNSUPPORTED;

    void* scratch = nullptr;
    nvfp4_status st = scratch_for_current_device((cudaStream_t)stream, &scratch);
    if (st != NVFP4_OK)
        return st;
    // the barrier counters, amax and status must start at zero
    if (cudaMemsetAsync(scratch, 0, kNoAllocScratchBytes, (cudaStream_t)stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;

    const QuantParams p = params_1x16(rows, cols, mode, sr_seed, q, sf, g_dec);
    return launch_quantize(QuantKind::k1x16, x, ld, p, static_cast<Workspace*>(scratch), (cudaStream_t)stream);
}
