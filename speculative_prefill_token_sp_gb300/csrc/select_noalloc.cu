// sp_select_noalloc: chunk selection for callers that cannot allocate device
// memory.
//
// sp_select needs a scratch workspace (chunk sums, means, pooled scores, keep
// flags, output offsets).  Some callers cannot provide one: code that runs
// inside a device-memory allocator or its out-of-memory handler (allocating
// there would re-enter the allocator), serving loops whose latency budget
// forbids cudaMalloc (it can synchronise the whole device), and plug-ins that
// a host framework hands only input and output buffers.  This entry point
// keeps its scratch in a fixed array in device memory that belongs to the
// library itself, so the caller passes only inputs and outputs.
//
// Limits and sharing:
//  * one prompt per call, at most kNoAllocMaxChunks chunks (ceil(M / chunk));
//    larger requests are rejected with SP_EUNSUPPORTED before any work;
//  * the array (kNoAllocScratchBytes) comes into being on a device when this
//    file's module is loaded there.  With CUDA's lazy module loading that is
//    the first call on the device: its cudaGetSymbolAddress (made with that
//    device current) loads the module, which may allocate device memory for
//    the array and the kernels' code.  Callers inside an allocator or an
//    out-of-memory handler must therefore make one call on every device ahead
//    of time (and before any stream capture); later calls allocate nothing,
//    and the array stays until the process exits;
//  * every call on a device uses the same array and leaves its contents
//    behind; each call clears what it needs cleared, but two calls whose work
//    overlaps on the GPU (different streams, no ordering) race on it.
#include "sp_common.cuh"

#include <mutex>

namespace {

constexpr int64_t kNoAllocMaxChunks = 65536;
constexpr size_t kNoAllocScratchBytes = 3u << 20;    // 3 MiB; holds the layout for kNoAllocMaxChunks
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_select_scratch on the current device (set up once per device).
sp_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        sp::set_error("sp_select_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
        return SP_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        sp::set_error("sp_select_noalloc: device ordinal %d is beyond the supported %d", dev, kMaxDevices);
        return SP_EUNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_select_scratch);
        if (e != cudaSuccess || p == nullptr) {
            sp::set_error("sp_select_noalloc: cudaGetSymbolAddress failed on device %d: %s", dev,
                          cudaGetErrorString(e));
            return SP_ECUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SP_OK;
}

}  // namespace

extern "C" sp_status sp_select_noalloc(const float* importance, int64_t M, int chunk, int pool_k, sp_mode mode,
                                       double rate, const sp_boost* boost, int32_t* kept_pos, int64_t* n_kept,
                                       void* stream) {
    sp::SelectProblem p;
    int64_t cu[2];
    sp_status s = sp::select_validate_single("sp_select_noalloc", importance, M, chunk, pool_k, mode, rate, boost,
                                             kept_pos, n_kept, &p, cu);
    if (s != SP_OK) return s;
    if (p.total_chunks > kNoAllocMaxChunks) {
        sp::set_error("sp_select_noalloc: %lld chunks exceed the fixed scratch limit of %lld chunks "
                      "(use sp_select with a workspace)", (long long)p.total_chunks,
                      (long long)kNoAllocMaxChunks);
        return SP_EUNSUPPORTED;
    }
    const size_t need = sp::select_ws_bytes(p);
    if (need > kNoAllocScratchBytes) {
        sp::set_error("sp_select_noalloc: needs %zu scratch bytes, the fixed array holds %zu", need,
                      kNoAllocScratchBytes);
        return SP_EUNSUPPORTED;
    }
    void* ws = nullptr;
    s = scratch_address(&ws);
    if (s != SP_OK) return s;
    s = sp::select_launch(p, ws, static_cast<cudaStream_t>(stream));
    if (s == SP_OK) sp::clear_error();
    return s;
}
