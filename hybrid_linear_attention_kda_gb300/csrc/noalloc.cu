// kda_prefill_chunked_noalloc: the chunked prefill for callers that cannot
// allocate device memory.
//
// kda_prefill_chunked needs a workspace from the caller.  Some callers cannot
// produce one at the moment they prefill: a serving process whose device memory
// is all handed out up front to its own pools, a plugin host that only lends
// the library a stream and the input/output buffers, or code that must not call
// cudaMalloc (or any allocating routine) on its latency-critical path.  This
// entry point takes the same arguments and uses one scratch array in the
// library's own static device memory instead; it allocates nothing.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// (64 MiB).  Every GPU on which the library's device code is loaded holds it
// until the process exits.  Batches whose workspace (as reported by
// kda_prefill_workspace_size) exceeds it are rejected.  All calls share the one
// array, so calls that overlap on the GPU (different streams or threads, without
// ordering between them) race on it; it keeps the last call's contents.  Every
// part of it that a call relies on is written by that call's own kernels before
// it is read (the chunk table and the count of listed exact items are rewritten
// by the first kernel, every record by the chunk-local stage before the carry
// reads it), so nothing needs clearing between calls.
//
// In host code the array's name is only a stand-in for the device variable; the
// device address comes from cudaGetSymbolAddress, looked up on the first call on
// each device (with that device current) and cached.  That first call should
// therefore come before any stream capture.
#include <mutex>

#include "chunk_common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

__device__ __align__(256) uint8_t g_prefill_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

kda_status_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return kda::record_error(KDA_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices) return kda::record_error(KDA_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_prefill_scratch);
        if (e != cudaSuccess || !p)
            return kda::record_error(KDA_ERR_CUDA, "cudaGetSymbolAddress of the static prefill scratch failed");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status_t kda_prefill_chunked_noalloc(const kda_prefill_args* args, void* stream) {
    if (!args) return kda::record_error(KDA_ERR_INVALID_ARG, "args is NULL");
    kda_prefill_args a = *args;
    const size_t need = kda_prefill_workspace_size(&a);
    if (need > kNoAllocScratchBytes)
        return kda::record_error(KDA_ERR_UNSUPPORTED,
                                 "this batch needs more workspace than the 64 MiB static scratch of "
                                 "kda_prefill_chunked_noalloc");
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    if (need > 0) {
        void* p = nullptr;
        const kda_status_t st = scratch_address(&p);
        if (st != KDA_OK) return st;
        a.workspace = p;
        a.workspace_bytes = kNoAllocScratchBytes;
    }
    return kda_prefill_chunked(&a, stream);
}
