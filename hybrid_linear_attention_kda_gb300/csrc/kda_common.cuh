// Internal helpers shared by the KDA kernels (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Element access for the two storage types of q, k, v, o.
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p) { return *p; }
    static __device__ __forceinline__ void store(float* p, float x) { *p = x; }
    static __device__ __forceinline__ float cvt(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float x) {
        *p = __float2bfloat16_rn(x);
    }
    static __device__ __forceinline__ __nv_bfloat16 cvt(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ void flag(uint32_t* status, uint32_t bit) {
    atomicOr(status, bit);
}

// Counts kernel launches (kda_launch_count); every launcher calls it once per launch.
void note_launch(int n = 1);

// Launches `kernel` with programmatic stream serialization: its CTAs may be
// scheduled while the previous kernel in the stream finishes, so its launch
// latency overlaps that kernel's tail.  Such a kernel calls griddep_wait()
// before it touches memory: the wait returns once the previous grid has
// completed and its writes are visible, so stream order is kept.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The first statement of a kernel started by launch_overlapped (a no-op when
// the kernel was launched plainly).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Records `message` as this host thread's last error (kda_last_error) and returns status.
kda_status_t record_error(kda_status_t status, const char* message);

// ----------------------------------------------------------------- launchers
// Each returns the cudaError_t of its launch.  Arguments were validated by the
// C-ABI layer.

struct DecodeLaunch {
    int32_t n_seqs, H, D, dtype;
    const void *q, *k, *v;
    const float *alpha, *beta;
    float* pool;
    int64_t n_slots;
    const int32_t* slot;
    void* o;
    float scale;
    uint32_t* status;
};
cudaError_t launch_decode(const DecodeLaunch& p, cudaStream_t s);

// Speculative decoding: T candidate tokens per sequence, [n_seqs, T, H, .] layouts.
struct SpecLaunch {
    int32_t n_seqs, T, H, D, dtype;
    const void *q, *k, *v;
    const float *alpha, *beta;
    float* pool;
    int64_t n_slots;
    const int32_t* slot;
    void* o;
    float* u;
    const int32_t* n_accept;
    float scale;
    uint32_t* status;
};
cudaError_t launch_verify(const SpecLaunch& p, cudaStream_t s);

// One fused decode step (prologue, update, epilogue); arguments as in the C ABI.
struct FusedDecodeLaunch {
    kda_fused_decode_args a;
    uint32_t* status;
};
cudaError_t launch_fused_decode(const FusedDecodeLaunch& L, cudaStream_t s);
cudaError_t launch_commit(const SpecLaunch& p, cudaStream_t s);

cudaError_t launch_gather(const float* pool, int64_t n_slots, const int32_t* slots, int32_t n,
                          int64_t slot_elems, float* dst, uint32_t* status, cudaStream_t s);
cudaError_t launch_restore(const float* src, float* pool, int64_t n_slots, const int32_t* slots,
                           int32_t n, int64_t slot_elems, uint32_t* status, cudaStream_t s);

}  // namespace kda
