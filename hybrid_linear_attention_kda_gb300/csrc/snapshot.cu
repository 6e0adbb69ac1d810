// Copies between the block-indexed state pool and contiguous state buffers:
// the private copy of copy-on-write reuse ("Kimi K3 Tech Intro", section 2.3:
// copy the cached state to the request's private memory, then continue on the
// copy while the cached original stays read-only).  Pure HBM streaming with
// 16-byte accesses; bit-exact.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;
constexpr int64_t kVecPerBlock = (int64_t)kThreads * kVecPerThread;

// dst[i] = pool[slots[i]] (zeros for slot -1)
__global__ void __launch_bounds__(kThreads)
gather_kernel(const float4* __restrict__ pool, int64_t n_slots, const int32_t* __restrict__ slots,
              int64_t slot_vecs, int64_t blocks_per_slot, float4* __restrict__ dst,
              uint32_t* status) {
    const int64_t i = blockIdx.x / blocks_per_slot;
    const int64_t base = (blockIdx.x % blocks_per_slot) * kVecPerBlock;
    const int32_t slot = slots[i];
    const bool zero = slot == -1;
    if (!zero && (slot < 0 || (int64_t)slot >= n_slots)) {
        if (threadIdx.x == 0) flag(status, KDA_DEV_BAD_SLOT);
        return;
    }
    float4* out = dst + i * slot_vecs;
    const float4* in = pool + (zero ? 0 : (int64_t)slot * slot_vecs);
    float4 r[kVecPerThread];
#pragma unroll
    for (int m = 0; m < kVecPerThread; ++m) {
        const int64_t e = base + m * kThreads + threadIdx.x;
        r[m] = (!zero && e < slot_vecs) ? __ldcs(in + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int m = 0; m < kVecPerThread; ++m) {
        const int64_t e = base + m * kThreads + threadIdx.x;
        if (e < slot_vecs) __stcs(out + e, r[m]);
    }
}

// pool[slots[i]] = src[i] (skip slot -1)
__global__ void __launch_bounds__(kThreads)
restore_kernel(const float4* __restrict__ src, float4* __restrict__ pool, int64_t n_slots,
               const int32_t* __restrict__ slots, int64_t slot_vecs, int64_t blocks_per_slot,
               uint32_t* status) {
    const int64_t i = blockIdx.x / blocks_per_slot;
    const int64_t base = (blockIdx.x % blocks_per_slot) * kVecPerBlock;
    const int32_t slot = slots[i];
    if (slot == -1) return;
    if (slot < 0 || (int64_t)slot >= n_slots) {
        if (threadIdx.x == 0) flag(status, KDA_DEV_BAD_SLOT);
        return;
    }
    const float4* in = src + i * slot_vecs;
    float4* out = pool + (int64_t)slot * slot_vecs;
    float4 r[kVecPerThread];
#pragma unroll
    for (int m = 0; m < kVecPerThread; ++m) {
        const int64_t e = base + m * kThreads + threadIdx.x;
        if (e < slot_vecs) r[m] = __ldcs(in + e);
    }
#pragma unroll
    for (int m = 0; m < kVecPerThread; ++m) {
        const int64_t e = base + m * kThreads + threadIdx.x;
        if (e < slot_vecs) __stcs(out + e, r[m]);
    }
}

}  // namespace

cudaError_t launch_gather(const float* pool, int64_t n_slots, const int32_t* slots, int32_t n,
                          int64_t slot_elems, float* dst, uint32_t* status, cudaStream_t s) {
    const int64_t slot_vecs = slot_elems / 4;
    const int64_t bps = (slot_vecs + kVecPerBlock - 1) / kVecPerBlock;
    note_launch();
    gather_kernel<<<(unsigned)(bps * n), kThreads, 0, s>>>(
        reinterpret_cast<const float4*>(pool), n_slots, slots, slot_vecs, bps,
        reinterpret_cast<float4*>(dst), status);
    return cudaGetLastError();
}

cudaError_t launch_restore(const float* src, float* pool, int64_t n_slots, const int32_t* slots,
                           int32_t n, int64_t slot_elems, uint32_t* status, cudaStream_t s) {
    const int64_t slot_vecs = slot_elems / 4;
    const int64_t bps = (slot_vecs + kVecPerBlock - 1) / kVecPerBlock;
    note_launch();
    restore_kernel<<<(unsigned)(bps * n), kThreads, 0, s>>>(
        reinterpret_cast<const float4*>(src), reinterpret_cast<float4*>(pool), n_slots, slots,
        slot_vecs, bps, status);
    return cudaGetLastError();
}

}  // namespace kda
