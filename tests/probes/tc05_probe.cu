// Probe of the tcgen05 building blocks (test code): one 128 x N x K bf16 MMA
// chain with operands placed in shared memory in the K-major or MN-major
// swizzled layout, the fp32 result read back from tensor memory.
#include <cuda_runtime.h>

#include "tc05.cuh"

using namespace kda::tc;

namespace {

constexpr int kM = 128;
constexpr uint32_t kRegionA = 32768 + 4096;   // A tile (<= 32 KiB) plus a gap
constexpr uint32_t kRegionB = 65536 + 4096;   // B tile (<= 64 KiB) plus a gap
constexpr size_t kSmem = 1024 + kRegionA + kRegionB;

__global__ void __launch_bounds__(128) probe_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B,
                                                    float* D, int N, int K, int a_mn, int b_mn,
                                                    int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kRegionA;
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t sboA = (kM / 64) * 1024, sboB = (uint32_t)(N / 64) * 1024;

    for (int idx = tid; idx < kM * K; idx += blockDim.x) {
        const int m = idx / K, k = idx % K;
        const uint32_t off = a_mn ? mnmajor_off(m, k, 1024, sboA) : kmajor_off(m, k, kM);
        *reinterpret_cast<__nv_bfloat16*>(sA + off) = A[idx];
    }
    for (int idx = tid; idx < N * K; idx += blockDim.x) {
        const int n = idx / K, k = idx % K;
        const uint32_t off = b_mn ? mnmajor_off(n, k, 1024, sboB) : kmajor_off(n, k, N);
        *reinterpret_cast<__nv_bfloat16*>(sB + off) = B[idx];
    }
    fence_async_smem();
    if (warp == 0) tmem_alloc(&tslot, 256);
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tslot;

    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(kM, N, a_mn != 0, b_mn != 0);
        for (int ks = 0; ks < K / 16; ++ks) {
            uint64_t ad, bd;
            if (a_mn) ad = sdesc(smem_u32(sA) + ks * 2 * sboA, 1024, sboA);
            else ad = sdesc(smem_u32(sA) + (ks / 4) * kM * 128 + (ks % 4) * 32, 16, 1024);
            if (b_mn) bd = sdesc(smem_u32(sB) + ks * 2 * sboB, 1024, sboB);
            else bd = sdesc(smem_u32(sB) + (ks / 4) * N * 128 + (ks % 4) * 32, 16, 1024);
            mma_bf16(tbase, ad, bd, idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0);
    if (!ok && tid == 0) atomicOr(err, 1);
    fence_after_sync();
    if (ok) {
        const int row = 32 * warp + (tid & 31);
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16) + c0, r);
            tmem_wait_ld();
            for (int j = 0; j < 16; ++j) D[row * N + c0 + j] = __uint_as_float(r[j]);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

// A bounded wait that runs out: an mbarrier that nothing arrives at.  The
// wait must give up after `limit` cycles and report it; the kernel then returns.
__global__ void wait_probe_kernel(long long limit, long long* out) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const long long t0 = clock64();
        const bool ok = mbar_wait(&bar, 0, limit);
        out[0] = ok ? 1 : 0;
        out[1] = clock64() - t0;
    }
}

}  // namespace

extern "C" int wait_probe(long long limit, long long* out) {
    wait_probe_kernel<<<1, 32>>>(limit, out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}

extern "C" int tc05_probe(const void* A, const void* B, float* D, int N, int K, int a_mn, int b_mn,
                          int* err) {
    if (N < 16 || N > 256 || N % 16 || K < 16 || K > 128 || K % 64 ||
        ((a_mn || b_mn) && N % 64))
        return -1;
    cudaError_t e = cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return (int)e;
    probe_kernel<<<1, 128, kSmem>>>(static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B),
                                    D, N, K, a_mn, b_mn, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    return (int)cudaDeviceSynchronize();
}
