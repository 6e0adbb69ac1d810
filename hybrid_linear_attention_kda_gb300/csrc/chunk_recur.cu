// Stage two of the chunked prefill: the fp32 state carried through the chunks of
// one (sequence, head), with snapshots and outputs.
//
// Everything runs transposed so that the value channel j (128 of them) is the
// MMA M dimension and the TMEM lane.  Per chunk, with S^T [j][c] the state:
//   (a) D1 = S^T W^T             U^T = U~^T - D1            (bf16 U^T to smem)
//   (b) D2 = S^T Q~^T
//   (c) D2 += U^T P^T            O^T = D2
//   (d) D3 = U^T Kbar            S^T <- S^T Diag(gamma) + D3  (fp32, registers)
// Thread (j, half) keeps 64 fp32 state entries S[c][j] for its half of the key
// channels c; the bf16 copy of S^T in shared memory is the A operand of (a) and
// (b).  The chunk records written by stage one arrive with bulk copies, two
// chunks in flight.  A snapshot is written after every chunk that ends at an
// absolute position that is a multiple of snap_interval ("Kimi K3 Tech Intro",
// sections 2.2-2.4), straight from the fp32 registers.
#include "chunk_common.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int kThreads = 256;
constexpr uint32_t kSa = 0;               // S^T bf16, K-major [j][c], two 64-wide regions
constexpr uint32_t kUa = 32768;           // U^T bf16, K-major [j][t]
constexpr uint32_t kStage0 = 49152;
constexpr uint32_t kStageStride = 74752;  // kRecBytes rounded up to 1024
constexpr uint32_t kMisc = kStage0 + 2 * kStageStride;
constexpr size_t kSmemBytes = kMisc + 64 + 1024;

struct Misc {
    uint64_t bar_load[2];
    uint64_t bar_mma;
    uint32_t tslot;
};

__device__ __forceinline__ void sts16(uint32_t saddr, uint4 v) { st_shared_v4(saddr, v.x, v.y, v.z, v.w); }

__global__ void __launch_bounds__(kThreads, 1) chunk_recur_kernel(ChunkLaunch p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc& ms = *reinterpret_cast<Misc*>(sm + kMisc);
    const uint32_t s_base = smem_u32(sm);

    const kda_prefill_args& a = p.a;
    const int H = a.n_heads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seq = (int)(blockIdx.x / H);
    const int h = (int)(blockIdx.x % H);
    int64_t tb, te, pos0;
    int32_t init;
    uint32_t bad;
    if (!seq_valid(a, seq, &tb, &te, &pos0, &init, &bad)) return;     // flagged by the meta kernel
    if (p.chain_flag[(int64_t)seq * H + h]) return;                    // recomputed token by token
    const int64_t g0 = p.chunk_base[seq];
    const int64_t nc = p.chunk_base[seq + 1] - g0;
    if (nc < 0 || g0 + nc > p.max_chunks) return;

    const int jq = warp & 3, ch = warp >> 2;
    const int j = 32 * jq + lane;          // value channel (TMEM lane)
    const int cbase = 64 * ch;             // this thread's key channels
    const uint32_t lanebase = (uint32_t)(32 * jq) << 16;
    const int64_t slot_stride = (int64_t)H * kD * kD;
    const int64_t head_off = (int64_t)h * kD * kD;

    float S[64];
    if (init >= 0) {
        const float* S0 = a.pool + (int64_t)init * slot_stride + head_off;
#pragma unroll
        for (int i = 0; i < 64; ++i) S[i] = S0[(int64_t)(cbase + i) * kD + j];
    } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) S[i] = 0.f;
    }
    auto write_sa = [&]() {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const uint4 v = make_uint4(pack_bf16(S[8 * m], S[8 * m + 1]), pack_bf16(S[8 * m + 2], S[8 * m + 3]),
                                       pack_bf16(S[8 * m + 4], S[8 * m + 5]), pack_bf16(S[8 * m + 6], S[8 * m + 7]));
            sts16(s_base + kSa + kmajor_off(j, cbase + 8 * m, kD), v);
        }
    };
    write_sa();

    if (warp == 0) tmem_alloc(&ms.tslot, 256);
    if (tid == 0) {
        mbar_init(&ms.bar_load[0], 1);
        mbar_init(&ms.bar_load[1], 1);
        mbar_init(&ms.bar_mma, 1);
        fence_mbar_init();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = ms.tslot;
    const uint32_t tD1 = tbase, tD2 = tbase + 64, tD3 = tbase + 128;

    auto rec_ptr = [&](int64_t lc) -> const uint8_t* {
        return p.records + ((size_t)(g0 + lc) * H + h) * kRecBytes;
    };
    if (tid == 0 && nc > 0) {
        mbar_expect_tx(&ms.bar_load[0], kRecBytes);
        bulk_g2s(sm + kStage0, rec_ptr(0), kRecBytes, &ms.bar_load[0]);
    }
    int64_t loads_issued = nc > 0 ? 1 : 0, loads_done = 0;   // uniform / per thread
    uint32_t mma_issued = 0, mma_done = 0;                    // commits issued / waited

    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.o);
    uint32_t mma_parity = 0;
    bool failed = false;
    for (int64_t lc = 0; lc < nc; ++lc) {
        const int st = (int)(lc & 1);
        const uint32_t stage = s_base + kStage0 + st * kStageStride;
        const uint8_t* stage_p = sm + kStage0 + st * kStageStride;
        if (lc + 1 < nc) {
            if (tid == 0) {
                mbar_expect_tx(&ms.bar_load[st ^ 1], kRecBytes);
                bulk_g2s(sm + kStage0 + (st ^ 1) * kStageStride, rec_ptr(lc + 1), kRecBytes, &ms.bar_load[st ^ 1]);
            }
            loads_issued = lc + 2;
        }
        bool ok = mbar_wait(&ms.bar_load[st], (uint32_t)((lc >> 1) & 1));
        if (ok) loads_done = lc + 1;
        if (ok) mma_issued += 1;
        if (tid == 0 && ok) {
            const uint32_t id64 = idesc_bf16(128, 64, false, true);
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const uint64_t ad = sdesc(s_base + kSa + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                mma_bf16(tD1, ad, sdesc(stage + kRecW + ks * 2048, 1024, 1024), id64, ks > 0 ? 1u : 0u);
            }
            mma_commit(&ms.bar_mma);
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const uint64_t ad = sdesc(s_base + kSa + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                mma_bf16(tD2, ad, sdesc(stage + kRecQ + ks * 2048, 1024, 1024), id64, ks > 0 ? 1u : 0u);
            }
        }
        ok = ok && mbar_wait(&ms.bar_mma, mma_parity);
        if (ok) {
            mma_parity ^= 1;
            mma_done += 1;
        }
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        fence_after_sync();

        // (a) epilogue: U^T = U~^T - D1 for this thread's 32 tokens
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t v[16];
            tmem_ld16(tD1 + lanebase + 32 * ch + 16 * hf, v);
            tmem_wait_ld();
#pragma unroll
            for (int e8 = 0; e8 < 2; ++e8) {
                const int cc = 4 * ch + 2 * hf + e8;
                const uint4 ut = *reinterpret_cast<const uint4*>(stage_p + kRecU + row64_chunk_off(j, cc));
                const uint32_t uw[4] = {ut.x, ut.y, ut.z, ut.w};
                uint32_t outw[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float u0 = __uint_as_float(uw[e2] << 16) - __uint_as_float(v[8 * e8 + 2 * e2]);
                    const float u1 = __uint_as_float(uw[e2] & 0xFFFF0000u) - __uint_as_float(v[8 * e8 + 2 * e2 + 1]);
                    outw[e2] = pack_bf16(u0, u1);
                }
                st_shared_v4(s_base + kUa + row64_chunk_off(j, cc), outw[0], outw[1], outw[2], outw[3]);
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        if (tid == 0) {
            const uint32_t id64 = idesc_bf16(128, 64, false, true);
            const uint32_t id128 = idesc_bf16(128, 128, false, false);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks) {
                const uint64_t ad = sdesc(s_base + kUa + ks * 32, 16, 1024);
                mma_bf16(tD2, ad, sdesc(stage + kRecP + ks * 2048, 1024, 1024), id64, 1u);
            }
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks) {
                const uint64_t ad = sdesc(s_base + kUa + ks * 32, 16, 1024);
                mma_bf16(tD3, ad, sdesc(stage + kRecK + ks * 32, 16, 1024), id128, ks > 0 ? 1u : 0u);
            }
            mma_commit(&ms.bar_mma);
        }
        mma_issued += 1;
        ok = mbar_wait(&ms.bar_mma, mma_parity);
        if (ok) {
            mma_parity ^= 1;
            mma_done += 1;
        }
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        fence_after_sync();

        // (d) epilogue: S <- gamma * S + D3 ; bf16 copy for the next chunk
        const float* gam = reinterpret_cast<const float*>(stage_p + kRecG) + cbase;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t v[16];
            tmem_ld16(tD3 + lanebase + cbase + 16 * q4, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) S[16 * q4 + e] = fmaf(gam[16 * q4 + e], S[16 * q4 + e], __uint_as_float(v[e]));
        }
        write_sa();
        const int64_t t0 = tb + lc * kC;
        const int n = (int)(te - t0 < kC ? te - t0 : kC);
        const int64_t p_end = pos0 + lc * kC + n;
        if (a.snap_table && p_end % a.snap_interval == 0) {
            const int64_t ord = p_end / a.snap_interval - 1;
            if (ord >= a.snap_table_stride) {
                if (tid == 0) flag(p.status, KDA_DEV_BAD_ORDINAL);
            } else {
                const int32_t slot = a.snap_table[(int64_t)seq * a.snap_table_stride + ord];
                if (slot >= 0 && (int64_t)slot < a.n_slots) {
                    float* dst = a.pool + (int64_t)slot * slot_stride + head_off;
#pragma unroll
                    for (int i = 0; i < 64; ++i) dst[(int64_t)(cbase + i) * kD + j] = S[i];
                } else if (slot != -1 && tid == 0) {
                    flag(p.status, KDA_DEV_BAD_SLOT);
                }
            }
        }
        // (c) epilogue: outputs of this thread's 32 tokens
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t v[16];
            tmem_ld16(tD2 + lanebase + 32 * ch + 16 * hf, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int t = 32 * ch + 16 * hf + e;
                if (t < n) og[((t0 + t) * H + h) * kD + j] = __float2bfloat16_rn(a.scale * __uint_as_float(v[e]));
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }

    if (failed) {
        // let this CTA's own copies and MMAs in flight land (bounded) before
        // the shared memory and tensor memory are released
        if (tid == 0) {
            flag(p.status, KDA_DEV_WAIT_TIMEOUT);
            for (int64_t l = loads_done; l < loads_issued; ++l)
                mbar_wait(&ms.bar_load[l & 1], (uint32_t)((l >> 1) & 1));
            for (uint32_t m = mma_done; m < mma_issued; ++m, mma_parity ^= 1)
                mbar_wait(&ms.bar_mma, mma_parity);
        }
    } else if (a.final_state) {
        float* dst = a.final_state + (int64_t)seq * slot_stride + head_off;
#pragma unroll
        for (int i = 0; i < 64; ++i) dst[(int64_t)(cbase + i) * kD + j] = S[i];
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

}  // namespace

cudaError_t launch_chunk_recur(const ChunkLaunch& p, cudaStream_t s) {
    const int64_t blocks = (int64_t)p.a.n_seqs * p.a.n_heads;
    if (blocks == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(chunk_recur_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    note_launch();
    chunk_recur_kernel<<<(unsigned)blocks, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
