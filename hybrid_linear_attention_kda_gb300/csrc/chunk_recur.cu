// Stage two of the chunked prefill: the fp32 state carried through the chunks of
// one (sequence, head), with snapshots and outputs.
//
// Everything runs transposed so that the value channel j (128 of them) is the
// MMA M dimension and the TMEM lane.  Per chunk, with S^T [j][c] the state:
//   (a) D1 = S^T W^T             U^T = U~^T - D1            (bf16 U^T to smem)
//   (b) D2 = S^T Q~^T
//   (c) D2 += U^T P^T            O^T = D2
//   (d) D3 = U^T Kbar            S^T <- S^T Diag(gamma) + D3  (fp32, registers)
// Thread (j, quarter) keeps 32 fp32 state entries S[c][j] for its quarter of the
// key channels c; the bf16 copy of S^T in shared memory is the A operand of (a) and
// (b).  The chunk records written by stage one arrive with bulk copies, two
// chunks in flight.  The output accumulator is double-buffered so that the
// outputs of one chunk are stored while the next chunk's MMAs run.  A snapshot is written after every chunk that ends at an
// absolute position that is a multiple of snap_interval ("Kimi K3 Tech Intro",
// sections 2.2-2.4), straight from the fp32 registers.
#include "chunk_common.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int kThreads = 512;      // 16 warps: 4 lane quarters x 4 key-channel quarters
constexpr uint32_t kSa = 0;               // S^T bf16, K-major [j][c], two 64-wide regions
constexpr uint32_t kUa = 32768;           // U^T bf16, K-major [j][t]
constexpr uint32_t kStage0 = 49152;
constexpr uint32_t kStageStride = 74752;  // kRecBytes rounded up to 1024
constexpr uint32_t kMisc = kStage0 + 2 * kStageStride;
constexpr size_t kSmemBytes = kMisc + 64 + 1024;

constexpr uint32_t kTmemCols = 512;       // [D1 | D2] x 2 at [0,128) and [128,256), D3 [256,384)

struct Misc {
    uint64_t bar_load[2];
    uint64_t bar_a;
    uint64_t bar_cd;
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
    const int cbase = 32 * ch;             // this thread's 32 key channels
    const int tq = 16 * ch;                // and its 16 tokens in the per-token epilogues
    const uint32_t lanebase = (uint32_t)(32 * jq) << 16;
    const int64_t slot_stride = (int64_t)H * kD * kD;
    const int64_t head_off = (int64_t)h * kD * kD;

    float S[32];
    if (init >= 0) {
        const float* S0 = a.pool + (int64_t)init * slot_stride + head_off;
#pragma unroll
        for (int i = 0; i < 32; ++i) S[i] = S0[(int64_t)(cbase + i) * kD + j];
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) S[i] = 0.f;
    }
    auto write_sa = [&]() {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const uint4 v = make_uint4(pack_bf16(S[8 * m], S[8 * m + 1]), pack_bf16(S[8 * m + 2], S[8 * m + 3]),
                                       pack_bf16(S[8 * m + 4], S[8 * m + 5]), pack_bf16(S[8 * m + 6], S[8 * m + 7]));
            sts16(s_base + kSa + kmajor_off(j, cbase + 8 * m, kD), v);
        }
    };
    write_sa();

    if (warp == 0) tmem_alloc(&ms.tslot, kTmemCols);
    if (tid == 0) {
        mbar_init(&ms.bar_load[0], 1);
        mbar_init(&ms.bar_load[1], 1);
        mbar_init(&ms.bar_a, 1);
        mbar_init(&ms.bar_cd, 1);
        fence_mbar_init();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = ms.tslot;
    const uint32_t tD3 = tbase + 256;
    // [D1 | D2] of chunk lc: one N = 128 accumulator, double-buffered
    auto tD1 = [&](int64_t lc) -> uint32_t { return tbase + 128 * (uint32_t)(lc & 1); };
    auto tD2 = [&](int64_t lc) -> uint32_t { return tbase + 128 * (uint32_t)(lc & 1) + 64; };

    // Thread 0 issues every copy and MMA and keeps the counts needed to drain
    // them if a wait ever times out.
    uint32_t ld_issued[2] = {0, 0}, ld_waited[2] = {0, 0};
    uint32_t a_issued = 0, a_waited = 0, cd_issued = 0, cd_waited = 0;
    auto rec_ptr = [&](int64_t lc) -> const uint8_t* {
        return p.records + ((size_t)(g0 + lc) * H + h) * kRecBytes;
    };
    auto stage_addr = [&](int64_t lc) -> uint32_t { return s_base + kStage0 + (uint32_t)(lc & 1) * kStageStride; };
    auto issue_load = [&](int64_t lc) {
        const int st = (int)(lc & 1);
        mbar_expect_tx(&ms.bar_load[st], kRecBytes);
        bulk_g2s(sm + kStage0 + st * kStageStride, rec_ptr(lc), kRecBytes, &ms.bar_load[st]);
        ld_issued[st] += 1;
    };
    const uint32_t id64 = idesc_bf16(128, 64, false, true);
    const uint32_t id128mn = idesc_bf16(128, 128, false, true);
    const uint32_t id128 = idesc_bf16(128, 128, false, false);
    // Descriptors are built once; a k-step only moves the start address, which
    // is the low 14-bit field (address >> 4; every operand here lies below
    // 256 KiB, so adding the step never carries out of the field).
    const uint64_t dSa = sdesc(s_base + kSa, 16, 1024);
    const uint64_t dUa = sdesc(s_base + kUa, 16, 1024);
    const uint64_t dMN = sdesc(0, 1024, 1024);       // MN-major record tile, start added per use
    // W and Q~ tiles are adjacent in the record (16 KiB apart): one MN-major
    // operand of N = 128 whose two 64-wide blocks are 16 KiB apart
    static_assert(kRecQ == kRecW + 16384, "record layout");
    const uint64_t dWQ = sdesc(0, 16384, 1024);
    const uint64_t dKM = sdesc(0, 16, 1024);         // K-major record tile
    auto at = [](uint64_t desc, uint32_t byte_off) -> uint64_t { return desc + (uint64_t)(byte_off >> 4); };
    // (a) D1 = S^T W^T and (b) D2 = S^T Q~^T for chunk lc, as one N = 128 MMA chain
    auto issue_ab = [&](int64_t lc) {
        const uint32_t stage = stage_addr(lc);
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
            mma_bf16(tD1(lc), at(dSa, (ks >> 2) * 16384 + (ks & 3) * 32), at(dWQ, stage + kRecW + ks * 2048),
                     id128mn, ks > 0 ? 1u : 0u);
        mma_commit(&ms.bar_a);
        a_issued += 1;
    };
    // (c) D2 += U^T P^T and (d) D3 = U^T Kbar for chunk lc
    auto issue_cd = [&](int64_t lc) {
        const uint32_t stage = stage_addr(lc);
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tD2(lc), at(dUa, ks * 32), at(dMN, stage + kRecP + ks * 2048), id64, 1u);
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks)
            mma_bf16(tD3, at(dUa, ks * 32), at(dKM, stage + kRecK + ks * 32), id128, ks > 0 ? 1u : 0u);
        mma_commit(&ms.bar_cd);
        cd_issued += 1;
    };
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.o);
    // outputs of chunk lc (its O^T is complete in D2(lc)): this thread's 16 tokens
    auto store_outputs = [&](int64_t lc) {
        const int64_t t0 = tb + lc * kC;
        const int n = (int)(te - t0 < kC ? te - t0 : kC);
        uint32_t v[16];
        tmem_ld16(tD2(lc) + lanebase + tq, v);
        tmem_wait_ld();
        __nv_bfloat16* orow = og + ((t0 + tq) * H + h) * kD + j;
        const int64_t ostride = (int64_t)H * kD;
#pragma unroll
        for (int e = 0; e < 16; ++e)
            if (tq + e < n) orow[e * ostride] = __float2bfloat16_rn(a.scale * __uint_as_float(v[e]));
    };

    bool ok = true;
    if (tid == 0 && nc > 0) {
        issue_load(0);
        if (nc > 1) issue_load(1);
        ok = mbar_wait(&ms.bar_load[0], 0);
        if (ok) {
            ld_waited[0] = 1;
            issue_ab(0);
        }
    }
    ok = !__syncthreads_or(!ok);
    for (int64_t lc = 0; lc < nc && ok; ++lc) {
        const int st = (int)(lc & 1);
        const uint8_t* stage_p = sm + kStage0 + st * kStageStride;
        const uint32_t par = (uint32_t)(lc & 1);
        // the record of chunk lc has landed (thread 0 saw it before issuing (a))
        ok = mbar_wait(&ms.bar_load[st], (uint32_t)((lc >> 1) & 1)) && mbar_wait(&ms.bar_a, par);
        if (tid == 0 && ok) a_waited += 1;
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        fence_after_sync();

        // (a) epilogue: U^T = U~^T - D1 for this thread's 16 tokens
        {
            uint32_t v[16];
            tmem_ld16(tD1(lc) + lanebase + tq, v);
            tmem_wait_ld();
#pragma unroll
            for (int e8 = 0; e8 < 2; ++e8) {
                const int cc = 2 * ch + e8;
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
        if (tid == 0) issue_cd(lc);

        // outputs of the previous chunk while (c) and (d) run
        if (lc > 0) store_outputs(lc - 1);

        ok = mbar_wait(&ms.bar_cd, par);
        if (tid == 0 && ok) cd_waited += 1;
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        fence_after_sync();

        // (d) epilogue: S <- gamma * S + D3 ; bf16 copy for the next chunk
        const float* gam = reinterpret_cast<const float*>(stage_p + kRecG) + cbase;
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
            uint32_t v[16];
            tmem_ld16(tD3 + lanebase + cbase + 16 * q4, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) S[16 * q4 + e] = fmaf(gam[16 * q4 + e], S[16 * q4 + e], __uint_as_float(v[e]));
        }
        write_sa();
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        // stage st is free again: refill it two chunks ahead; start the next chunk
        if (tid == 0) {
            if (lc + 2 < nc) issue_load(lc + 2);
            if (lc + 1 < nc) {
                const int st1 = st ^ 1;
                if (mbar_wait(&ms.bar_load[st1], (uint32_t)(((lc + 1) >> 1) & 1))) {
                    ld_waited[st1] += 1;
                    issue_ab(lc + 1);
                }
            }
        }

        // snapshot after this chunk, straight from the fp32 registers
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
                    for (int i = 0; i < 32; ++i) dst[(int64_t)(cbase + i) * kD + j] = S[i];
                } else if (slot != -1 && tid == 0) {
                    flag(p.status, KDA_DEV_BAD_SLOT);
                }
            }
        }
    }

    if (!ok) {
        // let this CTA's own copies and MMAs in flight land (bounded) before
        // the shared memory and tensor memory are released
        if (tid == 0) {
            flag(p.status, KDA_DEV_WAIT_TIMEOUT);
            for (int st = 0; st < 2; ++st)
                for (uint32_t l = ld_waited[st]; l < ld_issued[st]; ++l) mbar_wait(&ms.bar_load[st], l & 1);
            for (uint32_t m = a_waited; m < a_issued; ++m) mbar_wait(&ms.bar_a, m & 1);
            for (uint32_t m = cd_waited; m < cd_issued; ++m) mbar_wait(&ms.bar_cd, m & 1);
        }
    } else {
        if (nc > 0) store_outputs(nc - 1);
        if (a.final_state) {
            float* dst = a.final_state + (int64_t)seq * slot_stride + head_off;
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[(int64_t)(cbase + i) * kD + j] = S[i];
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
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
