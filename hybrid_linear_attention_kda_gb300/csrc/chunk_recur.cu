// Stage two of the chunked prefill: the fp32 state carried through the chunks of
// one (sequence, head), with snapshots and outputs.
//
// Everything runs transposed so that the value channel j (128 of them) is the
// MMA M dimension and the TMEM lane.  Per chunk, with S^T [j][c] the state:
//   (ab) [D1 | D2] = S^T [W^T | Q~^T]        one N = 128 MMA chain
//   (d)  D3  = U^T Kbar                       U^T = U~^T - D1 (bf16, smem)
//   (c)  D2 += U^T P^T                        O^T = D2
//   then S^T <- S^T Diag(gamma) + D3          fp32, registers
// The chain that carries the state is (ab) -> U -> (d) -> S -> next (ab); (c)
// and the outputs run beside it.  The CTA is split by role:
//   warps 0-7   state group: thread (j, half) keeps 64 fp32 entries S[c][j] for
//               its half of the key channels, builds U^T and the bf16 copy of
//               S^T (the A operand of (ab)), writes snapshots
//               ("Kimi K3 Tech Intro", sections 2.2-2.4) and the final state;
//   warps 8-11  output group: O^T from TMEM to the packed output;
//   warp 12     one thread issues the record copies (two chunks in flight) and
//               every MMA, in dependency order, through mbarriers.
// [D1 | D2] is double-buffered in TMEM so the outputs of one chunk are read while
// the next chunk's MMAs run.  Every mbarrier wait is placed where the barrier can
// be at most one phase ahead of it, as parity waits require.
#include "chunk_common.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int kStateWarps = 8, kOutWarps = 4;
constexpr int kThreads = 32 * (kStateWarps + kOutWarps + 1);
constexpr int kIssuerWarp = kStateWarps + kOutWarps;
constexpr uint32_t kSa = 0;               // S^T bf16, K-major [j][c], two 64-wide regions
constexpr uint32_t kUa = 32768;           // U^T bf16, K-major [j][t]
constexpr uint32_t kStage0 = 49152;
constexpr uint32_t kStageStride = 74752;  // kRecBytes rounded up to 1024
constexpr uint32_t kMisc = kStage0 + 2 * kStageStride;
constexpr size_t kSmemBytes = kMisc + 128 + 1024;
constexpr uint32_t kTmemCols = 512;       // [D1 | D2] x 2 at [0,128) and [128,256), D3 [256,384),
                                          // snapshot staging [384,512)

struct Misc {
    uint64_t bar_load[2];   // record copies (tx bytes)
    uint64_t bar_ab;        // MMA commit after (ab)
    uint64_t bar_d;         // MMA commit after (d)
    uint64_t bar_c;         // MMA commit after (c)
    uint64_t bar_u;         // state group: U^T written            (256 arrivals)
    uint64_t bar_s;         // state group: bf16 S^T written        (256 arrivals)
    uint64_t bar_o;         // output group: D2 read from TMEM     (128 arrivals)
    uint64_t bar_snap;      // state group: snapshot staged in TMEM (256 arrivals)
    uint64_t bar_snapfree;  // output group: staged snapshot written out (128 arrivals)
    uint32_t tslot;
    int32_t failed;
    int32_t map_stop;       // segment map: the state became exactly zero, so stays zero
};

static_assert(sizeof(Misc) <= 128, "barrier block");

__device__ __forceinline__ void sts16(uint32_t saddr, uint4 v) { st_shared_v4(saddr, v.x, v.y, v.z, v.w); }

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) chunk_recur_kernel(ChunkLaunch p) {
    griddep_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc& ms = *reinterpret_cast<Misc*>(sm + kMisc);
    const uint32_t s_base = smem_u32(sm);

    const kda_prefill_args& a = p.a;
    const int H = a.n_heads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int mode = MODE;
    const int h = (int)(blockIdx.x % H);
    int seq;
    int64_t coff = 0, ncs = -1;     // this chain's first chunk within its sequence, its chunks
    int32_t scr = -1;               // scratch index of a split segment
    if (mode == kCarryPlain) {
        seq = (int)(blockIdx.x / H);
    } else {
        const int64_t sidx = blockIdx.x / H;
        if (sidx >= p.seg_count[0]) return;
        const int4 si = p.seg_info[sidx];
        seq = si.x;
        coff = si.y;
        ncs = si.z;
        scr = si.w;
        if (mode != kCarryFinal && scr < 0) return;   // only split sequences have segment maps
        const bool first_seg = sidx == p.seg_count[1 + seq];
        const bool final_seg = sidx + 1 == p.seg_count[2 + seq];
        if (mode == kCarryTailMap) {
            // the window before this segment's start (none before the first)
            if (first_seg) return;
            const int64_t w = coff < kTailChunks ? coff : kTailChunks;
            coff -= w;
            ncs = w;
        } else if (mode == kCarryMap || mode == kCarryOffset) {
            if (final_seg) return;                    // no boundary after the last segment
            // the boundary at this segment's end (the next segment's start)
            if (!p.seg_slow[(int64_t)p.seg_info[sidx + 1].w * H + h]) {
                if (mode == kCarryMap) return;        // its tail map is zero: no map needed
                const int64_t w = ncs < kTailChunks ? ncs : kTailChunks;
                coff += ncs - w;                      // the offset over the tail window only
                ncs = w;
            }
        }
    }
    int64_t tb, te, pos0;
    int32_t init;
    uint32_t bad;
    if (!seq_valid(a, seq, &tb, &te, &pos0, &init, &bad)) return;     // flagged by the meta kernel
    const int64_t g_seq = p.chunk_base[seq];
    const int64_t nc_seq = p.chunk_base[seq + 1] - g_seq;
    if (nc_seq < 0 || g_seq + nc_seq > p.max_chunks) return;
    if (ncs < 0) ncs = nc_seq;
    if (coff < 0 || coff + ncs > nc_seq) return;
    const bool last_seg = coff + ncs == nc_seq;
    const bool writes_out = mode == kCarryPlain || mode == kCarryFinal;
    constexpr bool is_map = mode == kCarryMap || mode == kCarryTailMap;   // identity start, U~ = 0
    const int64_t g0 = g_seq + coff;
    const int64_t nc = ncs;
    tb += coff * kC;                // first packed token and absolute position of this chain
    pos0 += coff * kC;
    const int64_t slot_stride = (int64_t)H * kD * kD;
    const int64_t head_off = (int64_t)h * kD * kD;

    if (warp == 0) tmem_alloc(&ms.tslot, kTmemCols);
    if (tid == 0) {
        mbar_init(&ms.bar_load[0], 1);
        mbar_init(&ms.bar_load[1], 1);
        mbar_init(&ms.bar_ab, 1);
        mbar_init(&ms.bar_d, 1);
        mbar_init(&ms.bar_c, 1);
        mbar_init(&ms.bar_u, 32 * kStateWarps);
        mbar_init(&ms.bar_s, 32 * kStateWarps);
        mbar_init(&ms.bar_o, 32 * kOutWarps);
        mbar_init(&ms.bar_snap, 32 * kStateWarps);
        mbar_init(&ms.bar_snapfree, 32 * kOutWarps);
        ms.failed = 0;
        ms.map_stop = 0;
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = ms.tslot;
    const uint32_t tD3 = tbase + 256;
    const uint32_t tSnap = tbase + 384;       // S^T [j][c] of the latest snapshot
    // [D1 | D2] of chunk lc: one N = 128 accumulator, double-buffered
    auto tD1 = [&](int64_t lc) -> uint32_t { return tbase + 128 * (uint32_t)(lc & 1); };
    auto tD2 = [&](int64_t lc) -> uint32_t { return tbase + 128 * (uint32_t)(lc & 1) + 64; };
    auto stage_of = [&](int64_t lc) -> uint32_t { return kStage0 + (uint32_t)(lc & 1) * kStageStride; };
    // a bounded wait; a timeout marks the CTA failed (every role then stops)
    auto waitb = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_wait(bar, parity)) return true;
        atomicExch(&ms.failed, 1);
        return false;
    };

    // pool slot of the snapshot after chunk lc, or -1 (none, skipped, or a bad
    // index, which `report` flags)
    auto snap_slot = [&](int64_t lc, bool report) -> int32_t {
        if (!a.snap_table || !writes_out) return -1;
        // the state at a split segment's end is the next segment's scanned start:
        // the scan writes that snapshot
        if (scr >= 0 && !last_seg && lc == nc - 1) return -1;
        const int64_t t0 = tb + lc * kC;
        const int n = (int)(te - t0 < kC ? te - t0 : kC);
        const int64_t p_end = pos0 + lc * kC + n;
        if (p_end % a.snap_interval != 0) return -1;
        const int64_t ord = p_end / a.snap_interval - 1;
        if (ord >= a.snap_table_stride) {
            if (report) flag(p.status, KDA_DEV_BAD_ORDINAL);
            return -1;
        }
        const int32_t slot = a.snap_table[(int64_t)seq * a.snap_table_stride + ord];
        if (slot >= 0 && (int64_t)slot < a.n_slots) return slot;
        if (slot != -1 && report) flag(p.status, KDA_DEV_BAD_SLOT);
        return -1;
    };

    if (warp == kIssuerWarp) {
        // ------------------------------------------------------------------ issuer
        if (lane == 0) {
            uint32_t ld_issued[2] = {0, 0}, ld_waited[2] = {0, 0};
            uint32_t n_c = 0, w_c = 0;      // commits after (c) issued / waited by this thread
            const uint32_t id128mn = idesc_bf16(128, 128, false, true);
            const uint32_t id64 = idesc_bf16(128, 64, false, true);
            const uint32_t id128 = idesc_bf16(128, 128, false, false);
            // Descriptors are built once; a k-step only moves the start address,
            // the low 14-bit field (address >> 4; all operands lie below 256 KiB,
            // so adding a step never carries out of the field).
            const uint64_t dSa = sdesc(s_base + kSa, 16, 1024);
            const uint64_t dUa = sdesc(s_base + kUa, 16, 1024);
            const uint64_t dMN = sdesc(0, 1024, 1024);
            const uint64_t dKM = sdesc(0, 16, 1024);
            // W and Q~ tiles are adjacent in the record (16 KiB apart): one
            // MN-major operand of N = 128 whose two 64-wide blocks are 16 KiB apart
            static_assert(kRecQ == kRecW + 16384, "record layout");
            const uint64_t dWQ = sdesc(0, 16384, 1024);
            auto at = [](uint64_t desc, uint32_t byte_off) -> uint64_t { return desc + (uint64_t)(byte_off >> 4); };
            auto load = [&](int64_t lc) {
                const int st = (int)(lc & 1);
                mbar_expect_tx(&ms.bar_load[st], kRecBytes);
                bulk_g2s(sm + stage_of(lc), p.records + ((size_t)(g0 + lc) * H + h) * kRecBytes, kRecBytes,
                         &ms.bar_load[st]);
                ld_issued[st] += 1;
            };
            auto wait_load = [&](int64_t lc) -> bool {
                const int st = (int)(lc & 1);
                if (!waitb(&ms.bar_load[st], (uint32_t)((lc >> 1) & 1))) return false;
                ld_waited[st] += 1;
                return true;
            };
            auto issue_ab = [&](int64_t lc) {
                const uint32_t stage = s_base + stage_of(lc);
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    mma_bf16(tD1(lc), at(dSa, (ks >> 2) * 16384 + (ks & 3) * 32), at(dWQ, stage + kRecW + ks * 2048),
                             id128mn, ks > 0 ? 1u : 0u);
                mma_commit(&ms.bar_ab);
            };
            // (d): D3 = U^T Kbar, on the state chain; then (c): D2 += U^T P^T,
            // which runs while the state group updates S
            auto issue_dc = [&](int64_t lc) {
                const uint32_t stage = s_base + stage_of(lc);
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_bf16(tD3, at(dUa, ks * 32), at(dKM, stage + kRecK + ks * 32), id128, ks > 0 ? 1u : 0u);
                mma_commit(&ms.bar_d);
                if (!writes_out) return;            // the map / offset passes need no outputs
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_bf16(tD2(lc), at(dUa, ks * 32), at(dMN, stage + kRecP + ks * 2048), id64, 1u);
                mma_commit(&ms.bar_c);
                n_c += 1;
            };
            bool ok = true, stopped = false;
            if (nc > 0) {
                load(0);
                if (nc > 1) load(1);
                ok = waitb(&ms.bar_s, 0) && wait_load(0);           // initial bf16 state and record 0
                if (ok) issue_ab(0);
            }
            for (int64_t lc = 0; lc < nc && ok; ++lc) {
                const uint32_t par = (uint32_t)(lc & 1);
                if (!(ok = waitb(&ms.bar_u, par))) break;          // U^T of lc written
                // D2 of lc-1 read by the output group.  Waiting here, before (c) of
                // lc is issued, keeps that barrier at most one phase ahead of this
                // wait; the buffer is reused by (ab) of lc+1.
                if (writes_out && lc >= 1 && !(ok = waitb(&ms.bar_o, par ^ 1))) break;
                fence_after_sync();
                issue_dc(lc);
                if (!(ok = waitb(&ms.bar_s, par ^ 1))) break;      // state after lc written
                // every MMA of lc done: the state group has consumed (ab) and (d);
                // (c) runs only when outputs are written
                if (writes_out) {
                    if (!(ok = waitb(&ms.bar_c, par))) break;
                    w_c += 1;
                } else if (is_map && ms.map_stop) {
                    stopped = true;                                 // the map is zero from here on
                    break;
                }
                fence_after_sync();
                if (lc + 2 < nc) load(lc + 2);                      // record stage of lc is free
                if (lc + 1 < nc) {
                    if (!(ok = wait_load(lc + 1))) break;
                    issue_ab(lc + 1);
                }
            }
            if (!ok || stopped) {
                // let this CTA's own copies (and, on a failure, MMAs) land
                // (bounded) before shared and tensor memory are released
                for (int st = 0; st < 2; ++st)
                    for (uint32_t l = ld_waited[st]; l < ld_issued[st]; ++l) mbar_wait(&ms.bar_load[st], l & 1);
            }
            if (!ok) {
                for (uint32_t m = w_c; m < n_c; ++m) mbar_wait(&ms.bar_c, m & 1);
            }
        }
    } else if (warp < kStateWarps) {
        // ------------------------------------------------------------------ state group
        const int jq = warp & 3, ch = warp >> 2;
        const int j = 32 * jq + lane;          // value channel (TMEM lane)
        const int cbase = 64 * ch;             // this thread's 64 key channels
        const int tq = 32 * ch;                // and its 32 tokens in the U epilogue
        const uint32_t lanebase = (uint32_t)(32 * jq) << 16;
        float S[64];
        const float* S0 = nullptr;
        if (mode == kCarryFinal && scr >= 0) S0 = p.seg_state + ((int64_t)scr * H * 3 + (int64_t)h * 3 + 2) * kD * kD;
        else if ((mode == kCarryPlain || mode == kCarryFinal) && init >= 0) S0 = a.pool + (int64_t)init * slot_stride + head_off;
        if (S0) {
#pragma unroll
            for (int i = 0; i < 64; ++i) S[i] = S0[(int64_t)(cbase + i) * kD + j];
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) S[i] = (is_map && cbase + i == j) ? 1.f : 0.f;
        }
        auto write_sa = [&]() {
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint4 v = make_uint4(pack_bf16(S[8 * m], S[8 * m + 1]), pack_bf16(S[8 * m + 2], S[8 * m + 3]),
                                           pack_bf16(S[8 * m + 4], S[8 * m + 5]), pack_bf16(S[8 * m + 6], S[8 * m + 7]));
                sts16(s_base + kSa + kmajor_off(j, cbase + 8 * m, kD), v);
            }
            fence_async_smem();
            mbar_arrive(&ms.bar_s);
        };
        write_sa();
        bool ok = true;
        uint32_t n_snap = 0;
        for (int64_t lc = 0; lc < nc; ++lc) {
            const uint32_t par = (uint32_t)(lc & 1);
            const uint8_t* stage_p = sm + stage_of(lc);
            if (!(ok = waitb(&ms.bar_load[lc & 1], (uint32_t)((lc >> 1) & 1)) && waitb(&ms.bar_ab, par))) break;
            fence_after_sync();
            // U^T = U~^T - D1 for this thread's 32 tokens
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t v[16];
                tmem_ld16(tD1(lc) + lanebase + tq + 16 * hf, v);
                tmem_wait_ld();
#pragma unroll
                for (int e8 = 0; e8 < 2; ++e8) {
                    const int cc = 4 * ch + 2 * hf + e8;
                    // the segment map runs with U~ = 0
                    const uint4 ut = is_map ? make_uint4(0u, 0u, 0u, 0u)
                                                       : *reinterpret_cast<const uint4*>(stage_p + kRecU + row64_chunk_off(j, cc));
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
            mbar_arrive(&ms.bar_u);
            if (!(ok = waitb(&ms.bar_d, par))) break;
            fence_after_sync();
            // S <- gamma * S + D3, then the bf16 copy for the next chunk
            const float* gam = reinterpret_cast<const float*>(stage_p + kRecG) + cbase;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t v[16];
                tmem_ld16(tD3 + lanebase + cbase + 16 * q4, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    S[16 * q4 + e] = fmaf(gam[16 * q4 + e], S[16 * q4 + e], __uint_as_float(v[e]));
            }
            fence_before_sync();
            // the segment map: once the state is exactly zero every later chunk
            // keeps it zero, so the map of the whole segment is zero and the pass
            // stops (an AND over the 256 state threads at named barrier 3)
            bool map_zero = false;
            if (is_map) {
                uint32_t z = 1;
#pragma unroll
                for (int i = 0; i < 64; ++i) z &= S[i] == 0.f ? 1u : 0u;
                uint32_t all;
                asm volatile(
                    "{\n\t.reg .pred p, q;\n\t"
                    "setp.ne.u32 p, %1, 0;\n\t"
                    "bar.red.and.pred q, 3, 256, p;\n\t"
                    "selp.u32 %0, 1, 0, q;\n\t}"
                    : "=r"(all)
                    : "r"(z)
                    : "memory");
                map_zero = all != 0;
                if (map_zero && tid == 0) ms.map_stop = 1;
            }
            write_sa();
            if (map_zero) break;
            // snapshot after this chunk: the fp32 state goes to the snapshot
            // columns of TMEM (lane j, column c); the output group writes it to
            // the pool, off this chain
            if (snap_slot(lc, tid == 0) >= 0) {
                if (n_snap > 0 && !(ok = waitb(&ms.bar_snapfree, (n_snap - 1) & 1))) break;
                fence_after_sync();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(S[16 * q4 + e]);
                    tmem_st16(tSnap + lanebase + cbase + 16 * q4, v);
                }
                tmem_wait_st();
                fence_before_sync();
                mbar_arrive(&ms.bar_snap);
                n_snap += 1;
            }
        }
        float* dst = nullptr;
        if (mode == kCarryMap || mode == kCarryOffset)
            dst = p.seg_state + ((int64_t)scr * H * 3 + (int64_t)h * 3 + (mode == kCarryMap ? 0 : 1)) * kD * kD;
        else if (writes_out && last_seg && a.final_state)
            dst = a.final_state + (int64_t)seq * slot_stride + head_off;
        // the boundary's choice: a tail window that did not map every state to
        // exactly zero takes the full map / offset / scan
        if (mode == kCarryTailMap && tid == 0) p.seg_slow[(int64_t)scr * H + h] = (ok && ms.map_stop) ? 0 : 1;
        if (ok && dst) {
#pragma unroll
            for (int i = 0; i < 64; ++i) dst[(int64_t)(cbase + i) * kD + j] = S[i];
        }
    } else {
        // ------------------------------------------------------------------ output group
        const int jq = warp & 3;
        const int j = 32 * jq + lane;
        const uint32_t lanebase = (uint32_t)(32 * jq) << 16;
        __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.o);
        const int64_t ostride = (int64_t)H * kD;
        uint32_t n_snap = 0;
        // the map and offset passes write no outputs: (c) is not issued there
        for (int64_t lc = 0; lc < nc && writes_out; ++lc) {
            if (!waitb(&ms.bar_c, (uint32_t)(lc & 1))) break;
            fence_after_sync();
            uint32_t v[4][16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_ld16(tD2(lc) + lanebase + 16 * q4, v[q4]);
            tmem_wait_ld();
            fence_before_sync();
            mbar_arrive(&ms.bar_o);
            const int64_t t0 = tb + lc * kC;
            const int n = (int)(te - t0 < kC ? te - t0 : kC);
            __nv_bfloat16* orow = og + (t0 * H + h) * kD + j;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (writes_out && 16 * q4 + e < n)
                        orow[(16 * q4 + e) * ostride] = __float2bfloat16_rn(a.scale * __uint_as_float(v[q4][e]));
            }
            // a snapshot after this chunk: from the TMEM staging to the pool's [c][j] layout
            const int32_t slot = snap_slot(lc, false);
            if (slot >= 0) {
                if (!waitb(&ms.bar_snap, n_snap & 1)) break;
                fence_after_sync();
                float* dst = a.pool + (int64_t)slot * slot_stride + head_off + j;
#pragma unroll 2
                for (int q = 0; q < 8; ++q) {
                    uint32_t sv[16];
                    tmem_ld16(tSnap + lanebase + 16 * q, sv);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) dst[(int64_t)(16 * q + e) * kD] = __uint_as_float(sv[e]);
                }
                fence_before_sync();
                mbar_arrive(&ms.bar_snapfree);
                n_snap += 1;
            }
        }
    }

    if (ms.failed && tid == 0) flag(p.status, KDA_DEV_WAIT_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// ---------------------------------------------------------------- segments
// The segment table: a sequence of >= 2 kSegTokens tokens is split at the
// absolute positions that are multiples of kSegTokens (so a run resumed at such
// a position splits the same way); every other sequence is one segment.  A few
// sequences at most take this path (fewer chains than half the SMs), so one
// thread builds the table.
__global__ void segment_meta_kernel(ChunkLaunch p) {
    griddep_wait();
    if (threadIdx.x != 0) return;
    const kda_prefill_args& a = p.a;
    const int64_t max_scr = max_segments(a.total_tokens, a.n_seqs);
    int64_t nseg = 0, nscr = 0;
    for (int s = 0; s < a.n_seqs; ++s) {
        p.seg_count[1 + s] = (int32_t)nseg;
        int64_t tb, te, pos0;
        int32_t init;
        uint32_t bad;
        if (!seq_valid(a, s, &tb, &te, &pos0, &init, &bad)) continue;
        const int64_t nch = p.chunk_base[s + 1] - p.chunk_base[s];
        const int64_t L = te - tb;
        if (nch < 0) continue;
        // an empty sequence is one segment of no chunks: the final pass writes
        // its initial state (a pool slot, or zeros) as its final state
        if (L >= 2 * kSegTokens) {
            for (int64_t start = pos0; start < pos0 + L && nseg < p.max_segs && nscr < max_scr;) {
                const int64_t b = (start / kSegTokens + 1) * kSegTokens;
                const int64_t end = b < pos0 + L ? b : pos0 + L;
                p.seg_info[nseg++] = make_int4(s, (int32_t)((start - pos0) / kC),
                                               (int32_t)((end - start + kC - 1) / kC), (int32_t)nscr++);
                start = end;
            }
        } else if (nseg < p.max_segs) {
            p.seg_info[nseg++] = make_int4(s, 0, (int32_t)nch, -1);
        }
    }
    p.seg_count[1 + a.n_seqs] = (int32_t)nseg;
    p.seg_count[0] = (int32_t)nseg;
}

// Initial states of the segments of one (sequence, head):
//   S_in(0) = the sequence's initial state,  S_in(k) = A_{k-1} S_in(k-1) + B_{k-1}
// in fp32, with the snapshot at each segment boundary taken from S_in (the
// state the next segment continues from).  Each value column of S evolves on
// its own, so a CTA takes one block of kScanCols columns of one (sequence, head);
// each step stages A_{k-1} in shared memory.
constexpr int kScanThreads = 256;
constexpr int kScanCols = 16;
constexpr int kScanBlocks = kD / kScanCols;

__global__ void __launch_bounds__(kScanThreads) segment_scan_kernel(ChunkLaunch p) {
    griddep_wait();
    extern __shared__ float scan_smem[];
    const kda_prefill_args& a = p.a;
    const int H = a.n_heads;
    const int64_t sh = blockIdx.x / kScanBlocks;
    const int cb = (int)(blockIdx.x % kScanBlocks) * kScanCols;     // first column of this block
    const int seq = (int)(sh / H), h = (int)(sh % H);
    const int tid = threadIdx.x;
    const int32_t s0 = p.seg_count[1 + seq], s1 = p.seg_count[2 + seq];
    if (s1 - s0 < 1 || p.seg_info[s0].w < 0) return;          // not split
    int64_t tb, te, pos0;
    int32_t init;
    uint32_t bad;
    if (!seq_valid(a, seq, &tb, &te, &pos0, &init, &bad)) return;
    constexpr int DD = kD * kD;
    float* Am = scan_smem;                                       // [kD][kD + 4]
    constexpr int kLdA = kD + 4;
    float* Scur = scan_smem + kD * kLdA;                         // [kD][kScanCols]
    const int64_t head_off = (int64_t)h * DD;
    auto seg_state = [&](int32_t scr, int which) { return p.seg_state + ((int64_t)scr * H * 3 + (int64_t)h * 3 + which) * DD; };
    const int j = tid % kScanCols, rg = tid / kScanCols;         // column j, rows rg + 16 m
    {
        const float* S0 = init >= 0 ? a.pool + (int64_t)init * H * DD + head_off : nullptr;
        float* dst = seg_state(p.seg_info[s0].w, 2);
#pragma unroll
        for (int m = 0; m < kD / 16; ++m) {
            const int c = rg + 16 * m;
            const float x = S0 ? S0[c * kD + cb + j] : 0.f;
            Scur[c * kScanCols + j] = x;
            dst[c * kD + cb + j] = x;
        }
    }
    for (int32_t k = s0 + 1; k < s1; ++k) {
        const int32_t prev = p.seg_info[k - 1].w;
        const float* A = seg_state(prev, 0);
        const float* B = seg_state(prev, 1);
        // a boundary whose tail map is zero starts the segment from the tail-window
        // offset B alone
        const bool slow = p.seg_slow[(int64_t)p.seg_info[k].w * H + h] != 0;
        float acc[kD / 16];
#pragma unroll
        for (int m = 0; m < kD / 16; ++m) acc[m] = 0.f;
        if (slow) {
            __syncthreads();                                     // Scur written, Am free
            for (int e = tid; e < DD / 4; e += kScanThreads) {
                const int r = e / (kD / 4), c4 = e % (kD / 4);
                *reinterpret_cast<float4*>(Am + r * kLdA + 4 * c4) = reinterpret_cast<const float4*>(A)[e];
            }
            __syncthreads();
            for (int u = 0; u < kD; u += 4) {
                const float x0 = Scur[u * kScanCols + j], x1 = Scur[(u + 1) * kScanCols + j];
                const float x2 = Scur[(u + 2) * kScanCols + j], x3 = Scur[(u + 3) * kScanCols + j];
#pragma unroll
                for (int m = 0; m < kD / 16; ++m) {
                    const float4 av = *reinterpret_cast<const float4*>(Am + (rg + 16 * m) * kLdA + u);
                    acc[m] = fmaf(av.x, x0, acc[m]);
                    acc[m] = fmaf(av.y, x1, acc[m]);
                    acc[m] = fmaf(av.z, x2, acc[m]);
                    acc[m] = fmaf(av.w, x3, acc[m]);
                }
            }
        }
        // the segment's start state, and the snapshot at that boundary
        const int4 si = p.seg_info[k];
        float* dst = seg_state(si.w, 2);
        const int64_t pstart = pos0 + (int64_t)si.y * kC;
        float* snap = nullptr;
        if (a.snap_table && pstart % a.snap_interval == 0) {
            const int64_t ord = pstart / a.snap_interval - 1;
            if (ord < a.snap_table_stride) {
                const int32_t slot = a.snap_table[(int64_t)seq * a.snap_table_stride + ord];
                if (slot >= 0 && (int64_t)slot < a.n_slots) snap = a.pool + (int64_t)slot * H * DD + head_off;
            }
        }
        __syncthreads();                                         // every read of Scur done
#pragma unroll
        for (int m = 0; m < kD / 16; ++m) {
            const int c = rg + 16 * m;
            const float x = acc[m] + B[c * kD + cb + j];
            Scur[c * kScanCols + j] = x;
            dst[c * kD + cb + j] = x;
            if (snap) snap[c * kD + cb + j] = x;
        }
    }
}

}  // namespace

cudaError_t launch_segment_meta(const ChunkLaunch& p, cudaStream_t s) {
    note_launch();
    return launch_overlapped(segment_meta_kernel, dim3(1), dim3(32), 0, s, p);
}

cudaError_t launch_segment_scan(const ChunkLaunch& p, cudaStream_t s) {
    const int64_t blocks = (int64_t)p.a.n_seqs * p.a.n_heads * kScanBlocks;
    if (blocks == 0) return cudaSuccess;
    const size_t smem = ((size_t)kD * (kD + 4) + (size_t)kD * kScanCols) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(segment_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    note_launch();
    return launch_overlapped(segment_scan_kernel, dim3((unsigned)blocks), dim3(kScanThreads), smem, s, p);
}

template <int MODE>
cudaError_t launch_recur_mode(const ChunkLaunch& p, cudaStream_t s) {
    const int64_t blocks = (MODE == kCarryPlain ? (int64_t)p.a.n_seqs : p.max_segs) * p.a.n_heads;
    if (blocks == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(chunk_recur_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    note_launch();
    return launch_overlapped(chunk_recur_kernel<MODE>, dim3((unsigned)blocks), dim3(kThreads), kSmemBytes, s, p);
}

cudaError_t launch_chunk_recur(const ChunkLaunch& p, cudaStream_t s) {
    switch (p.mode) {
        case kCarryMap: return launch_recur_mode<kCarryMap>(p, s);
        case kCarryOffset: return launch_recur_mode<kCarryOffset>(p, s);
        case kCarryFinal: return launch_recur_mode<kCarryFinal>(p, s);
        case kCarryTailMap: return launch_recur_mode<kCarryTailMap>(p, s);
        default: return launch_recur_mode<kCarryPlain>(p, s);
    }
}

}  // namespace kda
