// Stage one of the chunked prefill: everything of a 64-token chunk that does not
// depend on the carried state, for all (chunk, head) pairs.
//
// A persistent kernel with two co-resident CTAs per SM, each walking its share of
// the (chunk, head) items one at a time: the phases of one CTA (gate products,
// MMA waits, the fp32 inversion, the load of its next item) run beside those of
// the other.  An item's q, k and alpha tiles ([64 tokens x 128 channels], token
// rows H*128 elements apart in the packed tensors) arrive by TMA tensor copies;
// v arrives in the 128-byte-swizzled layout the tensor cores read, as two
// [64 tokens x 64 channels] boxes, and is the A operand of the U~ product as it
// lies.  Once q, k and alpha sit in registers their 64 KiB hold the A/P
// operands, then A and T.  Q~ and Kbar go from registers to the record; P, W and
// U~ are staged in shared memory and leave by bulk copies.
//
// Decay factors are products of alphas over token ranges (no exp / log): with
// the chunk split into halves of 32 tokens and m the 16th token of a half,
//   Gamma_r = prod_{tau <= r} alpha              (chunk prefix, <= 1)
//   kappa_r = prod_{tau > r} alpha               (chunk suffix, <= 1)
//   phi_r   = exp(g_r - g_m)                     (own half's reference token)
//   psi_s   = 1 / phi_s
//   xi_s    = exp(g_47 - g_s)  for s in half 0   (<= 1)
// The intra-chunk products A and P come from one tcgen05 MMA (M = N = K = 128)
// whose rows are key tokens s and whose columns are query / key tokens r:
//   rows 0..63   k_s psi_s     x  cols 0..63    q_r phi_r   -> P within a half
//   rows 64..95  k_s xi_s                                  -> P, r in half 1, s in half 0
//                                 cols 64..127  k_r phi_r   -> A (same rows)
// For r in half 1, phi_r xi_s = exp(g_r - g_s) exactly; where xi_s underflows the
// true entry is below 2^-100 * e^-87 relative to the others.  Within a half phi,
// psi span at most 16 tokens; an item whose factors leave [2^-100, 2^100] is
// listed, and chunk_exact_kernel rewrites its P, W and U~ in fp32 from exact
// products of alphas (chunk_decay.cuh) before the carry reads them.
// T = (I + A)^-1 is inverted
// by 16 x 16 blocks in fp32, then W and U~ come from a second MMA
// (X^T T'^T and V^T T'^T with X = Gamma K and T' = T diag(beta)).
#include <cuda.h>

#include "chunk_common.cuh"
#include "chunk_decay.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 2;              // two co-resident CTAs overlap each other's phases
// Thread 0 waits on the mbarriers and issues the MMAs.  Two other threads issue
// the copies, so that a copy engine that is slow to accept work does not hold up
// thread 0's chain:
constexpr int kStoreThread = 32;           // the W / U~ stores and, after the first item, the v loads
constexpr int kLoadThread = 224;          // warp 7: the P stores (issued while warps 0-1 still invert)
                                           // and, after the first item, the q, k, alpha loads
// Shared memory of one CTA (1024-aligned base), one item at a time.  Channels are
// taken in two rounds of 64; round g's q, k and alpha boxes ([64 tokens][64
// channels], no swizzle) fill region g, which then takes the round's K-slices
// of the A/P operands (channels 64g .. 64g+63).
constexpr uint32_t kRound = 32768;         // region g at g * kRound
constexpr uint32_t kRq = 0, kRk = 8192, kRal = 16384;      // q, k bf16 [64][64]; alpha fp32 [64][64]
constexpr uint32_t kRa = 0, kRb = 16384;   // APa / APb K-slices: MN-major [8-channel group][128 rows]
constexpr uint32_t kSv = 65536;            // v: two 128-byte-swizzled [64 t][64 c] boxes, 8 KiB apart
constexpr uint32_t kVbox = 8192;
constexpr uint32_t kX = 81920;             // X^T = (Gamma k)^T, K-major [c][t]
constexpr uint32_t kLoadBytes = 65536;     // q, k and alpha of one item
constexpr uint32_t kVBytes = 16384;        // its v
constexpr uint32_t kLbo = 1024, kSbo = 2048;
// [0, 64 KiB) once the A/P MMA has read its operands:
constexpr int kAP = 68;                    // row stride (floats) of A and T: rows 4 banks apart
constexpr uint32_t kAmat = 0;              // A fp32 [64][kAP]
constexpr uint32_t kTf = 17408;            // T fp32 [64][kAP]
constexpr uint32_t kTscr = 34816;          // block-product scratch, 1536 fp32
constexpr uint32_t kTm = 98304;            // (T diag(beta))^T bf16, MN-major [s][r]; outside [0, 64 KiB)
                                           // so the next item's q, k, alpha may land while it is read
constexpr uint32_t kPst = 45056;           // P record tile, staged for its bulk store
constexpr uint32_t kWst = kSv;             // after the W/U~ MMA: W and U~ record tiles, staged
                                           // over v and X^T, so the next item's q, k, alpha can land
constexpr uint32_t kMisc = kTm + 8192;
constexpr uint32_t kTmemCols = 128;

struct Misc {
    float beta[2][kC];         // this item's and the next item's beta
    int4 info[2];              // this item's and the next item's chunk-table entry
    float qprod[2][4][64];     // per round: product of alpha over each 16-token quarter, per channel
    uint64_t bar_load;         // q, k and alpha
    uint64_t bar_v;            // v, waited for only by the W / U~ product
    uint64_t bar_mma;
    uint32_t tslot;
    int32_t guard_fail;
    // copies and MMAs issued (thread 0, kStoreThread, kLoadThread) and waited for
    // (thread 0), to drain on a timeout
    uint32_t ld_issued, ld_waited, v_issued, v_waited, mma_issued, mma_waited;
};
constexpr size_t kSmemBytes = kMisc + sizeof(Misc) + 1024;
static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");
static_assert(kLoadThread >= 128 && kLoadThread < kThreads, "the P stores follow warps 4-7's barrier");

struct LocalMaps {
    CUtensorMap q, k, v, alpha;   // 2-D views [T_tot rows x H*128 elements]
};

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    return make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                      pack_bf16(v[6], v[7]));
}
__device__ __forceinline__ void sts16(uint32_t saddr, uint4 v) { st_shared_v4(saddr, v.x, v.y, v.z, v.w); }
__device__ __forceinline__ void stg16(uint8_t* gaddr, uint4 v) { *reinterpret_cast<uint4*>(gaddr) = v; }
// A lane's 16 tokens (chunks 2 qq and 2 qq + 1) of record row `row` in the
// 128-byte-swizzled [row][64 tokens] tile: the two chunks land in one aligned
// 32-byte pair of the row, in swapped order when bit 0 of the row's swizzle is
// set, and leave as one 32-byte store (a full sector per lane).
__device__ __forceinline__ void stg_row_pair(uint8_t* tile, uint32_t row, uint32_t qq, const uint32_t (&lo)[4],
                                             const uint32_t (&hi)[4]) {
    const uint32_t x = row & 7u;
    uint8_t* dst = tile + (row >> 3) * 1024u + x * 128u + (((2u * qq) ^ (x & 6u)) << 4);
    const bool sw = (x & 1u) != 0;
    const uint32_t a0 = sw ? hi[0] : lo[0], a1 = sw ? hi[1] : lo[1], a2 = sw ? hi[2] : lo[2], a3 = sw ? hi[3] : lo[3];
    const uint32_t b0 = sw ? lo[0] : hi[0], b1 = sw ? lo[1] : hi[1], b2 = sw ? lo[2] : hi[2], b3 = sw ? lo[3] : hi[3];
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a0), "r"(a1), "r"(a2),
                 "r"(a3), "r"(b0), "r"(b1), "r"(b2), "r"(b3)
                 : "memory");
}
// two bf16 (low half the even token) times two bf16 factors, rounded once
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t x, uint32_t f) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(f));
    return r;
}

// byte offset of the 16-byte chunk (mn .. mn+7, k) of an MN-major tile
__device__ __forceinline__ uint32_t mn_chunk(uint32_t mn, uint32_t k) {
    return (k >> 3) * kSbo + (mn >> 6) * kLbo + (k & 7u) * 128u + ((((mn & 63u) >> 3) ^ (k & 7u)) << 4);
}

// T = (I + A)^-1 for a strictly lower triangular 64 x 64 A (fp32, rows kAP floats apart),
// by blocks, with T's 16 x 16 blocks T_ij and A's blocks A_ij:
//   stage 1  the four diagonal blocks T_ii by forward substitution (warps 0-1;
//            warps 4-7 run the caller's side work, then meet at named barrier 3
//            and thread kLoadThread, one of them, runs after_stage1);
//   stage 2  T_10 = -T_11 (A_10 T_00) on warps 0 and 2, T_32 = -T_33 (A_32 T_22)
//            on warps 1 and 3 (each pair meets at a named barrier between its two
//            products), while warps 4-7 form the parts of M = A_LL T_00(32) that
//            need only diagonal blocks: A_L0 T_00 (M's columns 0-15, first term)
//            and A_L1 T_11 (columns 16-31), with A_LL = [A_L0 | A_L1] the lower-left
//            32 x 32 block of A;
//   stage 3  M's columns 0-15 += A_L1 T_10;
//   stage 4  T_LL = -T_11(32) M, skipping the zero column groups of the
//            triangular T_11(32) with a bound uniform per warp.
// T's entries above the diagonal are never written and never read.  Each stage
// also writes its entries of T' = T diag(beta) into the bf16 MN-major [s][r]
// operand at tm (stage 1 the diagonal blocks and the zeros above them), so T'
// is complete at the end.  scr holds 1536 floats: M (32 x 32) and two 16 x 16
// scratch blocks.  Ends with a barrier.
template <class Side, class AfterStage1>
__device__ __forceinline__ void invert_unit_lower(const float* A, float* Tf, float* scr, int tid, Side side,
                                                  AfterStage1 after_stage1, uint32_t tm, const float* bsm) {
    const int warp = tid >> 5, lane = tid & 31;
    // entry (r, s) of T' = T diag(beta) into the MN-major [s][r] bf16 operand at tm
    auto put_tp = [&](int r, int s, float t) {
        const __nv_bfloat16 x = __float2bfloat16_rn(t * bsm[s]);
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(tm + row64_chunk_off(s, r >> 3) + (r & 7) * 2),
                     "h"(*reinterpret_cast<const uint16_t*>(&x))
                     : "memory");
    };
    if (tid < kC) {
        const int o = 16 * (tid >> 4), jj = tid & 15;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) t[r] = r == jj ? 1.f : 0.f;
        // columns u in groups of four, read as one 16-byte row piece per row r;
        // each t[r] still takes its updates in increasing u, and rows are visited
        // in increasing order, so every t[u] is final when it is used
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
#pragma unroll
            for (int r = 4 * g4 + 1; r < 16; ++r) {
                const float4 a4 = *reinterpret_cast<const float4*>(A + (o + r) * kAP + o + 4 * g4);
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * g4 + e < r) t[r] = fmaf(-av[e], t[4 * g4 + e], t[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tf[(o + r) * kAP + o + jj] = t[r];
        // T' row s = o + jj: its 16 entries of this diagonal block, and zeros
        // for every r below the block (T is lower triangular)
        const int s = o + jj;
        const float bs = bsm[s];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 8 * h2 + e >= jj ? t[8 * h2 + e] * bs : 0.f;
            sts16(tm + row64_chunk_off(s, (o >> 3) + h2), pack8(x));
        }
#pragma unroll
        for (int cz = 0; cz < 6; ++cz)
            if (cz < (o >> 3)) sts16(tm + row64_chunk_off(s, cz), make_uint4(0u, 0u, 0u, 0u));
    } else if (tid >= 2 * kC) {
        side();       // warps 4-7: work of the caller's that does not depend on T
        // warps 4-7's side work is complete: the caller's follow-up runs on one
        // of them while warps 0-1 still solve the diagonal blocks
        asm volatile("bar.sync 3, 128;" ::: "memory");
        if (tid == kLoadThread) after_stage1();
    }
    __syncthreads();
    float* M = scr;                      // [32][32]: rows 32..63 of A, columns 0..31 of T
    if (warp < 4) {
        // stage 2: warp pair (b, b + 2) forms T_ij, (i, j) = (1, 0) for b = 0, (3, 2) for b = 1
        const int b = warp & 1, pt = (warp >> 1) * 32 + lane;         // 0..63 within the pair
        const int i = 2 * b + 1, j = 2 * b;
        float* X = scr + 1024 + 256 * b;                              // [16][16]
        const int r = pt >> 2, c = 4 * (pt & 3);                      // four outputs X[r][c .. c+3]
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* ar = A + (16 * i + r) * kAP + 16 * j;
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
            const float4 a4 = *reinterpret_cast<const float4*>(ar + 4 * u4);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 t4 = *reinterpret_cast<const float4*>(Tf + (16 * j + 4 * u4 + e) * kAP + 16 * j + c);
                acc.x = fmaf(av[e], t4.x, acc.x);
                acc.y = fmaf(av[e], t4.y, acc.y);
                acc.z = fmaf(av[e], t4.z, acc.z);
                acc.w = fmaf(av[e], t4.w, acc.w);
            }
        }
        *reinterpret_cast<float4*>(X + r * 16 + c) = acc;
        // the pair's X is complete (named barriers 1 and 2, one per pair)
        if (b == 0) asm volatile("bar.sync 1, 64;" ::: "memory");
        else asm volatile("bar.sync 2, 64;" ::: "memory");
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* tr = Tf + (16 * i + r) * kAP + 16 * i;
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
            const float4 t4 = *reinterpret_cast<const float4*>(tr + 4 * u4);
            const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 x4 = *reinterpret_cast<const float4*>(X + (4 * u4 + e) * 16 + c);
                acc.x = fmaf(tv[e], x4.x, acc.x);
                acc.y = fmaf(tv[e], x4.y, acc.y);
                acc.z = fmaf(tv[e], x4.z, acc.z);
                acc.w = fmaf(tv[e], x4.w, acc.w);
            }
        }
        *reinterpret_cast<float4*>(Tf + (16 * i + r) * kAP + 16 * j + c) =
            make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        put_tp(16 * i + r, 16 * j + c, -acc.x);
        put_tp(16 * i + r, 16 * j + c + 1, -acc.y);
        put_tp(16 * i + r, 16 * j + c + 2, -acc.z);
        put_tp(16 * i + r, 16 * j + c + 3, -acc.w);
    } else {
        // stage 2, beside it: M[r][8 cg .. 8 cg + 7] for column groups 0-1 (A_L0 T_00)
        // and 2-3 (A_L1 T_11), each a 16-term product with one row piece of A
        const int tc = tid - 4 * 32, r = tc >> 2, cg = tc & 3, blk = cg >> 1;
        const float* ar = A + (32 + r) * kAP + 16 * blk;
        const float* tb = Tf + (16 * blk) * kAP + 16 * blk + 8 * (cg & 1);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
            const float4 a4 = *reinterpret_cast<const float4*>(ar + 4 * u4);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 t0 = *reinterpret_cast<const float4*>(tb + (4 * u4 + e) * kAP);
                const float4 t1 = *reinterpret_cast<const float4*>(tb + (4 * u4 + e) * kAP + 4);
                acc[0] = fmaf(av[e], t0.x, acc[0]);
                acc[1] = fmaf(av[e], t0.y, acc[1]);
                acc[2] = fmaf(av[e], t0.z, acc[2]);
                acc[3] = fmaf(av[e], t0.w, acc[3]);
                acc[4] = fmaf(av[e], t1.x, acc[4]);
                acc[5] = fmaf(av[e], t1.y, acc[5]);
                acc[6] = fmaf(av[e], t1.z, acc[6]);
                acc[7] = fmaf(av[e], t1.w, acc[7]);
            }
        }
        *reinterpret_cast<float4*>(M + r * 32 + 8 * cg) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4*>(M + r * 32 + 8 * cg + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    __syncthreads();
    {   // stage 3: M[r][c], c < 16, += sum_u A_L1[r][u] T_10[u][c]  (two outputs a thread)
        const int r = tid >> 3, c = 2 * (tid & 7);
        const float* ar = A + (32 + r) * kAP + 16;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
            const float4 a4 = *reinterpret_cast<const float4*>(ar + 4 * u4);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 t2 = *reinterpret_cast<const float2*>(Tf + (16 + 4 * u4 + e) * kAP + c);
                a0 = fmaf(av[e], t2.x, a0);
                a1 = fmaf(av[e], t2.y, a1);
            }
        }
        float2* m2 = reinterpret_cast<float2*>(M + r * 32 + c);
        const float2 mv = *m2;
        *m2 = make_float2(mv.x + a0, mv.y + a1);
    }
    __syncthreads();
    {   // stage 4: T_LL = -T_11(32) M
        const int cc = tid & 31, r0 = tid >> 5;       // rows r0, r0 + 8, r0 + 16, r0 + 24
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        // T_11 is lower triangular: row r0 + 8m needs the column groups u / 4 <=
        // (r0 + 8m) / 4 = 2m + (r0 >> 2) only; r0 is the warp index, so the bound
        // is the same for the whole warp, and the skipped terms are exact zeros
        const int extra = r0 >> 2;
#pragma unroll
        for (int ug = 0; ug < 8; ++ug) {
            if (ug > 6 + extra) break;
            const int u = 4 * ug;
            const float s0 = scr[u * 32 + cc], s1 = scr[(u + 1) * 32 + cc];
            const float s2 = scr[(u + 2) * 32 + cc], s3 = scr[(u + 3) * 32 + cc];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (ug > 2 * m + extra) continue;
                const float4 t4 = *reinterpret_cast<const float4*>(Tf + (32 + r0 + 8 * m) * kAP + 32 + u);
                acc[m] = fmaf(t4.x, s0, acc[m]);
                acc[m] = fmaf(t4.y, s1, acc[m]);
                acc[m] = fmaf(t4.z, s2, acc[m]);
                acc[m] = fmaf(t4.w, s3, acc[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            Tf[(32 + r0 + 8 * m) * kAP + cc] = -acc[m];
            put_tp(32 + r0 + 8 * m, cc, -acc[m]);
        }
        // T' complete for the tensor core (async proxy); TMEM reads of this
        // item ordered before the MMA issued after the barrier
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }
}

// Tokens n .. 63 of both rounds' staged tiles become alpha = 1, q = k = 0 (a
// partial chunk; kept out of line, off the path of whole chunks).
__device__ __noinline__ void mask_tail_tokens(uint8_t* sm, int n, int tid) {
    const int rows = kC - n;
    for (int idx = tid; idx < 2 * rows * 64; idx += kThreads) {
        const int g = idx / (rows * 64), rem = idx - g * rows * 64;
        const int e = (n + (rem >> 6)) * 64 + (rem & 63);
        uint8_t* R = sm + g * kRound;
        reinterpret_cast<float*>(R + kRal)[e] = 1.f;
        reinterpret_cast<uint16_t*>(R + kRq)[e] = 0;
        reinterpret_cast<uint16_t*>(R + kRk)[e] = 0;
    }
}

struct Item {
    int64_t g;     // global chunk
    int h;         // head
    int seq;
    int64_t t0;    // first packed token of the chunk
    int n;         // tokens in the chunk
};

// An item's chunk-table entry (one 16-byte load; the caller issues it early).
__device__ __forceinline__ int4 item_info(const ChunkLaunch& p, int64_t item, int64_t n_items) {
    return item < n_items ? p.chunk_info[item / p.a.n_heads] : make_int4(0, 0, 0, 0);
}

__device__ __forceinline__ Item decode_item(const ChunkLaunch& p, int64_t item, int4 info) {
    Item it;
    const int H = p.a.n_heads;
    it.g = item / H;
    it.h = (int)(item % H);
    it.t0 = info.x;
    it.n = info.y;
    it.seq = info.z;
    return it;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
chunk_local_kernel(const __grid_constant__ ChunkLaunch p, const __grid_constant__ LocalMaps tm) {
    griddep_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc& ms = *reinterpret_cast<Misc*>(sm + kMisc);
    const uint32_t s_base = smem_u32(sm);

    const kda_prefill_args& a = p.a;
    const int H = a.n_heads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t total_chunks = p.chunk_base[a.n_seqs] < p.max_chunks ? p.chunk_base[a.n_seqs] : p.max_chunks;
    const int64_t n_items = total_chunks * H;
    const int64_t first = blockIdx.x, step = gridDim.x;
    if (first >= n_items) return;

    if (warp == 0) tmem_alloc(&ms.tslot, kTmemCols);
    if (tid == 0) {
        mbar_init(&ms.bar_load, 1);
        mbar_init(&ms.bar_v, 1);
        mbar_init(&ms.bar_mma, 1);
        ms.guard_fail = 0;
        ms.ld_issued = ms.ld_waited = ms.v_issued = ms.v_waited = ms.mma_issued = ms.mma_waited = 0;
        fence_mbar_init();
    }
    // each issuing thread counts the copies it starts, to drain on a timeout:
    // an item's q, k and alpha, then, once the staging above them has been read,
    // its v on a barrier of its own (the gate products start without it)
    auto issue_load_qka = [&](int64_t item, int4 info) {
        const Item it = decode_item(p, item, info);
        mbar_expect_tx(&ms.bar_load, kLoadBytes);
        const int32_t x = it.h * kD, y = (int32_t)it.t0;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            uint8_t* R = sm + g * kRound;
            tma_load_2d(R + kRq, &tm.q, x + 64 * g, y, &ms.bar_load);
            tma_load_2d(R + kRk, &tm.k, x + 64 * g, y, &ms.bar_load);
            tma_load_2d(R + kRal, &tm.alpha, x + 64 * g, y, &ms.bar_load);
        }
        ms.ld_issued += 1;
    };
    auto issue_load_v = [&](int64_t item, int4 info) {
        const Item it = decode_item(p, item, info);
        const int32_t x = it.h * kD, y = (int32_t)it.t0;
        mbar_expect_tx(&ms.bar_v, kVBytes);
#pragma unroll
        for (int g = 0; g < 2; ++g) tma_load_2d(sm + kSv + g * kVbox, &tm.v, x + 64 * g, y, &ms.bar_v);
        ms.v_issued += 1;
    };
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = ms.tslot;
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm.q)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm.k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm.v)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm.alpha)) : "memory");
    }
    if (tid == 0) {
        const int4 info0 = item_info(p, first, n_items);
        ms.info[0] = info0;
        issue_load_qka(first, info0);
        issue_load_v(first, info0);
    }
    __syncthreads();
    if (tid < kC) {
        const Item it0 = decode_item(p, first, ms.info[0]);
        ms.beta[0][tid] = tid < it0.n ? a.beta[(it0.t0 + tid) * H + it0.h] : 0.f;
    }

    const int cl = tid & 63;       // channel within a round
    const int qq = tid >> 6;       // which 16-token quarter of the chunk this thread walks
    const int hh = qq >> 1;        // its half
    const int sub = qq & 1;        // 0: local tokens 0..15 of the half, 1: 16..31
    const uint32_t lanebase = (uint32_t)(32 * (warp & 3)) << 16;
    bool ok = true;
    int k = 0;
    for (int64_t item = first; item < n_items; item += step, ++k) {
        const int nb = (k + 1) & 1;             // the next item's buffers
        const Item it = decode_item(p, item, ms.info[k & 1]);
        const int n = it.n;
        uint8_t* rec = p.records + ((size_t)it.g * H + it.h) * kRecBytes;
        const float* bsm = ms.beta[k & 1];
        // the next item's chunk-table entry (thread 0; read after later barriers)
        if (tid == 0) ms.info[nb] = item_info(p, item + step, n_items);

        // thread 0 alone polls the mbarrier; the others wait at the CTA barrier,
        // which takes no issue slots from the co-resident CTA
        if (tid == 0) {
            ok = mbar_wait(&ms.bar_load, (uint32_t)(k & 1));
            if (ok) ms.ld_waited += 1;
        } else if (tid == kStoreThread && k > 0) {
            // the previous item's W and U~ staging lies where this item's v and
            // X^T go: once the bulk stores (this thread's) have read it, v may land
            // there; the wait runs beside thread 0's wait for q, k and alpha
            bulk_wait_read();
            issue_load_v(item, ms.info[k & 1]);
        }
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }

        if (n < kC) {
            // a partial chunk: its missing tokens become alpha = 1, q = k = 0 in
            // the staged tiles, so the gate products need no token masks
            mask_tail_tokens(sm, n, tid);
            __syncthreads();
        }

        // ------------------------------------------------------------ phase 1: gates, operands
        // Decay factors of channel c for the quarter's tokens, with m the 16th
        // token of the half: Gamma (chunk prefix), kappa (chunk suffix),
        // phi = exp(g_r - g_m) and psi = 1/phi (sub 1 walks up from m, sub 0
        // down to it), xi = exp(g_47 - g_s) for half 0.
        bool guard_bad = false;
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
            const int c = 64 * g + cl;
            const uint8_t* R = sm + g * kRound;
            const uint32_t Rs = s_base + g * kRound;
            const float* sal = reinterpret_cast<const float*>(R + kRal);
            const uint16_t* sq = reinterpret_cast<const uint16_t*>(R + kRq);
            const uint16_t* sk = reinterpret_cast<const uint16_t*>(R + kRk);
            const int r_base = 16 * qq;
            float al[16];
            uint32_t qp[8], kp[8];
            float own = 1.f;
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const int r = r_base + i;
                al[i] = sal[r * 64 + cl];
                al[i + 1] = sal[(r + 1) * 64 + cl];
                qp[i >> 1] = (uint32_t)sq[r * 64 + cl] | ((uint32_t)sq[(r + 1) * 64 + cl] << 16);
                kp[i >> 1] = (uint32_t)sk[r * 64 + cl] | ((uint32_t)sk[(r + 1) * 64 + cl] << 16);
                own *= al[i];
                own *= al[i + 1];
            }
            ms.qprod[g][qq][cl] = own;
            // every thread holds its inputs: region g now takes the operand slices
            __syncthreads();
            const float Q0 = ms.qprod[g][0][cl], Q1 = ms.qprod[g][1][cl];
            const float Q2 = ms.qprod[g][2][cl], Q3 = ms.qprod[g][3][cl];
            const float before = qq == 0 ? 1.f : qq == 1 ? Q0 : qq == 2 ? Q0 * Q1 : (Q0 * Q1) * Q2;
            const float after = qq == 3 ? 1.f : qq == 2 ? Q3 : qq == 1 ? Q2 * Q3 : Q1 * (Q2 * Q3);
            const float xi_rest = qq == 0 ? Q1 * Q2 : Q2;      // tokens after the quarter, up to 47
            if (qq == 0) reinterpret_cast<float*>(rec + kRecG)[c] = (Q0 * Q1) * (Q2 * Q3);
            const uint32_t apa = Rs + kRa, apb = Rs + kRb;
            // Each factor is formed in fp32 and rounded to bf16 once; a pair of
            // tokens (2j, 2j+1) of one channel is scaled by one packed multiply.
            {   // forward: Gamma -> Q~ (record), X^T = Gamma k
                float G = before;
                uint32_t gq[2][4], xk[4];
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float G0 = G * al[i];
                    G = G0 * al[i + 1];
                    const uint32_t f = pack_bf16(G0, G);
                    gq[i >> 3][(i & 7) >> 1] = mul_bf16x2(qp[i >> 1], f);
                    xk[(i & 7) >> 1] = mul_bf16x2(kp[i >> 1], f);
                    if ((i & 7) == 6) {
                        const uint32_t r0 = r_base + (i & ~7);
                        sts16(s_base + kX + row64_chunk_off(c, r0 >> 3), make_uint4(xk[0], xk[1], xk[2], xk[3]));
                    }
                }
                stg_row_pair(rec + kRecQ, c, qq, gq[0], gq[1]);
            }
            if (sub) {   // up from the half's reference token: phi = E, psi = 1/E
                float E = 1.f;
                uint32_t dq[4], dk[4], dd[4];
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float E0 = E * al[i];
                    E = E0 * al[i + 1];
                    guard_bad |= !(E >= kGuardMin);      // alphas lie in [0, 1]: E <= E0
                    const uint32_t fe = pack_bf16(E0, E);
                    const uint32_t fi = pack_bf16(__fdividef(1.f, E0), __fdividef(1.f, E));
                    dq[(i & 7) >> 1] = mul_bf16x2(qp[i >> 1], fe);
                    dk[(i & 7) >> 1] = mul_bf16x2(kp[i >> 1], fe);
                    dd[(i & 7) >> 1] = mul_bf16x2(kp[i >> 1], fi);
                    if ((i & 7) == 6) {
                        const uint32_t r0 = r_base + (i & ~7);
                        sts16(apb + mn_chunk(r0, cl), make_uint4(dq[0], dq[1], dq[2], dq[3]));
                        sts16(apb + mn_chunk(64 + r0, cl), make_uint4(dk[0], dk[1], dk[2], dk[3]));
                        sts16(apa + mn_chunk(r0, cl), make_uint4(dd[0], dd[1], dd[2], dd[3]));
                    }
                }
            }
            {   // backward: kappa -> Kbar (record); half 0 also xi
                float Qa = after, Qx = xi_rest;     // the suffix product times the factor beyond the quarter
                uint32_t kb[2][4], kx[4];
#pragma unroll
                for (int i = 14; i >= 0; i -= 2) {
                    const float a1 = Qa, x1 = Qx;   // token i + 1
                    Qa *= al[i + 1];
                    kb[i >> 3][(i & 7) >> 1] = mul_bf16x2(kp[i >> 1], pack_bf16(Qa, a1));
                    if (!hh) {
                        Qx *= al[i + 1];
                        kx[(i & 7) >> 1] = mul_bf16x2(kp[i >> 1], pack_bf16(Qx, x1));
                        Qx *= al[i];
                    }
                    Qa *= al[i];
                    if ((i & 7) == 0 && !hh) sts16(apa + mn_chunk(64 + r_base + i, cl), make_uint4(kx[0], kx[1], kx[2], kx[3]));
                }
                stg_row_pair(rec + kRecK, c, qq, kb[0], kb[1]);
            }
            if (!sub) {  // down to the half's reference token: phi = 1/D, psi = D
                float D = 1.f;
                uint32_t dq[4], dk[4], dd[4];
#pragma unroll
                for (int i = 14; i >= 0; i -= 2) {
                    const float D1 = D;             // token i + 1
                    D *= al[i + 1];                 // token i
                    guard_bad |= !(D >= kGuardMin); // alphas lie in [0, 1]: D <= D1
                    const uint32_t fi = pack_bf16(__fdividef(1.f, D), __fdividef(1.f, D1));
                    const uint32_t fd = pack_bf16(D, D1);
                    dq[(i & 7) >> 1] = mul_bf16x2(qp[i >> 1], fi);
                    dk[(i & 7) >> 1] = mul_bf16x2(kp[i >> 1], fi);
                    dd[(i & 7) >> 1] = mul_bf16x2(kp[i >> 1], fd);
                    if ((i & 7) == 0) {
                        const uint32_t r0 = r_base + i;
                        sts16(apb + mn_chunk(r0, cl), make_uint4(dq[0], dq[1], dq[2], dq[3]));
                        sts16(apb + mn_chunk(64 + r0, cl), make_uint4(dk[0], dk[1], dk[2], dk[3]));
                        sts16(apa + mn_chunk(r0, cl), make_uint4(dd[0], dd[1], dd[2], dd[3]));
                    }
                    D *= al[i];
                }
            }
        }
        if (guard_bad) atomicOr(&ms.guard_fail, 1);
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        if (tid == 0) {
            if (ms.guard_fail) {
                // factors outside the operand range: chunk_exact_kernel rewrites
                // this item's P, W and U~ from exact products of alphas
                const uint32_t idx = atomicAdd(p.exact_count, 1u);
                if (idx < (uint64_t)n_items) p.exact_items[idx] = item;
                ms.guard_fail = 0;
            }
            const uint32_t idesc = idesc_bf16(128, 128, true, true);
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const uint32_t R = s_base + (ks >> 2) * kRound + (ks & 3) * 2 * kSbo;
                mma_bf16(tbase, sdesc(R + kRa, kLbo, kSbo), sdesc(R + kRb, kLbo, kSbo), idesc, ks > 0 ? 1u : 0u);
            }
            mma_commit(&ms.bar_mma);
            ms.mma_issued += 1;
        }
        if (tid == 0) {
            ok = mbar_wait(&ms.bar_mma, 0);
            if (ok) ms.mma_waited += 1;
        }
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        fence_after_sync();

        // ------------------------------------------------------------ phase 2: P to the record, A to smem
        // A to shared memory: warps w and w + 4 share TMEM lane quarter w (16 columns
        // each); warps 3 and 7 hold no lanes with data and write A's zero block
        {
            float* Am = reinterpret_cast<float*>(sm + kAmat);
            const int wq = warp & 3, hf = warp >> 2;
            if (wq < 3) {
                const int s = wq == 2 ? lane : lane + 32 * wq;
                const int col0 = (wq == 0 ? 64 : 96) + 16 * hf;     // columns 64 + r
                uint32_t v[16];
                tmem_ld16(tbase + lanebase + col0, v);
                tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int r4 = col0 - 64 + 4 * e4;
                    const float4 b4 = *reinterpret_cast<const float4*>(bsm + r4);
                    const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = r4 + e;
                        Am[r * kAP + s] = (wq == 2 || r > s) ? bb[e] * __uint_as_float(v[4 * e4 + e]) : 0.f;
                    }
                }
            } else {                      // rows 16 hf .. 16 hf + 15, columns 32..63 (above the diagonal)
                const int s = lane + 32;
#pragma unroll 8
                for (int r = 16 * hf; r < 16 * hf + 16; ++r) Am[r * kAP + s] = 0.f;
            }
        }
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        // the next item's beta: loaded now, stored after phase 4, so the global
        // load's latency passes while T is inverted
        float beta_nx = 0.f;
        if (tid < kC && item + step < n_items) {
            const Item nx = decode_item(p, item + step, ms.info[nb]);
            if (tid < nx.n) beta_nx = a.beta[(nx.t0 + tid) * H + nx.h];
        }
        // ------------------------------------------------------------ phase 3: T
        // P leaves TMEM while the diagonal blocks of T are solved: warps 4-6 hold
        // TMEM lane quarters 0-2, warp 7 writes P's zero block
        auto p_to_staging = [&]() {
            const int wq = warp & 3;
            if (wq < 3) {
                const int s = wq == 2 ? lane : lane + 32 * wq;      // key token of this TMEM lane
                const int col0 = wq == 0 ? 0 : 32;
                uint32_t v[2][16];
                tmem_ld16(tbase + lanebase + col0, v[0]);
                tmem_ld16(tbase + lanebase + col0 + 16, v[1]);
                tmem_wait_ld();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                    for (int e8 = 0; e8 < 2; ++e8) {
                        const int r0 = col0 + 16 * hf + 8 * e8;
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            x[e] = (wq == 2 || r0 + e >= s) ? __uint_as_float(v[hf][8 * e8 + e]) : 0.f;
                        sts16(s_base + kPst + row64_chunk_off(s, r0 >> 3), pack8(x));
                    }
                }
            } else {                      // rows 32..63, columns 0..31 (keys after the query)
                const int s = lane + 32;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) sts16(s_base + kPst + row64_chunk_off(s, cc), make_uint4(0u, 0u, 0u, 0u));
            }
            fence_async_smem();
        };
        auto store_p = [&]() {
            bulk_s2g(rec + kRecP, sm + kPst, 8192);
            bulk_commit();
        };
        // T and, beside it, T'^T (row s = beta_s times column s of T), the MN-major
        // [s][r] operand of the W / U~ product
        invert_unit_lower(reinterpret_cast<const float*>(sm + kAmat), reinterpret_cast<float*>(sm + kTf),
                          reinterpret_cast<float*>(sm + kTscr), tid, p_to_staging, store_p, s_base + kTm, bsm);
        // [0, 64 KiB) is free once the staged P has been read (A and T are consumed,
        // T' lies above it): the next item's q, k and alpha load while this item's
        // W / U~ product runs
        if (tid == kLoadThread && item + step < n_items) {
            bulk_wait_read();
            issue_load_qka(item + step, ms.info[nb]);
        }

        if (tid == 0) {
            ok = mbar_wait(&ms.bar_v, (uint32_t)(k & 1));
            if (ok) ms.v_waited += 1;
        }
        if (tid == 0 && ok) {
            // W^T = X^T T'^T (X^T K-major); U~^T = V^T T'^T with V^T the swizzled
            // v tile read MN-major (64-channel blocks 8 KiB apart, 8-token groups 1 KiB apart)
            const uint32_t idesc_k = idesc_bf16(128, 64, false, true);
            const uint32_t idesc_mn = idesc_bf16(128, 64, true, true);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tbase, sdesc(s_base + kX + ks * 32, 16, 1024), sdesc(s_base + kTm + ks * 2048, 1024, 1024),
                         idesc_k, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_bf16(tbase + 64, sdesc(s_base + kSv + ks * 2048, kVbox, 1024),
                         sdesc(s_base + kTm + ks * 2048, 1024, 1024), idesc_mn, ks > 0 ? 1u : 0u);
            mma_commit(&ms.bar_mma);
            ms.mma_issued += 1;
        }
        if (tid == 0 && ok) {
            ok = mbar_wait(&ms.bar_mma, 1);
            if (ok) ms.mma_waited += 1;
        }
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        fence_after_sync();

        // ------------------------------------------------------------ phase 4: W and U~ to the record
        {
            const int row = 32 * (warp & 3) + lane;
            const uint32_t col0 = warp < 4 ? 0u : 64u;
            const uint32_t dst = s_base + kWst + (warp < 4 ? 0u : 16384u);
            uint32_t v[4][16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_ld16(tbase + lanebase + col0 + 16 * q4, v[q4]);
            tmem_wait_ld();
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(v[e8 >> 1][8 * (e8 & 1) + e]);
                sts16(dst + row64_chunk_off(row, e8), pack8(x));
            }
        }
        if (tid < kC) ms.beta[nb][tid] = beta_nx;
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (tid == kStoreThread) {
            bulk_s2g(rec + kRecW, sm + kWst, 16384);
            bulk_s2g(rec + kRecU, sm + kWst + 16384, 16384);
            bulk_commit();
        }
    }

    if (tid == kStoreThread || tid == kLoadThread) bulk_wait_all();   // staged records written out
    if (!ok && tid == 0) {
        // let this CTA's own copies and MMAs in flight land (bounded) before
        // shared and tensor memory are released
        flag(p.status, KDA_DEV_WAIT_TIMEOUT);
        for (uint32_t l = ms.ld_waited; l < ms.ld_issued; ++l) mbar_wait(&ms.bar_load, l & 1);
        for (uint32_t l = ms.v_waited; l < ms.v_issued; ++l) mbar_wait(&ms.bar_v, l & 1);
        for (uint32_t m = ms.mma_waited; m < ms.mma_issued; ++m) mbar_wait(&ms.bar_mma, m & 1);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// ---------------------------------------------------------------- exact items
// Items whose decay factors left the MMA form's operand range get their P, W
// and U~ tiles rewritten here, in fp32 from exact products of alphas
// (chunk_decay.cuh): A and P by pairs, T = (I + A)^-1 by forward substitution,
// W = T diag(beta) (Gamma * K) and U~ = T diag(beta) V, stored in the record's
// bf16 layout.  Their Q~, Kbar and gamma involve no reference factor and stand
// as chunk_local_kernel wrote them.
constexpr int kExactThreads = 256;

struct ExactSmem {
    float A[64][65];
    float T[64][65];
    DecayBlock D;
    float V[64][kDecayLd];
    float beta[64];
};

__device__ __forceinline__ void st_bf16(uint8_t* p, float x) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(x);
}

__global__ void __launch_bounds__(kExactThreads) chunk_exact_kernel(ChunkLaunch p) {
    griddep_wait();
    extern __shared__ __align__(16) uint8_t exact_smem[];
    ExactSmem& sm = *reinterpret_cast<ExactSmem*>(exact_smem);
    const kda_prefill_args& a = p.a;
    const int H = a.n_heads;
    const int tid = threadIdx.x;
    const int64_t total_chunks = p.chunk_base[a.n_seqs] < p.max_chunks ? p.chunk_base[a.n_seqs] : p.max_chunks;
    const int64_t n_items = total_chunks * H;
    const uint32_t listed = *p.exact_count;
    const int64_t count = (int64_t)listed < n_items ? (int64_t)listed : n_items;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v);
    DecayBlock& D = sm.D;
    const int r = tid >> 2, cs = tid & 3;
    for (int64_t i = blockIdx.x; i < count; i += gridDim.x) {
        const int64_t item = p.exact_items[i];
        if (item < 0 || item >= n_items) continue;
        const int64_t g = item / H;
        const int h = (int)(item % H);
        const int4 info = p.chunk_info[g];
        const int64_t t0 = info.x;
        const int n = info.y;
        uint8_t* rec = p.records + (size_t)item * kRecBytes;
        __syncthreads();
        if (tid < 64) sm.beta[tid] = tid < n ? a.beta[(t0 + tid) * H + h] : 0.f;
        float accA[16], accP[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) accA[m] = accP[m] = 0.f;
        auto load_block = [&](int cb, bool with_q) {
            __syncthreads();
            for (int e = tid; e < 64 * kDecayCB; e += kExactThreads) {
                const int t = e / kDecayCB, c = e % kDecayCB;
                const bool in = t < n;
                const size_t off = ((size_t)(t0 + t) * H + h) * kD + cb + c;
                D.k[t][c] = in ? __bfloat162float(k[off]) : 0.f;
                D.q[t][c] = in && with_q ? __bfloat162float(q[off]) : 0.f;
                D.al[t][c] = in ? a.alpha[off] : 1.f;
                if (!with_q) sm.V[t][c] = in ? __bfloat162float(v[off]) : 0.f;
            }
            __syncthreads();
            decay_tables(D, tid, kExactThreads);
            __syncthreads();
        };
        for (int cb = 0; cb < kD; cb += kDecayCB) {
            load_block(cb, true);
            accumulate_ap(D, r, cs, accA, accP);
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int s = cs + 4 * m;
            sm.A[r][s] = s < r ? sm.beta[r] * accA[m] : 0.f;
            // P tile: row s (key token), column r
            st_bf16(rec + kRecP + row64_chunk_off(s, r >> 3) + (r & 7) * 2, s <= r ? accP[m] : 0.f);
        }
        __syncthreads();
        if (tid < 64) {                       // T = (I + A)^-1, column j per thread
            const int j = tid;
            for (int x = 0; x < j; ++x) sm.T[x][j] = 0.f;
            sm.T[j][j] = 1.f;
            for (int x = j + 1; x < 64; ++x) {
                float acc = 0.f;
                for (int s = j; s < x; ++s) acc = fmaf(sm.A[x][s], sm.T[s][j], acc);
                sm.T[x][j] = -acc;
            }
        }
        __syncthreads();
        for (int e = tid; e < 64 * 64; e += kExactThreads) sm.T[e >> 6][e & 63] *= sm.beta[e & 63];
        // W_tc = sum_s T'_ts Gamma_sc k_sc and U~_tj = sum_s T'_ts v_sj, 16 channels at a time
        for (int cb = 0; cb < kD; cb += kDecayCB) {
            load_block(cb, false);
            for (int e = tid; e < 64 * kDecayCB; e += kExactThreads) {   // X = Gamma * K over k
                const int t = e / kDecayCB, c = e % kDecayCB;
                D.q[t][c] = prefix_decay(D, t, c) * D.k[t][c];
            }
            __syncthreads();
            for (int e = tid; e < 64 * kDecayCB; e += kExactThreads) {
                const int t = e % 64, c = e / 64;
                float w = 0.f, u = 0.f;
                for (int s = 0; s <= t; ++s) {
                    const float tt = sm.T[t][s];
                    w = fmaf(tt, D.q[s][c], w);
                    u = fmaf(tt, sm.V[s][c], u);
                }
                const uint32_t off = row64_chunk_off(cb + c, t >> 3) + (t & 7) * 2;
                st_bf16(rec + kRecW + off, w);
                st_bf16(rec + kRecU + off, u);
            }
        }
    }
}

// ---------------------------------------------------------------- meta: chunk table
// chunk_base[s] = first global chunk of sequence s (exclusive scan of
// ceil(L_s / 64) over valid sequences).
__global__ void __launch_bounds__(1024) chunk_meta_kernel(ChunkLaunch p) {
    griddep_wait();
    const kda_prefill_args& a = p.a;
    const int n = a.n_seqs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ int64_t warp_tot[32];
    __shared__ int64_t carry;
    if (tid == 0) {
        carry = 0;
        *p.exact_count = 0;
    }
    __syncthreads();
    for (int base = 0; base < n; base += 1024) {
        const int s = base + tid;
        int64_t nc = 0;
        if (s < n) {
            int64_t tb, te, pos0;
            int32_t init;
            uint32_t bad;
            if (seq_valid(a, s, &tb, &te, &pos0, &init, &bad)) nc = (te - tb + kC - 1) / kC;
            else flag(p.status, bad);
        }
        int64_t x = nc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int64_t w = warp_tot[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            warp_tot[lane] = w;   // inclusive over warps
        }
        __syncthreads();
        const int64_t incl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x;
        if (s < n) p.chunk_base[s] = (int32_t)(incl - nc);
        __syncthreads();
        if (tid == 0) carry += warp_tot[31];
        __syncthreads();
    }
    if (tid == 0) {
        if (carry > p.max_chunks) {        // only reachable with overlapping sequences
            flag(p.status, KDA_DEV_BAD_SEQLENS);
            carry = 0;
        }
    }
    __syncthreads();
    if (carry == 0)
        for (int s = tid; s < n; s += blockDim.x) p.chunk_base[s] = 0;
    if (tid == 0) p.chunk_base[n] = (int32_t)carry;
    __syncthreads();
    // per-chunk table: first packed token, token count, sequence
    for (int64_t g = tid; g < carry; g += blockDim.x) {
        int lo = 0, hi = n - 1;   // last sequence whose first chunk is <= g
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.chunk_base[mid] <= g) lo = mid;
            else hi = mid - 1;
        }
        const int64_t tb = a.cu_seqlens[lo], te = a.cu_seqlens[lo + 1];
        const int64_t t0 = tb + (g - p.chunk_base[lo]) * kC;
        p.chunk_info[g] = make_int4((int32_t)t0, (int32_t)(te - t0 < kC ? te - t0 : kC), lo, 0);
    }
}

}  // namespace

cudaError_t launch_chunk_exact(const ChunkLaunch& p, cudaStream_t s) {
    const int64_t max_items = p.max_chunks * p.a.n_heads;
    if (max_items == 0 || p.a.total_tokens == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(ExactSmem);
    e = cudaFuncSetAttribute(chunk_exact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = max_items < 2 * (int64_t)sms ? max_items : 2 * (int64_t)sms;
    note_launch();
    return launch_overlapped(chunk_exact_kernel, dim3((unsigned)grid), dim3(kExactThreads), smem, s, p);
}

cudaError_t launch_chunk_meta(const ChunkLaunch& p, cudaStream_t s) {
    note_launch();
    return launch_overlapped(chunk_meta_kernel, dim3(1), dim3(1024), 0, s, p);
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once; the initialisation of a
// function-local static is thread-safe, so concurrent first calls all see it.
EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(f);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// [rows x cols] row-major tensor, boxes of 64 rows x box_cols elements, with or
// without the 128-byte swizzle; rows past the end read as zero.  Every box here
// starts at a column that is a multiple of 64, a multiple of 16 bytes.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* base, int64_t rows,
              int64_t cols, uint32_t box_cols, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)kC};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_local(const ChunkLaunch& p, cudaStream_t s) {
    const int64_t max_items = p.max_chunks * p.a.n_heads;
    if (max_items == 0 || p.a.total_tokens == 0) return cudaSuccess;
    LocalMaps tm;
    const int64_t rows = p.a.total_tokens, cols = (int64_t)p.a.n_heads * kD;
    const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE, sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_map(&tm.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.a.q, rows, cols, 64, none) ||
        !make_map(&tm.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.a.k, rows, cols, 64, none) ||
        !make_map(&tm.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.a.v, rows, cols, 64, sw128) ||
        !make_map(&tm.alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.a.alpha, rows, cols, 64, none))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chunk_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chunk_local_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    const int64_t slots = (int64_t)kCtasPerSm * sms;
    const int64_t grid = max_items < slots ? max_items : slots;
    note_launch();
    return launch_overlapped(chunk_local_kernel, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, s, p, tm);
}

}  // namespace kda
