// Stage one of the chunked prefill: everything of a 64-token chunk that does not
// depend on the carried state, for all (chunk, head) pairs in parallel.
//
// Decay factors are products of alphas over token ranges (no exp / log): with
// the chunk split into halves of 32 tokens,
//   Gamma_r    = prod_{tau <= r} alpha            (chunk prefix, <= 1)
//   kappa_r    = prod_{tau > r} alpha             (chunk suffix, <= 1)
//   rho_r      = prod_{32 <= tau <= r} alpha      (r in half 1: exp(g_r - g_31))
//   sigma_s    = prod_{s < tau <= 31} alpha       (s in half 0: exp(g_31 - g_s))
//   phi_r      = exp(g_r - g_m) with m the 16th token of r's half, psi = 1/phi.
// The intra-chunk products A and P come from one tcgen05 MMA whose rows are the
// key tokens s and whose columns are query / key tokens r:
//   rows 0..63   k_s psi_s        x  cols 0..63   q_r phi_r    -> P, same half
//   rows 64..95  k_s sigma_s         cols 64..95  q_r rho_r    -> P, r in half 1, s in half 0
//                                    cols 96..159 k_r phi_r    -> A, same half
//                                    cols 160..191 k_r rho_r   -> A, r in half 1, s in half 0
// Within a half the factors phi, psi span at most 16 tokens; a chunk whose
// factors leave [2^-100, 2^100] flags its (sequence, head) for the token-serial
// kernel.  T = (I + A)^-1 is inverted by 16 x 16 blocks in fp32, then W and U~ come
// from a second MMA (X^T T^T and Y^T T^T with X = diag(beta) Gamma K,
// Y = diag(beta) V).
#include "chunk_common.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int kThreads = 256;
// shared memory (1024-aligned base)
constexpr uint32_t kAPa = 0;            // A/P MMA operand A: MN-major [c][128 rows s]
constexpr uint32_t kAPb = 32768;        // A/P MMA operand B: MN-major [c][192 cols]
constexpr uint32_t kLboA = 1024, kSboA = 2048, kLboB = 1024, kSboB = 3072;
constexpr uint32_t kAmat = 0;           // after the A/P MMA: A fp32 [64][64]
constexpr uint32_t kTm = 16384;         //   T as MN-major [s][r] bf16
constexpr uint32_t kXt = 24576;         //   X^T K-major [c][s]
constexpr uint32_t kYt = 40960;         //   Y^T K-major [j][s]
constexpr uint32_t kTf = 57344;         //   T fp32 [64][64]
constexpr uint32_t kTscr = 73728;       //   block-product scratch, 3 x 16 x 16 fp32
constexpr uint32_t kMisc = 81920;
constexpr size_t kSmemBytes = kMisc + 2048 + 1024;

struct Misc {
    float beta[kC];
    float tot[2][kD];
    uint64_t bar;
    uint32_t tslot;
    int32_t guard_fail;
};
static_assert(sizeof(Misc) <= 2048, "misc");

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    return make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                      pack_bf16(v[6], v[7]));
}
__device__ __forceinline__ void sts16(uint32_t saddr, uint4 v) { st_shared_v4(saddr, v.x, v.y, v.z, v.w); }
__device__ __forceinline__ void stg16(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// byte offset of the 16-byte chunk (mn .. mn+7, k) in an MN-major tile
__device__ __forceinline__ uint32_t mn_chunk(uint32_t mn, uint32_t k, uint32_t lbo, uint32_t sbo) {
    return (k >> 3) * sbo + (mn >> 6) * lbo + (k & 7u) * 128u + ((((mn & 63u) >> 3) ^ (k & 7u)) << 4);
}


// T = (I + A)^-1 for a strictly lower triangular 64 x 64 A (fp32, row-major),
// by 16 x 16 blocks: the four diagonal blocks by forward substitution, then the
// off-diagonal blocks one block-diagonal at a time,
//     T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj .
// All 256 threads take part; T (including zeros above the diagonal inside the
// diagonal blocks) goes to Tf, row-major.  Ends with a barrier.
__device__ __forceinline__ void invert_unit_lower(const float* A, float* Tf, float* scr, int tid) {
    if (tid < kC) {
        const int o = 16 * (tid >> 4), jj = tid & 15;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = r == jj ? 1.f : 0.f;
#pragma unroll
            for (int u = 0; u < r; ++u) acc = fmaf(-A[(o + r) * kC + o + u], t[u], acc);
            t[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tf[(o + r) * kC + o + jj] = t[r];
    }
    __syncthreads();
#pragma unroll
    for (int dist = 1; dist < 4; ++dist) {
        const int nblk = 4 - dist;
        for (int e = tid; e < nblk * 256; e += kThreads) {       // M = sum_k A_ik T_kj
            const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
            const int i = dist + blk, jb = i - dist;
            float acc = 0.f;
            for (int kb = jb; kb < i; ++kb) {
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    acc = fmaf(A[(16 * i + rr) * kC + 16 * kb + u], Tf[(16 * kb + u) * kC + 16 * jb + cc], acc);
            }
            scr[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nblk * 256; e += kThreads) {       // T_ij = -T_ii M
            const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
            const int i = dist + blk, jb = i - dist;
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u)
                acc = fmaf(Tf[(16 * i + rr) * kC + 16 * i + u], scr[(blk << 8) + (u << 4) + cc], acc);
            Tf[(16 * i + rr) * kC + 16 * jb + cc] = -acc;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads, 2) chunk_local_kernel(ChunkLaunch p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc& ms = *reinterpret_cast<Misc*>(sm + kMisc);
    const uint32_t s_base = smem_u32(sm);

    const kda_prefill_args& a = p.a;
    const int H = a.n_heads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t g = blockIdx.x / H;
    const int h = (int)(blockIdx.x % H);
    const int n_seqs = a.n_seqs;
    const int64_t total_chunks = p.chunk_base[n_seqs];
    if (g >= total_chunks || g >= p.max_chunks) return;
    int lo = 0, hi = n_seqs - 1;   // last sequence whose first chunk is <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.chunk_base[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    const int seq = lo;
    int64_t tb, te, pos0;
    int32_t init;
    uint32_t bad;
    if (!seq_valid(a, seq, &tb, &te, &pos0, &init, &bad)) return;
    const int64_t t0 = tb + (g - p.chunk_base[seq]) * kC;
    const int n = (int)(te - t0 < kC ? te - t0 : kC);
    uint8_t* rec = p.records + ((size_t)g * H + h) * kRecBytes;
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(a.v);
    const int64_t tstride = (int64_t)H * kD;       // elements between consecutive tokens
    const int64_t ebase = (t0 * H + h) * kD;       // element (token 0 of the chunk, channel 0)

    // ---------------------------------------------------------------- phase 1: gates, operands
    if (warp == 0) tmem_alloc(&ms.tslot, 256);
    if (tid == 0) {
        ms.guard_fail = 0;
        mbar_init(&ms.bar, 1);
        fence_mbar_init();
    }
    if (tid < kC) ms.beta[tid] = tid < n ? a.beta[(t0 + tid) * H + h] : 0.f;

    const int c = tid & (kD - 1);
    const int hh = tid >> 7;       // which half of the chunk this thread walks
    float al[32];
    uint32_t qp[16], kp[16];
    {
        float prod = 1.f;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const int r = 32 * hh + i;
            const int64_t e0 = ebase + (int64_t)r * tstride + c, e1 = e0 + tstride;
            const bool v0 = r < n, v1 = r + 1 < n;
            al[i] = v0 ? a.alpha[e0] : 1.f;
            al[i + 1] = v1 ? a.alpha[e1] : 1.f;
            const uint32_t q0 = v0 ? __bfloat16_as_ushort(qg[e0]) : 0u, q1 = v1 ? __bfloat16_as_ushort(qg[e1]) : 0u;
            const uint32_t k0 = v0 ? __bfloat16_as_ushort(kg[e0]) : 0u, k1 = v1 ? __bfloat16_as_ushort(kg[e1]) : 0u;
            qp[i >> 1] = q0 | (q1 << 16);
            kp[i >> 1] = k0 | (k1 << 16);
            prod *= al[i];
            prod *= al[i + 1];
        }
        ms.tot[hh][c] = prod;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = ms.tslot;
    const float H0 = ms.tot[0][c], H1 = ms.tot[1][c];
    if (hh == 1) reinterpret_cast<float*>(rec + kRecG)[c] = H0 * H1;

    bool guard_bad = false;
    const uint32_t apa = s_base + kAPa, apb = s_base + kAPb;
    // Each walk below keeps one running product; splitting the walks keeps only
    // a few 8-token staging groups live at a time.
    {   // forward: Gamma (Q~ to the record), rho (half 1: q rho, k rho)
        float P = 1.f;
        float gq[8], oq[8], ok[8];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float qf = (i & 1) ? bf_hi(qp[i >> 1]) : bf_lo(qp[i >> 1]);
            const float kf = (i & 1) ? bf_hi(kp[i >> 1]) : bf_lo(kp[i >> 1]);
            P *= al[i];
            gq[i & 7] = qf * (hh ? H0 * P : P);
            oq[i & 7] = qf * P;
            ok[i & 7] = kf * P;
            if ((i & 7) == 7) {
                const uint32_t r0 = 32 * hh + (i & ~7);
                stg16(rec + kRecQ + row64_chunk_off(c, r0 >> 3), pack8(gq));
                if (hh) {
                    sts16(apb + mn_chunk(64 + (i & ~7), c, kLboB, kSboB), pack8(oq));
                    sts16(apb + mn_chunk(160 + (i & ~7), c, kLboB, kSboB), pack8(ok));
                }
            }
        }
    }
    {   // forward from the half's reference token: phi = E, psi = 1/E (local tokens 16..31)
        float E = 1.f;
        float dq[8], dk[8], dd[8];
#pragma unroll
        for (int i = 16; i < 32; ++i) {
            const float qf = (i & 1) ? bf_hi(qp[i >> 1]) : bf_lo(qp[i >> 1]);
            const float kf = (i & 1) ? bf_hi(kp[i >> 1]) : bf_lo(kp[i >> 1]);
            E *= al[i];
            guard_bad |= !(E >= kGuardMin);
            const float inv = __fdividef(1.f, E);
            dq[i & 7] = qf * E;
            dk[i & 7] = kf * E;
            dd[i & 7] = kf * inv;
            if ((i & 7) == 7) {
                const uint32_t r0 = 32 * hh + (i & ~7);
                sts16(apb + mn_chunk(r0, c, kLboB, kSboB), pack8(dq));
                sts16(apb + mn_chunk(96 + r0, c, kLboB, kSboB), pack8(dk));
                sts16(apa + mn_chunk(r0, c, kLboA, kSboA), pack8(dd));
            }
        }
    }
    {   // backward: kappa (Kbar to the record), sigma (half 0: k sigma); zero pad rows
        float Q = 1.f;
        float kb[8], kc[8];
#pragma unroll
        for (int i = 31; i >= 0; --i) {
            const float kf = (i & 1) ? bf_hi(kp[i >> 1]) : bf_lo(kp[i >> 1]);
            kb[i & 7] = kf * (hh ? Q : Q * H1);
            kc[i & 7] = kf * Q;
            if ((i & 7) == 0) {
                const uint32_t r0 = 32 * hh + i;
                stg16(rec + kRecK + row64_chunk_off(c, r0 >> 3), pack8(kb));
                if (!hh) sts16(apa + mn_chunk(64 + i, c, kLboA, kSboA), pack8(kc));
                else sts16(apa + mn_chunk(96 + i, c, kLboA, kSboA), make_uint4(0u, 0u, 0u, 0u));
            }
            Q *= al[i];
        }
    }
    {   // backward to the half's reference token: phi = 1/D, psi = D (local tokens 0..15)
        float Dd = 1.f;
        float dq[8], dk[8], dd[8];
#pragma unroll
        for (int i = 15; i >= 0; --i) {
            const float qf = (i & 1) ? bf_hi(qp[i >> 1]) : bf_lo(qp[i >> 1]);
            const float kf = (i & 1) ? bf_hi(kp[i >> 1]) : bf_lo(kp[i >> 1]);
            guard_bad |= !(Dd >= kGuardMin);
            const float inv = __fdividef(1.f, Dd);
            dq[i & 7] = qf * inv;
            dk[i & 7] = kf * inv;
            dd[i & 7] = kf * Dd;
            if ((i & 7) == 0) {
                const uint32_t r0 = 32 * hh + i;
                sts16(apb + mn_chunk(r0, c, kLboB, kSboB), pack8(dq));
                sts16(apb + mn_chunk(96 + r0, c, kLboB, kSboB), pack8(dk));
                sts16(apa + mn_chunk(r0, c, kLboA, kSboA), pack8(dd));
            }
            Dd *= al[i];
        }
    }
    if (guard_bad) atomicOr(&ms.guard_fail, 1);
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    if (tid == 0) {
        if (ms.guard_fail) atomicOr(&p.chain_flag[(int64_t)seq * H + h], 1);
        const uint32_t idesc = idesc_bf16(128, 192, true, true);
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            const uint64_t ad = sdesc(apa + ks * 2 * kSboA, kLboA, kSboA);
            const uint64_t bd = sdesc(apb + ks * 2 * kSboB, kLboB, kSboB);
            mma_bf16(tbase, ad, bd, idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(&ms.bar);
    }
    bool ok = mbar_wait(&ms.bar, 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) flag(p.status, KDA_DEV_WAIT_TIMEOUT);
        if (warp == 0) tmem_dealloc(tbase, 256);
        return;
    }
    fence_after_sync();

    // ---------------------------------------------------------------- phase 2: P to the record, A to smem
    const uint32_t lanebase = (uint32_t)(32 * (warp & 3)) << 16;
    if (warp < 3) {
        const int s = warp == 2 ? lane : lane + 32 * warp;      // key token of this TMEM lane
        const int col0 = 32 * warp;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t v[16];
            tmem_ld16(tbase + lanebase + col0 + 16 * hf, v);
            tmem_wait_ld();
#pragma unroll
            for (int e8 = 0; e8 < 2; ++e8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int col = col0 + 16 * hf + 8 * e8 + e;
                    const int r = warp == 2 ? 32 + (col - 64) : col;
                    const float d = __uint_as_float(v[8 * e8 + e]);
                    x[e] = (warp == 2 || r >= s) ? d : 0.f;
                }
                const int r0 = warp == 2 ? 32 + 16 * hf + 8 * e8 : col0 + 16 * hf + 8 * e8;
                stg16(rec + kRecP + row64_chunk_off(s, r0 >> 3), pack8(x));
            }
        }
        if (warp == 1) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) stg16(rec + kRecP + row64_chunk_off(s, cc), make_uint4(0u, 0u, 0u, 0u));
        }
    } else if (warp >= 4 && warp < 7) {
        const int wq = warp - 4;
        const int s = wq == 2 ? lane : lane + 32 * wq;
        const int col0 = wq == 0 ? 96 : (wq == 1 ? 128 : 160);
        const int rbase = wq == 0 ? 0 : 32;
        float* Am = reinterpret_cast<float*>(sm + kAmat);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t v[16];
            tmem_ld16(tbase + lanebase + col0 + 16 * hf, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int r = rbase + 16 * hf + e;
                const float d = __uint_as_float(v[e]);
                Am[r * kC + s] = (wq == 2 || r > s) ? ms.beta[r] * d : 0.f;
            }
        }
        if (wq == 1) {
            for (int r = 0; r < 32; ++r) Am[r * kC + s] = 0.f;
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---------------------------------------------------------------- phase 3: X^T, Y^T, T
    // X^T / Y^T rows from this thread's 32 tokens of channel c (two rounds of 16
    // tokens, to bound the loads in flight per thread), then T.
    {
        float Gm = hh ? ms.tot[0][c] : 1.f;
#pragma unroll 1
        for (int rnd = 0; rnd < 2; ++rnd) {
            float ax[16];
            uint32_t kq[8], vq[8];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const int r = 32 * hh + 16 * rnd + i;
                const int64_t e0 = ebase + (int64_t)r * tstride + c, e1 = e0 + tstride;
                const bool v0 = r < n, v1 = r + 1 < n;
                ax[i] = v0 ? a.alpha[e0] : 1.f;
                ax[i + 1] = v1 ? a.alpha[e1] : 1.f;
                kq[i >> 1] = (v0 ? (uint32_t)__bfloat16_as_ushort(kg[e0]) : 0u) |
                             ((v1 ? (uint32_t)__bfloat16_as_ushort(kg[e1]) : 0u) << 16);
                vq[i >> 1] = (v0 ? (uint32_t)__bfloat16_as_ushort(vg[e0]) : 0u) |
                             ((v1 ? (uint32_t)__bfloat16_as_ushort(vg[e1]) : 0u) << 16);
            }
            // X^T row c: beta_r Gamma_rc k_rc ;  Y^T row c: beta_r v_rc
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                float x[8], y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = 8 * c2 + e;
                    const float b = ms.beta[32 * hh + 16 * rnd + i];
                    Gm *= ax[i];
                    const float kf = (i & 1) ? bf_hi(kq[i >> 1]) : bf_lo(kq[i >> 1]);
                    const float vf = (i & 1) ? bf_hi(vq[i >> 1]) : bf_lo(vq[i >> 1]);
                    x[e] = b * kf * Gm;
                    y[e] = b * vf;
                }
                const int cc = 4 * hh + 2 * rnd + c2;
                sts16(s_base + kXt + row64_chunk_off(c, cc), pack8(x));
                sts16(s_base + kYt + row64_chunk_off(c, cc), pack8(y));
            }
        }
    }
    invert_unit_lower(reinterpret_cast<const float*>(sm + kAmat), reinterpret_cast<float*>(sm + kTf),
                      reinterpret_cast<float*>(sm + kTscr), tid);
    {
        // T^T row s (= column s of T, zero above the diagonal) as the MN-major [s][r] operand
        const float* Tf = reinterpret_cast<const float*>(sm + kTf);
        const int srow = tid >> 2;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
            const int cc = 2 * (tid & 3) + q2;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int r = 8 * cc + e;
                x[e] = r >= srow ? Tf[r * kC + srow] : 0.f;
            }
            sts16(s_base + kTm + row64_chunk_off(srow, cc), pack8(x));
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks) {
            const uint64_t bd = sdesc(s_base + kTm + ks * 2048, 1024, 1024);
            mma_bf16(tbase, sdesc(s_base + kXt + ks * 32, 16, 1024), bd, idesc, ks > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks) {
            const uint64_t bd = sdesc(s_base + kTm + ks * 2048, 1024, 1024);
            mma_bf16(tbase + 64, sdesc(s_base + kYt + ks * 32, 16, 1024), bd, idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(&ms.bar);
    }
    ok = mbar_wait(&ms.bar, 1);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) flag(p.status, KDA_DEV_WAIT_TIMEOUT);
        if (warp == 0) tmem_dealloc(tbase, 256);
        return;
    }
    fence_after_sync();

    // ---------------------------------------------------------------- phase 4: W and U~ to the record
    {
        const int row = 32 * (warp & 3) + lane;
        const uint32_t col0 = warp < 4 ? 0u : 64u;
        uint8_t* dst = rec + (warp < 4 ? kRecW : kRecU);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t v[16];
            tmem_ld16(tbase + lanebase + col0 + 16 * q4, v);
            tmem_wait_ld();
#pragma unroll
            for (int e8 = 0; e8 < 2; ++e8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(v[8 * e8 + e]);
                stg16(dst + row64_chunk_off(row, 2 * q4 + e8), pack8(x));
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

// ---------------------------------------------------------------- meta: chunk table
// chunk_base[s] = first global chunk of sequence s (exclusive scan of
// ceil(L_s / 64) over valid sequences); chain flags cleared.
__global__ void __launch_bounds__(1024) chunk_meta_kernel(ChunkLaunch p) {
    const kda_prefill_args& a = p.a;
    const int n = a.n_seqs, H = a.n_heads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ int64_t warp_tot[32];
    __shared__ int64_t carry;
    for (int64_t i = tid; i < (int64_t)n * H; i += blockDim.x) p.chain_flag[i] = 0;
    if (tid == 0) carry = 0;
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
}

}  // namespace

cudaError_t launch_chunk_meta(const ChunkLaunch& p, cudaStream_t s) {
    note_launch();
    chunk_meta_kernel<<<1, 1024, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_chunk_local(const ChunkLaunch& p, cudaStream_t s) {
    const int64_t blocks = p.max_chunks * p.a.n_heads;
    if (blocks == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(chunk_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    note_launch();
    chunk_local_kernel<<<(unsigned)blocks, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
