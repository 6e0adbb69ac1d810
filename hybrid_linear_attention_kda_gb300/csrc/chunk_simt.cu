// The chunked prefill in fp32 SIMT arithmetic, for the inputs the tensor-core
// kernels do not take: fp32 q/k/v (whose 1e-4 accuracy bf16 operands cannot
// reach) and d_k = d_v = 64.  It is the same algorithm as the tensor-core pair
// (the block-matrix form of the yunthe.com "Kimi K3 open-source practice" page,
// FlashKDA paragraph) on the same chunk table: a chunk-local kernel writes one
// record per (chunk, head), a carry kernel takes the fp32 state of each
// (sequence, head) through its chunks, with snapshots every 256 absolute
// positions ("Kimi K3 Tech Intro", sections 2.2-2.4) and resume.
//
// For a chunk of n <= 64 tokens r entering with state S (d x d), with the
// decay factor f_rsc = prod_{s < tau <= r} alpha_tau,c (chunk_decay.cuh) and
// Gamma_r = prod_{tau <= r} alpha_tau per channel:
//   A_rs = beta_r sum_c k_rc k_sc f_rsc   (s < r),   P_rs = sum_c q_rc k_sc f_rsc   (s <= r)
//   T = (I + A)^-1,  T' = T diag(beta)
//   W = T' (Gamma * K),  U~ = T' V,  Q~ = Gamma * Q,
//   Kbar_s = (prod_{tau > s} alpha_tau) k_s,  gamma = Gamma_{n-1}
// the carry is  U = U~ - W S,  O = Q~ S + P U,  S <- Diag(gamma) S + Kbar^T U.
// Every factor is a product of alphas, so nothing overflows and an underflow is
// the true (negligible) value.
//
// Record of one (chunk, head), fp32, token-major rows:
//   W [64][D], Q~ [64][D], Kbar [64][D], U~ [64][D], P [64][64], gamma [D]
#include "async_copy.cuh"
#include "chunk_common.cuh"
#include "chunk_decay.cuh"

namespace kda {

size_t simt_record_bytes(int d) { return (size_t)(4 * 64 * d + 64 * 64 + d) * sizeof(float); }

namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtCols = 16;        // value columns per carry CTA
constexpr int kCB = kDecayCB;            // channels per block in the chunk-local passes
constexpr int kLd = kDecayLd;

template <int D>
struct SimtRec {
    static constexpr size_t W = 0, Q = 64 * D, K = 2 * 64 * D, U = 3 * 64 * D, P = 4 * 64 * D;
    static constexpr size_t G = 4 * 64 * D + 64 * 64;
    static constexpr size_t floats = G + D;
};

// Shared memory of the chunk-local kernel (dynamic).
struct LocalSmem {
    float A[64][65];          // A (strictly lower, beta_r scaled)
    float T[64][65];          // T, then T' = T diag(beta)
    union {
        DecayBlock p1;        // pass 1: one block of channels
        struct {              // pass 2
            float X[64][kLd], V[64][kLd];
        } p2;
    } u;
    float beta[64];
};

// The A and P sums of one block of channels, taken by key token: the thread
// holds the pairs (r, s) with r = rs + 4 m, m = 0..15, of key s, and adds the
// block's channels to them in channel order, as accumulate_ap does for its
// pairs.  The factor of a pair is the one pair_decay forms: within s's 16-token
// group G the left-to-right product alpha_{s+1} ... alpha_r, here the running
// product as r walks up the group (one multiply per token, no per-pair chain);
// from a later group, pout_s pin_r times the whole groups between.  G is uniform
// in a warp, so every accumulator index is known at compile time.
template <int G>
__device__ __forceinline__ void accumulate_ap_key_group(const DecayBlock& D, int s, int rs, float (&accA)[16],
                                                        float (&accP)[16]) {
    const int us = s & 15;
#pragma unroll 1
    for (int c = 0; c < kDecayCB; ++c) {
        const float ks = D.k[s][c];
        float f = 1.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int r = 16 * G + u;
            if (u > us) f *= D.al[r][c];
            if (u >= us && (u & 3) == rs) {
                const float e = f * ks;
                accP[4 * G + (u >> 2)] = fmaf(D.q[r][c], e, accP[4 * G + (u >> 2)]);
                accA[4 * G + (u >> 2)] = fmaf(D.k[r][c], e, accA[4 * G + (u >> 2)]);
            }
        }
#pragma unroll
        for (int m = 4 * (G + 1); m < 16; ++m) {
            const int r = rs + 4 * m;
            float fx = D.pout[s][c] * D.pin[r][c];
#pragma unroll
            for (int b = G + 1; b < (m >> 2); ++b) fx *= D.btot[b][c];
            const float e = fx * ks;
            accP[m] = fmaf(D.q[r][c], e, accP[m]);
            accA[m] = fmaf(D.k[r][c], e, accA[m]);
        }
    }
}
__device__ __forceinline__ void accumulate_ap_by_key(const DecayBlock& D, int s, int rs, float (&accA)[16],
                                                     float (&accP)[16]) {
    switch (s >> 4) {
        case 0: accumulate_ap_key_group<0>(D, s, rs, accA, accP); break;
        case 1: accumulate_ap_key_group<1>(D, s, rs, accA, accP); break;
        case 2: accumulate_ap_key_group<2>(D, s, rs, accA, accP); break;
        default: accumulate_ap_key_group<3>(D, s, rs, accA, accP); break;
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads) simt_local_kernel(ChunkLaunch p) {
    griddep_wait();
    using R = SimtRec<D>;
    extern __shared__ __align__(16) uint8_t simt_smem[];
    LocalSmem& sm = *reinterpret_cast<LocalSmem*>(simt_smem);
    const kda_prefill_args& a = p.a;
    const int H = a.n_heads;
    const int tid = threadIdx.x;
    const int64_t total_chunks = p.chunk_base[a.n_seqs] < p.max_chunks ? p.chunk_base[a.n_seqs] : p.max_chunks;
    const int64_t item = blockIdx.x;
    if (item >= total_chunks * H) return;
    const int64_t g = item / H;
    const int h = (int)(item % H);
    const int4 info = p.chunk_info[g];
    const int64_t t0 = info.x;
    const int n = info.y;
    float* rec = reinterpret_cast<float*>(p.records) + (size_t)item * R::floats;

    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    if (tid < 64) sm.beta[tid] = tid < n ? a.beta[(t0 + tid) * H + h] : 0.f;

    // this thread's 16 (r, s) pairs: key s, rows r = rs + 4 m
    const int s = tid >> 2, rs = tid & 3;
    float accA[16], accP[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) accA[m] = accP[m] = 0.f;

    // ---------------------------------------------------------------- pass 1
    DecayBlock& D1 = sm.u.p1;
    for (int cb = 0; cb < D; cb += kCB) {
        __syncthreads();
        for (int e = tid; e < 64 * kCB; e += kSimtThreads) {
            const int t = e / kCB, c = e % kCB;
            const bool in = t < n;
            const size_t off = ((size_t)(t0 + t) * H + h) * D + cb + c;
            D1.k[t][c] = in ? Elem<T>::load(k + off) : 0.f;
            D1.q[t][c] = in ? Elem<T>::load(q + off) : 0.f;
            D1.al[t][c] = in ? a.alpha[off] : 1.f;
        }
        __syncthreads();
        decay_tables(D1, tid, kSimtThreads);
        __syncthreads();
        // Q~, Kbar, gamma and (for the second pass) X = Gamma * K into the record
        for (int e = tid; e < 64 * kCB; e += kSimtThreads) {
            const int t = e / kCB, c = e % kCB;
            const float G = prefix_decay(D1, t, c);
            rec[R::Q + t * D + cb + c] = G * D1.q[t][c];
            rec[R::K + t * D + cb + c] = suffix_decay(D1, t, c) * D1.k[t][c];
            rec[R::W + t * D + cb + c] = G * D1.k[t][c];
            if (t == 63) rec[R::G + cb + c] = G;
        }
        accumulate_ap_by_key(D1, s, rs, accA, accP);
    }
    // A (strictly lower, beta_r scaled) to shared memory; P to the record
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int r = rs + 4 * m;
        sm.A[r][s] = s < r ? sm.beta[r] * accA[m] : 0.f;
        rec[R::P + r * 64 + s] = s <= r ? accP[m] : 0.f;
    }
    __syncthreads();
    // T = (I + A)^-1 by forward substitution, one column j per thread
    if (tid < 64) {
        const int j = tid;
        for (int i = 0; i < j; ++i) sm.T[i][j] = 0.f;
        sm.T[j][j] = 1.f;
        for (int i = j + 1; i < 64; ++i) {
            float acc = 0.f;
#pragma unroll 8
            for (int s = j; s < i; ++s) acc = fmaf(sm.A[i][s], sm.T[s][j], acc);
            sm.T[i][j] = -acc;
        }
    }
    __syncthreads();
    for (int e = tid; e < 64 * 64; e += kSimtThreads) sm.T[e >> 6][e & 63] *= sm.beta[e & 63];

    // ---------------------------------------------------------------- pass 2
    // W = T' X and U~ = T' V, one block of channels at a time; the block of X
    // is read from the record's W rows before W overwrites them
    const int orow = tid >> 2, oc = (tid & 3) * 4;      // 4 outputs of one row per thread
    for (int cb = 0; cb < D; cb += kCB) {
        __syncthreads();
        for (int e = tid; e < 64 * kCB; e += kSimtThreads) {
            const int t = e / kCB, c = e % kCB;
            sm.u.p2.X[t][c] = rec[R::W + t * D + cb + c];
            sm.u.p2.V[t][c] = t < n ? Elem<T>::load(v + ((size_t)(t0 + t) * H + h) * D + cb + c) : 0.f;
        }
        __syncthreads();
        float w4[4] = {0.f, 0.f, 0.f, 0.f}, u4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int s = 0; s <= orow; ++s) {
            const float t = sm.T[orow][s];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w4[i] = fmaf(t, sm.u.p2.X[s][oc + i], w4[i]);
                u4[i] = fmaf(t, sm.u.p2.V[s][oc + i], u4[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            rec[R::W + orow * D + cb + oc + i] = w4[i];
            rec[R::U + orow * D + cb + oc + i] = u4[i];
        }
    }
}

// The carry of one (sequence, head): the fp32 state S [D][D] in shared memory.
template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads) simt_recur_kernel(ChunkLaunch p) {
    griddep_wait();
    using R = SimtRec<D>;
    // Every column of S evolves on its own (U, O and the update of column j read
    // only column j of S and U), so a chain is split over D / kSimtCols CTAs, one
    // block of value columns each; the arithmetic of every element is unchanged.
    constexpr int JB = kSimtCols;
    constexpr int G = kSimtThreads / JB;     // thread groups over the second index
    extern __shared__ __align__(16) uint8_t simt_smem[];
    float* S = reinterpret_cast<float*>(simt_smem);          // [D][JB]
    float* U = S + D * JB;                                   // [64][JB]
    // the chunk's record, staged: W, Q~, Kbar [64][D] each and P [64][64],
    // gamma [D] in the record's order, then this CTA's columns of U~ [64][JB]
    float* sW = U + 64 * JB;
    float* sQ = sW + 64 * D;
    float* sK = sQ + 64 * D;
    float* sP = sK + 64 * D;
    float* sG = sP + 64 * 64;
    float* sU = sG + D;
    const kda_prefill_args& a = p.a;
    const int H = a.n_heads;
    const int tid = threadIdx.x;
    const int64_t chain = blockIdx.x / (D / JB);
    const int jb = (int)(blockIdx.x % (D / JB)) * JB;
    const int seq = (int)(chain / H), h = (int)(chain % H);
    int64_t tb, te, pos0;
    int32_t init;
    uint32_t bad;
    if (!seq_valid(a, seq, &tb, &te, &pos0, &init, &bad)) return;     // flagged by the meta kernel
    const int64_t g0 = p.chunk_base[seq];
    const int64_t nc = p.chunk_base[seq + 1] - g0;
    if (nc < 0 || g0 + nc > p.max_chunks) return;
    const int64_t slot_stride = (int64_t)H * D * D;
    const int64_t head_off = (int64_t)h * D * D;
    const int jl = tid % JB, grp = tid / JB, j = jb + jl;   // this thread's value column

    const float* S0 = init >= 0 ? a.pool + (int64_t)init * slot_stride + head_off : nullptr;
    for (int e = tid; e < D * JB; e += kSimtThreads) S[e] = S0 ? S0[(e / JB) * D + jb + e % JB] : 0.f;
    T* o = static_cast<T*>(a.o);

    for (int64_t lc = 0; lc < nc; ++lc) {
        const int64_t t0 = tb + lc * kC;
        const int n = (int)(te - t0 < kC ? te - t0 : kC);
        const float* rec = reinterpret_cast<const float*>(p.records) + (size_t)((g0 + lc) * H + h) * R::floats;
        __syncthreads();                                         // S complete, staging free
        // the record into shared memory by 16-byte asynchronous copies (records
        // and their rows are 16-byte aligned): W, Q~ and Kbar are one range of the
        // record, P and gamma another
        for (int e = tid; e < 3 * 64 * D / 4; e += kSimtThreads) cp_async16(sW + 4 * e, rec + R::W + 4 * e);
        for (int e = tid; e < (64 * 64 + D) / 4; e += kSimtThreads) cp_async16(sP + 4 * e, rec + R::P + 4 * e);
        for (int e = tid; e < 64 * JB / 4; e += kSimtThreads) {
            const int t = e / (JB / 4), i = 4 * (e % (JB / 4));
            cp_async16(sU + t * JB + i, rec + R::U + t * D + jb + i);
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();
        // U = U~ - W S (rows read as 16-byte pieces; the sums keep their order)
        for (int t = grp; t < n; t += G) {
            const float4* w = reinterpret_cast<const float4*>(sW + t * D);
            float acc = sU[t * JB + jl];
#pragma unroll
            for (int c4 = 0; c4 < D / 4; ++c4) {
                const float4 w4 = w[c4];
                const float* sc = S + 4 * c4 * JB + jl;
                acc = fmaf(-w4.x, sc[0], acc);
                acc = fmaf(-w4.y, sc[JB], acc);
                acc = fmaf(-w4.z, sc[2 * JB], acc);
                acc = fmaf(-w4.w, sc[3 * JB], acc);
            }
            U[t * JB + jl] = acc;
        }
        __syncthreads();
        // O = Q~ S + P U
        for (int t = grp; t < n; t += G) {
            const float4* qt = reinterpret_cast<const float4*>(sQ + t * D);
            const float* pt = sP + t * 64;
            float acc = 0.f;
#pragma unroll
            for (int c4 = 0; c4 < D / 4; ++c4) {
                const float4 q4 = qt[c4];
                const float* sc = S + 4 * c4 * JB + jl;
                acc = fmaf(q4.x, sc[0], acc);
                acc = fmaf(q4.y, sc[JB], acc);
                acc = fmaf(q4.z, sc[2 * JB], acc);
                acc = fmaf(q4.w, sc[3 * JB], acc);
            }
            const int full = (t + 1) & ~3;              // P row entries s < full in 16-byte pieces
            for (int s = 0; s < full; s += 4) {
                const float4 p4 = *reinterpret_cast<const float4*>(pt + s);
                const float* us = U + s * JB + jl;
                acc = fmaf(p4.x, us[0], acc);
                acc = fmaf(p4.y, us[JB], acc);
                acc = fmaf(p4.z, us[2 * JB], acc);
                acc = fmaf(p4.w, us[3 * JB], acc);
            }
            for (int s = full; s <= t; ++s) acc = fmaf(pt[s], U[s * JB + jl], acc);
            Elem<T>::store(o + ((t0 + t) * H + h) * D + j, a.scale * acc);
        }
        __syncthreads();                                         // every read of S done
        // S <- Diag(gamma) S + Kbar^T U
        for (int c = grp; c < D; c += G) {
            float acc = sG[c] * S[c * JB + jl];
            for (int t = 0; t < n; ++t) acc = fmaf(sK[t * D + c], U[t * JB + jl], acc);
            S[c * JB + jl] = acc;
        }
        // a snapshot after this chunk
        const int64_t p_end = pos0 + lc * kC + n;
        if (a.snap_table && p_end % a.snap_interval == 0) {
            const int64_t ord = p_end / a.snap_interval - 1;
            int32_t slot = -1;
            if (ord >= a.snap_table_stride) {
                if (tid == 0 && jb == 0) flag(p.status, KDA_DEV_BAD_ORDINAL);
            } else {
                slot = a.snap_table[(int64_t)seq * a.snap_table_stride + ord];
                if (slot != -1 && (slot < 0 || (int64_t)slot >= a.n_slots)) {
                    if (tid == 0 && jb == 0) flag(p.status, KDA_DEV_BAD_SLOT);
                    slot = -1;
                }
            }
            if (slot >= 0) {
                __syncthreads();
                float* dst = a.pool + (int64_t)slot * slot_stride + head_off;
                for (int e = tid; e < D * JB; e += kSimtThreads) dst[(e / JB) * D + jb + e % JB] = S[e];
            }
        }
    }
    __syncthreads();
    if (a.final_state) {
        float* dst = a.final_state + (int64_t)seq * slot_stride + head_off;
        for (int e = tid; e < D * JB; e += kSimtThreads) dst[(e / JB) * D + jb + e % JB] = S[e];
    }
}

template <typename T, int D>
cudaError_t launch_simt_pair(const ChunkLaunch& p, cudaStream_t s, bool local) {
    if (local) {
        const int64_t items = p.max_chunks * p.a.n_heads;
        if (items == 0 || p.a.total_tokens == 0) return cudaSuccess;
        const size_t smem = sizeof(LocalSmem);
        cudaError_t e = cudaFuncSetAttribute(simt_local_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        note_launch();
        return launch_overlapped(simt_local_kernel<T, D>, dim3((unsigned)items), dim3(kSimtThreads), smem, s, p);
    }
    const int64_t chains = (int64_t)p.a.n_seqs * p.a.n_heads;
    if (chains == 0) return cudaSuccess;
    const size_t smem = (size_t)(D * kSimtCols + 64 * kSimtCols + 3 * 64 * D + 64 * 64 + D + 64 * kSimtCols) *
                        sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(simt_recur_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    note_launch();
    return launch_overlapped(simt_recur_kernel<T, D>, dim3((unsigned)(chains * (D / kSimtCols))), dim3(kSimtThreads),
                             smem, s, p);
}

cudaError_t launch_simt(const ChunkLaunch& p, cudaStream_t s, bool local) {
    const bool f32 = p.a.dtype == KDA_FP32;
    if (p.a.d_k == 64) return f32 ? launch_simt_pair<float, 64>(p, s, local) : launch_simt_pair<__nv_bfloat16, 64>(p, s, local);
    return f32 ? launch_simt_pair<float, 128>(p, s, local) : launch_simt_pair<__nv_bfloat16, 128>(p, s, local);
}

}  // namespace

cudaError_t launch_simt_local(const ChunkLaunch& p, cudaStream_t s) { return launch_simt(p, s, true); }
cudaError_t launch_simt_recur(const ChunkLaunch& p, cudaStream_t s) { return launch_simt(p, s, false); }

}  // namespace kda
