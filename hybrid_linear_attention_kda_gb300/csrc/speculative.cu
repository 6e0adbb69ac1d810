// Speculative decoding for KDA ("Kimi K3 Tech Intro", section 6): a draft model
// proposes several tokens per sequence and the target model checks them all in
// one step, keeps the accepted prefix and falls back on the rest.  A recurrent
// state cannot be rolled back, so the step is split in two:
//
//   verify  reads each state once and runs the T candidate tokens through it in
//           registers, writing for every token t its output
//               o_t = scale S_t^T q_t
//           and its update vector
//               u_t = beta_t (v_t - (Diag(alpha_t) S_{t-1})^T k_t),
//           but never the state;
//   commit  reads each state once more, applies the updates of the accepted
//           tokens only,
//               S <- Diag(alpha_t) S + k_t u_t^T      for t < n_accept,
//           and writes it back (no reduction is needed: u_t is known).
//
// Both keep the single-token decode kernel's per-thread data (one CTA per
// (sequence, head), the whole state in registers, 16-byte coalesced access) and
// its arithmetic in the same order, so verify(1) followed by commit(1) gives the
// decode step's results bit for bit.  Verify groups its threads so that the sums
// over the state rows stay inside warps: its token loop has no CTA barrier.  All candidate tokens' inputs are staged in
// shared memory next to the state load, so the token loop waits on no global
// load.
#include "async_copy.cuh"
#include "kda_common.cuh"

namespace kda {
namespace {

template <int D, int NT>
struct Tile {
    static constexpr int TJ = D;              // columns per CTA: the whole head
    static constexpr int LPR = TJ / 4;        // lanes per state row (one float4 each)
    static constexpr int RPW = 32 / LPR;      // rows covered by one warp instruction
    static constexpr int NW = NT / 32;
    static constexpr int RPT = D / (NW * RPW);   // rows held by each thread
    static_assert(LPR * RPW == 32 && RPT * NW * RPW == D, "tile shape");
};

// Shared memory of one verify CTA, per candidate token: alpha, k, alpha k and
// alpha q in a padded row layout (four spare floats after every 16 rows, so the
// eight row groups of a warp read distinct banks), q and v unpadded, beta and
// q.k.
template <int D>
__host__ __device__ constexpr int verify_row_stride() { return D + D / 4; }
template <int D>
__host__ __device__ constexpr size_t verify_smem(int T) {
    return (size_t)T * (4 * verify_row_stride<D>() + 2 * D + 2) * sizeof(float);
}
__device__ __forceinline__ int vpad(int i) { return i + (i >> 4) * 4; }

// The verify CTA keeps the decode kernel's per-thread data: the same state rows
// and four columns, summed by the same fmaf chains.  It groups the threads
// differently: warp W holds columns 16W .. 16W+15, and its lane l takes column
// quad 4W + (l & 3) of decode's row group g = l >> 2 (decode's warp g / RPW,
// sub-row g % RPW).  The sum over the eight row groups of a column then runs
// inside one warp, through warp-private shared memory and in decode's order,
// and the token loop needs no CTA barrier.
template <typename T, int D, int NT>
__global__ void __launch_bounds__(NT) verify_kernel(SpecLaunch p) {
    using L = Tile<D, NT>;
    constexpr int RPW = L::RPW, RPT = L::RPT, NW = L::NW;
    constexpr int NG = 8;                       // row groups per column quad
    constexpr int DP = verify_row_stride<D>();
    constexpr int RED = 2 * NG * 16 + 16;       // one warp's a and b partials, b offset by 144 floats
    static_assert(NT / (D / 4) == NG, "eight row groups per column quad");
    static_assert(RPT % 4 == 0, "rows per group in float4 pieces");
    extern __shared__ __align__(16) float dyn[];
    const int nT = p.T;
    float* s_a = dyn;                  // [T][DP]
    float* s_k = s_a + nT * DP;
    float* s_ka = s_k + nT * DP;
    float* s_qa = s_ka + nT * DP;
    float* s_q = s_qa + nT * DP;       // [T][D]
    float* s_v = s_q + nT * D;
    float* s_beta = s_v + nT * D;      // [T]
    float* s_qk = s_beta + nT;         // [T]
    __shared__ __align__(16) float s_red[NW][RED];
    __shared__ __align__(16) float s_uw[NW][16];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t sh = blockIdx.x;           // seq * H + head
    const int seq = (int)(sh / p.H);
    const int h = (int)(sh - (int64_t)seq * p.H);
    const int32_t slot = p.slot[seq];
    if (slot < 0 || (int64_t)slot >= p.n_slots) {
        if (tid == 0) flag(p.status, KDA_DEV_BAD_SLOT);
        return;
    }
    const float* S = p.pool + ((int64_t)slot * p.H + h) * D * D;
    const int quad = lane & 3;               // column quad within the warp
    const int g = lane >> 2;                 // decode's row group
    const int c0 = 16 * warp + 4 * quad;     // first of this lane's four columns
    const int rfirst = (g / RPW) * (RPT * RPW) + g % RPW;
    float4 st[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m)
        st[m] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(rfirst + m * RPW) * D + c0));

    // every candidate token's inputs ([n_seqs, T, H, D] rows) first: they are
    // small and return before the state
    for (int e = tid; e < nT * D; e += NT) {
        const int t = e / D, i = e - t * D;
        const int64_t vec = (((int64_t)seq * nT + t) * p.H + h) * D;
        const float a = p.alpha[vec + i];
        const float ki = Elem<T>::load(static_cast<const T*>(p.k) + vec + i);
        const float qi = Elem<T>::load(static_cast<const T*>(p.q) + vec + i);
        const int ip = t * DP + vpad(i);
        s_a[ip] = a;
        s_k[ip] = ki;
        s_ka[ip] = a * ki;
        s_qa[ip] = a * qi;
        s_q[e] = qi;
        s_v[e] = Elem<T>::load(static_cast<const T*>(p.v) + vec + i);
    }
    for (int t = tid; t < nT; t += NT) s_beta[t] = p.beta[((int64_t)seq * nT + t) * p.H + h];
    __syncthreads();
    for (int t = warp; t < nT; t += NW) {   // q . k of every token, one warp each
        float acc = 0.f;
        for (int i = lane; i < D; i += 32) acc = fmaf(s_q[t * D + i], s_k[t * DP + vpad(i)], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) s_qk[t] = acc;
    }
    __syncthreads();

    float* red = s_red[warp];
    const int col = lane & 15, which = lane >> 4;   // the output this lane finishes
    for (int t = 0; t < nT; ++t) {
        const int tb = t * DP;
        float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int ip = tb + vpad(rfirst + m * RPW);
            const float ka = s_ka[ip], qa = s_qa[ip];
            pa[0] = fmaf(ka, st[m].x, pa[0]);
            pa[1] = fmaf(ka, st[m].y, pa[1]);
            pa[2] = fmaf(ka, st[m].z, pa[2]);
            pa[3] = fmaf(ka, st[m].w, pa[3]);
            pb[0] = fmaf(qa, st[m].x, pb[0]);
            pb[1] = fmaf(qa, st[m].y, pb[1]);
            pb[2] = fmaf(qa, st[m].z, pb[2]);
            pb[3] = fmaf(qa, st[m].w, pb[3]);
        }
        *reinterpret_cast<float4*>(red + g * 16 + 4 * quad) = make_float4(pa[0], pa[1], pa[2], pa[3]);
        *reinterpret_cast<float4*>(red + 144 + g * 16 + 4 * quad) = make_float4(pb[0], pb[1], pb[2], pb[3]);
        __syncwarp();
        // decode's order: each decode warp's sub-rows combined first, then the
        // warps summed in order from zero
        float acc = 0.f;
        const float* rw = red + 144 * which + col;
#pragma unroll
        for (int w = 0; w < NG / RPW; ++w) {
            float comb = rw[(w * RPW) * 16];
            if (RPW == 2) comb = comb + rw[(w * RPW + 1) * 16];
            acc += comb;
        }
        const int j = 16 * warp + col;
        const int64_t vec = (((int64_t)seq * nT + t) * p.H + h) * D;
        if (which == 0) {
            const float u = s_beta[t] * (s_v[t * D + j] - acc);
            s_uw[warp][col] = u;
            p.u[vec + j] = u;
        }
        __syncwarp();
        if (which == 1) Elem<T>::store(static_cast<T*>(p.o) + vec + j, p.scale * fmaf(s_uw[warp][col], s_qk[t], acc));
        const float4 u4 = *reinterpret_cast<const float4*>(&s_uw[warp][4 * quad]);
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int ip = tb + vpad(rfirst + m * RPW);
            const float ai = s_a[ip], ki = s_k[ip];
            st[m].x = fmaf(ai, st[m].x, ki * u4.x);
            st[m].y = fmaf(ai, st[m].y, ki * u4.y);
            st[m].z = fmaf(ai, st[m].z, ki * u4.z);
            st[m].w = fmaf(ai, st[m].w, ki * u4.w);
        }
        __syncwarp();        // the next token's partials and u may overwrite this token's
    }
}

// Shared memory of one commit CTA: alpha and u ([T][D] fp32) and k ([T][D] in
// its element type, within a [T][D] fp32-sized slot) of the accepted tokens.
template <int D>
__host__ __device__ constexpr size_t commit_smem(int T) {
    return (size_t)T * 3 * D * sizeof(float);
}


template <typename T, int D, int NT>
__global__ void __launch_bounds__(NT) commit_kernel(SpecLaunch p) {
    using L = Tile<D, NT>;
    constexpr int LPR = L::LPR, RPW = L::RPW, RPT = L::RPT;
    extern __shared__ __align__(16) float dyn[];
    const int nT = p.T;
    float* s_a = dyn;
    T* s_k = reinterpret_cast<T*>(s_a + nT * D);
    float* s_u = s_a + 2 * nT * D;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t sh = blockIdx.x;
    const int seq = (int)(sh / p.H);
    const int h = (int)(sh - (int64_t)seq * p.H);
    const int32_t slot = p.slot[seq];
    if (slot < 0 || (int64_t)slot >= p.n_slots) {
        if (tid == 0) flag(p.status, KDA_DEV_BAD_SLOT);
        return;
    }
    const int32_t m_acc = p.n_accept[seq];
    if (m_acc < 0 || m_acc > nT) {
        if (tid == 0) flag(p.status, KDA_DEV_BAD_ACCEPT);
        return;
    }
    if (m_acc == 0) return;                  // nothing accepted: the state stays as it is
    float* S = p.pool + ((int64_t)slot * p.H + h) * D * D;
    const int cq = lane % LPR;
    const int rbase = warp * (RPT * RPW) + lane / LPR;
    // the accepted tokens' alpha, u and k ([n_seqs, T, H, D] rows, 16-byte
    // aligned) by asynchronous copies, then the state
    constexpr int F4 = D / 4;                          // 16-byte pieces of an fp32 row
    constexpr int KP = D * (int)sizeof(T) / 16;        // 16-byte pieces of a k row
    for (int e = tid; e < m_acc * F4; e += NT) {
        const int t = e / F4, i = 4 * (e - t * F4);
        const int64_t vec = (((int64_t)seq * nT + t) * p.H + h) * D;
        cp_async16(s_a + t * D + i, p.alpha + vec + i);
        cp_async16(s_u + t * D + i, p.u + vec + i);
    }
    for (int e = tid; e < m_acc * KP; e += NT) {
        const int t = e / KP, i = e - t * KP;
        const int64_t vec = (((int64_t)seq * nT + t) * p.H + h) * D;
        cp_async16(reinterpret_cast<uint8_t*>(s_k + t * D) + 16 * i,
                   reinterpret_cast<const uint8_t*>(static_cast<const T*>(p.k) + vec) + 16 * i);
    }
    cp_async_commit();
    float4 st[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m)
        st[m] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(rbase + m * RPW) * D + 4 * cq));
    cp_async_wait_all();
    __syncthreads();
    for (int t = 0; t < m_acc; ++t) {
        const float4 u4 = *reinterpret_cast<const float4*>(&s_u[t * D + 4 * cq]);
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = rbase + m * RPW;
            const float ai = s_a[t * D + i], ki = Elem<T>::load(s_k + t * D + i);
            st[m].x = fmaf(ai, st[m].x, ki * u4.x);
            st[m].y = fmaf(ai, st[m].y, ki * u4.y);
            st[m].z = fmaf(ai, st[m].z, ki * u4.z);
            st[m].w = fmaf(ai, st[m].w, ki * u4.w);
        }
    }
#pragma unroll
    for (int m = 0; m < RPT; ++m)
        __stcs(reinterpret_cast<float4*>(S + (int64_t)(rbase + m * RPW) * D + 4 * cq), st[m]);
}

template <typename T, int D, int NT>
struct VerifyK {
    static cudaError_t run(const SpecLaunch& p, cudaStream_t s) {
        const size_t smem = verify_smem<D>(p.T);
        cudaError_t e = cudaFuncSetAttribute(verify_kernel<T, D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        note_launch();
        verify_kernel<T, D, NT><<<(unsigned)((int64_t)p.n_seqs * p.H), NT, smem, s>>>(p);
        return cudaGetLastError();
    }
};
template <typename T, int D, int NT>
struct CommitK {
    static cudaError_t run(const SpecLaunch& p, cudaStream_t s) {
        note_launch();
        commit_kernel<T, D, NT><<<(unsigned)((int64_t)p.n_seqs * p.H), NT, commit_smem<D>(p.T), s>>>(p);
        return cudaGetLastError();
    }
};

template <template <typename, int, int> class K>
cudaError_t dispatch(const SpecLaunch& p, cudaStream_t s) {
    if (p.D == 128)
        return p.dtype == KDA_BF16 ? K<__nv_bfloat16, 128, 256>::run(p, s) : K<float, 128, 256>::run(p, s);
    return p.dtype == KDA_BF16 ? K<__nv_bfloat16, 64, 128>::run(p, s) : K<float, 64, 128>::run(p, s);
}

}  // namespace

cudaError_t launch_verify(const SpecLaunch& p, cudaStream_t s) { return dispatch<VerifyK>(p, s); }
cudaError_t launch_commit(const SpecLaunch& p, cudaStream_t s) { return dispatch<CommitK>(p, s); }

}  // namespace kda
