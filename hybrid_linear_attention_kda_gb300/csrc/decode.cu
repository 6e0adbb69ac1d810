// Batched single-token KDA decode: one in-place read-modify-write of each fp32
// state ("Kimi K3 Tech Intro", section 4.1: the fused decode kernel updates the
// recurrent state in place).
//
// Per (sequence, head) and per value column j, with S the state before the step:
//     a_j = sum_i (alpha_i k_i) S_ij        (= (S'^T k)_j,  S' = Diag(alpha) S)
//     b_j = sum_i (alpha_i q_i) S_ij        (= (S'^T q)_j)
//     u_j = beta (v_j - a_j)
//     S_ij <- alpha_i S_ij + k_i u_j         (= S' + k u^T)
//     o_j = scale (b_j + u_j (q . k))        (= scale (S^T q)_j after the update)
// so the state is read once and written once.  The kernel is bound by HBM: each
// CTA owns a TJ-column tile of one head's state, reads it with coalesced 16-byte
// loads (a warp instruction covers whole rows of the tile), keeps it in
// registers, reduces a_j and b_j over the d_k rows with warp shuffles plus one
// shared-memory step across warps, and writes the tile back with 16-byte stores.
#include "kda_common.cuh"

namespace kda {
namespace {

template <typename T, int D, int TJ, int NT>
__global__ void __launch_bounds__(NT) decode_kernel(DecodeLaunch p) {
    constexpr int LPR = TJ / 4;          // lanes per state row (one float4 each)
    constexpr int RPW = 32 / LPR;        // rows covered by one warp instruction
    constexpr int NW = NT / 32;
    constexpr int RPT = D / (NW * RPW);  // rows held by each thread
    constexpr int NTILE = D / TJ;
    static_assert(LPR * RPW == 32 && RPT * NW * RPW == D, "tile shape");

    __shared__ float s_a[D], s_ka[D], s_qa[D], s_k[D], s_q[D];
    __shared__ float s_red_a[NW][TJ], s_red_b[NW][TJ];
    __shared__ __align__(16) float s_u[TJ];
    __shared__ float s_qk;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = blockIdx.x % NTILE;
    const int64_t sh = blockIdx.x / NTILE;  // seq * H + head
    const int seq = (int)(sh / p.H);
    const int j0 = tile * TJ;

    const int32_t slot = p.slot[seq];
    if (slot < 0 || (int64_t)slot >= p.n_slots) {
        if (tid == 0) flag(p.status, KDA_DEV_BAD_SLOT);
        return;
    }
    const int64_t head = (int64_t)slot * p.H + (sh - (int64_t)seq * p.H);
    float* S = p.pool + head * D * D;

    // issue the state loads first: RPT independent 16-byte loads per thread
    const int cq = lane % LPR;
    const int rbase = warp * (RPT * RPW) + lane / LPR;
    float4 st[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = rbase + m * RPW;
        st[m] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)i * D + j0 + 4 * cq));
    }

    // stage this token's q, k, alpha
    const int64_t vec = sh * D;
    for (int i = tid; i < D; i += NT) {
        const float a = p.alpha[vec + i];
        const float ki = Elem<T>::load(static_cast<const T*>(p.k) + vec + i);
        const float qi = Elem<T>::load(static_cast<const T*>(p.q) + vec + i);
        s_a[i] = a;
        s_ka[i] = a * ki;
        s_qa[i] = a * qi;
        s_k[i] = ki;
        s_q[i] = qi;
    }
    __syncthreads();
    if (warp == 0) {
        float acc = 0.f;
        for (int i = lane; i < D; i += 32) acc = fmaf(s_q[i], s_k[i], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) s_qk = acc;
    }

    // partial a_j, b_j over this thread's rows, then over the warp's row groups
    float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = rbase + m * RPW;
        const float ka = s_ka[i], qa = s_qa[i];
        pa[0] = fmaf(ka, st[m].x, pa[0]);
        pa[1] = fmaf(ka, st[m].y, pa[1]);
        pa[2] = fmaf(ka, st[m].z, pa[2]);
        pa[3] = fmaf(ka, st[m].w, pa[3]);
        pb[0] = fmaf(qa, st[m].x, pb[0]);
        pb[1] = fmaf(qa, st[m].y, pb[1]);
        pb[2] = fmaf(qa, st[m].z, pb[2]);
        pb[3] = fmaf(qa, st[m].w, pb[3]);
    }
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            pa[c] += __shfl_xor_sync(0xffffffffu, pa[c], off);
            pb[c] += __shfl_xor_sync(0xffffffffu, pb[c], off);
        }
    }
    if (lane < LPR) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            s_red_a[warp][4 * cq + c] = pa[c];
            s_red_b[warp][4 * cq + c] = pb[c];
        }
    }
    __syncthreads();

    if (tid < TJ) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            a += s_red_a[w][tid];
            b += s_red_b[w][tid];
        }
        const int j = j0 + tid;
        const float vj = Elem<T>::load(static_cast<const T*>(p.v) + vec + j);
        const float u = p.beta[sh] * (vj - a);
        s_u[tid] = u;
        Elem<T>::store(static_cast<T*>(p.o) + vec + j, p.scale * fmaf(u, s_qk, b));
    }
    __syncthreads();

    const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * cq]);
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = rbase + m * RPW;
        const float ai = s_a[i], ki = s_k[i];
        float4 r;
        r.x = fmaf(ai, st[m].x, ki * u4.x);
        r.y = fmaf(ai, st[m].y, ki * u4.y);
        r.z = fmaf(ai, st[m].z, ki * u4.z);
        r.w = fmaf(ai, st[m].w, ki * u4.w);
        __stcs(reinterpret_cast<float4*>(S + (int64_t)i * D + j0 + 4 * cq), r);
    }
}

template <typename T, int D, int TJ, int NT>
cudaError_t launch_t(const DecodeLaunch& p, cudaStream_t s) {
    const int64_t blocks = (int64_t)p.n_seqs * p.H * (D / TJ);
    note_launch();
    decode_kernel<T, D, TJ, NT><<<(unsigned)blocks, NT, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& p, cudaStream_t s) {
    if (p.D == 128)
        return p.dtype == KDA_BF16 ? launch_t<__nv_bfloat16, 128, 128, 256>(p, s)
                                   : launch_t<float, 128, 128, 256>(p, s);
    return p.dtype == KDA_BF16 ? launch_t<__nv_bfloat16, 64, 64, 128>(p, s)
                               : launch_t<float, 64, 64, 128>(p, s);
}

}  // namespace kda
