// One fused decode step of the KDA layer ("Kimi K3 Tech Intro", section 4.1: the
// causal convolution, the q/k norm, the gates, the recurrent update and the gated
// RMSNorm in one kernel, with the convolution state and the recurrent state
// updated in place; section 2.1: the two per-request states S and C).
//
// Per (sequence, head), from the raw projections xq, xk, xv, a, b, g of one token:
//   for x in (q, k, v):  y_x = silu(sum_tau w_x[tau] * [C_x, x][tau])   (width K = 4)
//                        C_x <- [C_x[1:], x]
//   q = y_q |y_q|^-1,  k = y_k |y_k|^-1,  v = y_v        (norms with a 1e-6 floor)
//   alpha = exp(-softplus(a)) = 1 / (1 + e^a),  beta = sigmoid(b)
//   u = beta (v - (Diag(alpha) S)^T k),  S <- Diag(alpha) S + k u^T,  o = S^T q
//   y = norm_w * o * (mean(o^2) + eps)^-1/2 * sigmoid(g)
// The update uses the tile layout and arithmetic of the single-token decode
// kernel: one CTA per (sequence, head), the fp32 state read once into registers
// and written once.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kConv = 4;
constexpr float kQkEps = 1e-6f;

__device__ __forceinline__ float bf(const void* p, int64_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}
__device__ __forceinline__ float sigmoidf(float x) { return 1.f / (1.f + expf(-x)); }

template <int D, int NT>
__global__ void __launch_bounds__(NT) fused_decode_kernel(FusedDecodeLaunch L) {
    const kda_fused_decode_args& p = L.a;
    constexpr int TJ = D;
    constexpr int LPR = TJ / 4, RPW = 32 / LPR, NW = NT / 32, RPT = D / (NW * RPW);
    static_assert(LPR * RPW == 32 && RPT * NW * RPW == D, "tile shape");
    static_assert(3 * D >= NT && TJ <= NT, "thread mapping");
    __shared__ float s_y[3][D];                // convolution outputs of q, k, v
    __shared__ float s_a[D], s_ka[D], s_qa[D], s_k[D];
    __shared__ float s_red_a[NW][TJ], s_red_b[NW][TJ];
    __shared__ __align__(16) float s_u[TJ];
    __shared__ float s_sum[3];                 // |y_q|^2, |y_k|^2, y_q . y_k
    __shared__ float s_osq[TJ / 32];           // sum of o^2 per warp

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t sh = blockIdx.x;             // seq * H + head
    const int H = p.n_heads;
    const int seq = (int)(sh / H);
    const int h = (int)(sh - (int64_t)seq * H);
    const int32_t slot = p.state_slot[seq];
    if (slot < 0 || (int64_t)slot >= p.n_slots) {
        if (tid == 0) flag(L.status, KDA_DEV_BAD_SLOT);
        return;
    }
    const int64_t head = (int64_t)slot * H + h;
    float* S = p.pool + head * D * D;
    const int cq = lane % LPR;
    const int rbase = warp * (RPT * RPW) + lane / LPR;

    // the prologue's operands first (small, so they return before the state):
    // each thread takes the (tensor, channel) pairs e = tid + NT j of q, k, v
    constexpr int NE = (3 * D + NT - 1) / NT;
    const int64_t vec = sh * D;
    __nv_bfloat16* cst = static_cast<__nv_bfloat16*>(p.conv_state) + head * 3 * (kConv - 1) * D;
    __nv_bfloat16 cv[NE][kConv];               // the window: 3 stored inputs, then the token
    float wv[NE][kConv];
#pragma unroll
    for (int j = 0; j < NE; ++j) {
        const int e = tid + NT * j;
        if (e < 3 * D) {
            const int which = e / D, c = e - which * D;
            const void* xsrc = which == 0 ? p.xq : which == 1 ? p.xk : p.xv;
            const __nv_bfloat16* cs = cst + (int64_t)which * (kConv - 1) * D + c;
            const float* w = p.conv_w + ((int64_t)(h * 3 + which) * kConv) * D + c;
#pragma unroll
            for (int tau = 0; tau < kConv - 1; ++tau) cv[j][tau] = cs[tau * D];
            cv[j][kConv - 1] = static_cast<const __nv_bfloat16*>(xsrc)[vec + c];
#pragma unroll
            for (int tau = 0; tau < kConv; ++tau) wv[j][tau] = w[tau * D];
        }
    }
    float av[(D + NT - 1) / NT];
#pragma unroll
    for (int j = 0; j < (D + NT - 1) / NT; ++j) {
        const int c = tid + NT * j;
        av[j] = c < D ? bf(p.a, vec + c) : 0.f;
    }
    // the epilogue's inputs too: beta's logit, and per output channel the norm
    // weight and the output gate's logit
    const float b_logit = bf(p.b, sh);
    float nw = 0.f, g_logit = 0.f;
    if (tid < TJ) {
        nw = p.norm_w[(int64_t)h * D + tid];
        g_logit = bf(p.g, vec + tid);
    }

    // then the state, held in registers until the update
    float4 st[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m)
        st[m] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(rbase + m * RPW) * D + 4 * cq));

    // ---- prologue: causal convolution of q, k, v with the state update
#pragma unroll
    for (int j = 0; j < NE; ++j) {
        const int e = tid + NT * j;
        if (e < 3 * D) {
            const int which = e / D, c = e - which * D;
            float acc = wv[j][0] * __bfloat162float(cv[j][0]);
#pragma unroll
            for (int tau = 1; tau < kConv; ++tau) acc = fmaf(wv[j][tau], __bfloat162float(cv[j][tau]), acc);
            s_y[which][c] = acc * sigmoidf(acc);    // silu
            __nv_bfloat16* cs = cst + (int64_t)which * (kConv - 1) * D + c;
#pragma unroll
            for (int tau = 0; tau < kConv - 1; ++tau) cs[tau * D] = cv[j][tau + 1];
        }
    }
#pragma unroll
    for (int j = 0; j < (D + NT - 1) / NT; ++j) {
        const int c = tid + NT * j;
        if (c < D) s_a[c] = 1.f / (1.f + expf(av[j]));     // exp(-softplus(a))
    }
    __syncthreads();
    if (warp < 3) {                             // |y_q|^2, |y_k|^2, y_q . y_k
        float acc = 0.f;
        for (int c = lane; c < D; c += 32) {
            const float x0 = s_y[warp == 1 ? 1 : 0][c], x1 = s_y[warp == 0 ? 0 : 1][c];
            acc = fmaf(x0, x1, acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) s_sum[warp] = acc;
    }
    __syncthreads();
    const float rq = 1.f / sqrtf(s_sum[0] + kQkEps), rk = 1.f / sqrtf(s_sum[1] + kQkEps);
    const float qk = s_sum[2] * rq * rk;
    for (int c = tid; c < D; c += NT) {
        const float qi = s_y[0][c] * rq, ki = s_y[1][c] * rk, a = s_a[c];
        s_ka[c] = a * ki;
        s_qa[c] = a * qi;
        s_k[c] = ki;
    }
    __syncthreads();

    // ---- the recurrent update (as in the decode kernel)
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
    float o = 0.f;
    if (tid < TJ) {
        float av = 0.f, bv = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            av += s_red_a[w][tid];
            bv += s_red_b[w][tid];
        }
        const float beta = sigmoidf(b_logit);
        const float u = beta * (s_y[2][tid] - av);
        s_u[tid] = u;
        o = fmaf(u, qk, bv);
        float sq = o * o;                        // mean(o^2): warps of the first TJ threads
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
        if (lane == 0) s_osq[warp] = sq;
    }
    __syncthreads();
    // the state leaves first, then the gated RMSNorm output
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
        __stcs(reinterpret_cast<float4*>(S + (int64_t)(rbase + m * RPW) * D + 4 * cq), r);
    }
    if (tid < TJ) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < TJ / 32; ++w) tot += s_osq[w];
        const float r = 1.f / sqrtf(tot / (float)TJ + p.norm_eps);
        const float yj = nw * o * r * sigmoidf(g_logit);
        static_cast<__nv_bfloat16*>(p.y)[vec + tid] = __float2bfloat16_rn(yj);
    }
}

}  // namespace

cudaError_t launch_fused_decode(const FusedDecodeLaunch& L, cudaStream_t s) {
    const unsigned blocks = (unsigned)((int64_t)L.a.n_seqs * L.a.n_heads);
    note_launch();
    if (L.a.d == 128) fused_decode_kernel<128, 256><<<blocks, 256, 0, s>>>(L);
    else fused_decode_kernel<64, 128><<<blocks, 128, 0, s>>>(L);
    return cudaGetLastError();
}

}  // namespace kda
