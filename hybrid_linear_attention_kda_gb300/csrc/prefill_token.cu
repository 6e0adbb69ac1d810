// Token-serial KDA prefill: the recurrence evaluated one token at a time with the
// fp32 state held in registers.  It serves fp32 q/k/v (where the chunked bf16
// tensor-core form cannot reach fp32 accuracy) and every shape the chunked
// kernels do not cover (d_k = 64).
//
// The state update is the gated delta rule of "Kimi K3 Tech Intro", section 2.1
// (one fixed-size state per head, updated in place for every token):
//     S' = Diag(alpha) S ;  u = beta (v - S'^T k) ;  S <- S' + k u^T ;  o = scale S^T q
// evaluated per value column j in one pass over the state:
//     a_j = sum_i (alpha_i k_i) S_ij ,  b_j = sum_i (alpha_i q_i) S_ij ,
//     u_j = beta (v_j - a_j) ,  o_j = scale (b_j + u_j (q . k)) ,
//     S_ij <- alpha_i S_ij + k_i u_j .
// Snapshots ("Kimi K3 Tech Intro", sections 2.2-2.4): after the token that ends at
// absolute position p with p % snap_interval == 0, the state goes to pool slot
// snap_table[seq][p / snap_interval - 1] (skipped when -1).
//
// One CTA owns a TJ-column tile of one (sequence, head) state, so the CTAs of a
// head run independently; each token costs two block barriers.
#include "kda_common.cuh"

namespace kda {
namespace {

template <typename T, int D, int TJ, int NT>
__global__ void __launch_bounds__(NT) prefill_token_kernel(PrefillLaunch p) {
    constexpr int LPR = TJ / 4;          // lanes per state row (one float4 each)
    constexpr int RPW = 32 / LPR;        // rows covered by one warp instruction
    constexpr int NW = NT / 32;
    constexpr int RPT = D / (NW * RPW);  // rows held by each thread
    constexpr int NTILE = D / TJ;
    static_assert(LPR * RPW == 32 && RPT * NW * RPW == D && NT >= D && NT >= TJ, "tile shape");

    __shared__ float s_ka[2][D], s_qa[2][D], s_a[2][D], s_k[2][D], s_qk_part[2][NW];
    __shared__ float s_v[2][TJ], s_beta[2];
    __shared__ float s_red_a[NW][TJ], s_red_b[NW][TJ];
    __shared__ __align__(16) float s_u[TJ];

    const kda_prefill_args& a = p.a;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.n_heads;
    const int tile = blockIdx.x % NTILE;
    const int64_t sh = blockIdx.x / NTILE;
    const int seq = (int)(sh / H);
    const int head = (int)(sh - (int64_t)seq * H);
    const int j0 = tile * TJ;
    if (p.chain_flag && !p.chain_flag[sh]) return;

    const int64_t t_begin = a.cu_seqlens[seq], t_end = a.cu_seqlens[seq + 1];
    if (t_end < t_begin || t_end > a.total_tokens || t_begin < 0) {
        if (tid == 0) flag(p.status, KDA_DEV_BAD_SEQLENS);
        return;
    }
    const int64_t pos0 = a.start_pos ? a.start_pos[seq] : 0;
    if (pos0 < 0 || pos0 % a.snap_interval != 0) {
        if (tid == 0) flag(p.status, KDA_DEV_BAD_START);
        return;
    }
    const int32_t init = a.init_slot ? a.init_slot[seq] : -1;
    if (init < -1 || (init >= 0 && (int64_t)init >= a.n_slots)) {
        if (tid == 0) flag(p.status, KDA_DEV_BAD_SLOT);
        return;
    }

    const int64_t slot_stride = (int64_t)H * D * D;   // floats per pool slot
    const int64_t head_off = (int64_t)head * D * D;
    const int cq = lane % LPR;
    const int rbase = warp * (RPT * RPW) + lane / LPR;

    float4 st[RPT];
    if (init >= 0) {
        const float* S0 = a.pool + (int64_t)init * slot_stride + head_off;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = rbase + m * RPW;
            st[m] = *reinterpret_cast<const float4*>(S0 + (int64_t)i * D + j0 + 4 * cq);
        }
    } else {
#pragma unroll
        for (int m = 0; m < RPT; ++m) st[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    T* o = static_cast<T*>(a.o);

    // Stage token t's vectors into buffer b (threads tid < D handle channel tid).
    auto stage = [&](int64_t t, int b) {
        const int64_t row = t * H + head;
        if (tid < D) {
            const float al = a.alpha[row * D + tid];
            const float kk = Elem<T>::load(k + row * D + tid);
            const float qq = Elem<T>::load(q + row * D + tid);
            s_a[b][tid] = al;
            s_ka[b][tid] = al * kk;
            s_qa[b][tid] = al * qq;
            s_k[b][tid] = kk;
            float pq = qq * kk;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) pq += __shfl_xor_sync(0xffffffffu, pq, off);
            if (lane == 0) s_qk_part[b][warp] = pq;
        }
        if (tid < TJ) s_v[b][tid] = Elem<T>::load(v + row * D + j0 + tid);
        if (tid == 0) s_beta[b] = a.beta[row];
    };

    if (t_begin < t_end) stage(t_begin, 0);
    __syncthreads();

    for (int64_t t = t_begin; t < t_end; ++t) {
        const int b = (int)((t - t_begin) & 1);
        // partial a_j, b_j over this thread's rows, then across the warp's row groups
        float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = rbase + m * RPW;
            const float ka = s_ka[b][i], qa = s_qa[b][i];
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
        // prefetch the next token into the other buffer (its previous readers
        // finished before the barrier above)
        if (t + 1 < t_end) stage(t + 1, b ^ 1);

        if (tid < TJ) {
            float sa = 0.f, sb = 0.f, qk = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                sa += s_red_a[w][tid];
                sb += s_red_b[w][tid];
            }
#pragma unroll
            for (int w = 0; w < (D + 31) / 32; ++w) qk += s_qk_part[b][w];
            const float u = s_beta[b] * (s_v[b][tid] - sa);
            s_u[tid] = u;
            o[(t * H + head) * D + j0 + tid] = Elem<T>::cvt(a.scale * fmaf(u, qk, sb));
        }
        __syncthreads();

        const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * cq]);
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = rbase + m * RPW;
            const float ai = s_a[b][i], ki = s_k[b][i];
            st[m].x = fmaf(ai, st[m].x, ki * u4.x);
            st[m].y = fmaf(ai, st[m].y, ki * u4.y);
            st[m].z = fmaf(ai, st[m].z, ki * u4.z);
            st[m].w = fmaf(ai, st[m].w, ki * u4.w);
        }

        // snapshot after the token that ends at a multiple of snap_interval
        const int64_t p_after = pos0 + (t - t_begin) + 1;
        if (a.snap_table && p_after % a.snap_interval == 0) {
            const int64_t ord = p_after / a.snap_interval - 1;
            if (ord >= a.snap_table_stride) {
                if (tid == 0) flag(p.status, KDA_DEV_BAD_ORDINAL);
            } else {
                const int32_t slot = a.snap_table[(int64_t)seq * a.snap_table_stride + ord];
                if (slot >= 0 && (int64_t)slot < a.n_slots) {
                    float* dst = a.pool + (int64_t)slot * slot_stride + head_off;
#pragma unroll
                    for (int m = 0; m < RPT; ++m) {
                        const int i = rbase + m * RPW;
                        *reinterpret_cast<float4*>(dst + (int64_t)i * D + j0 + 4 * cq) = st[m];
                    }
                } else if (slot != -1 && tid == 0) {
                    flag(p.status, KDA_DEV_BAD_SLOT);
                }
            }
        }
    }

    if (a.final_state) {
        float* dst = a.final_state + (int64_t)seq * slot_stride + head_off;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = rbase + m * RPW;
            *reinterpret_cast<float4*>(dst + (int64_t)i * D + j0 + 4 * cq) = st[m];
        }
    }
}

template <typename T, int D, int TJ, int NT>
cudaError_t launch_t(const PrefillLaunch& p, cudaStream_t s) {
    const int64_t blocks = (int64_t)p.a.n_seqs * p.a.n_heads * (D / TJ);
    if (blocks == 0) return cudaSuccess;
    note_launch();
    prefill_token_kernel<T, D, TJ, NT><<<(unsigned)blocks, NT, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_token(const PrefillLaunch& p, cudaStream_t s) {
    if (p.a.d_k == 128)
        return p.a.dtype == KDA_BF16 ? launch_t<__nv_bfloat16, 128, 32, 128>(p, s)
                                     : launch_t<float, 128, 32, 128>(p, s);
    return p.a.dtype == KDA_BF16 ? launch_t<__nv_bfloat16, 64, 32, 64>(p, s)
                                 : launch_t<float, 64, 32, 64>(p, s);
}

}  // namespace kda
