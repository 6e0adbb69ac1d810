/*
 * kda_oracle.c -- plain float64 CPU oracle of the KDA (Kimi Delta Attention) layer.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this library.  It shares no code, header, table or
 * constant with the GPU library, and it never calls it.
 *
 * What it computes.  "Kimi K3 Tech Intro" (tim-wang blog), section 2.1: a KDA layer
 * keeps, per head, one fixed-size recurrent state matrix S (plus a conv state,
 * not modelled here) that does not grow with the sequence and is updated in
 * place for every token.  The update is the gated delta rule with a per-channel
 * decay alpha_t in (0,1)^{d_k} and a write strength beta_t in (0,1):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t                     (scale = 1 in every workload)
 *
 * with S in R^{d_k x d_v}.  This file evaluates it token by token in float64 in
 * the algebraically identical split form
 *
 *     S'  = Diag(alpha_t) S_{t-1}         (the decay scales the d_k row index)
 *     u   = beta_t (v_t - S'^T k_t)
 *     S_t = S' + k_t u^T
 *
 * Every sum over the d_k index runs in ascending order, and the file is built
 * with -ffp-contract=off, so results are identical on every host and a resumed
 * run reproduces a full run bit for bit.
 *
 * Snapshots.  "Kimi K3 Tech Intro" sections 2.2-2.4: the state is cached at the
 * prefix-match unit (256 tokens there), decoupled from the 4096-token physical
 * block, and a later request resumes from the cached state at a hash boundary.
 * Here the snapshot with ordinal m of a sequence is S after the token that ends
 * at absolute position p = (m + 1) * interval, i.e. after token p - 1; absolute
 * positions start at start_pos[seq] (0 when start_pos is NULL), so a resumed
 * sequence keeps the ordinals of the run it continues.
 *
 * Inputs are read in their stored precision and widened exactly to float64:
 * q, k, v as bf16 bit patterns, fp32 or fp64; alpha and beta as fp32 or fp64.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_BF16 = 0, ORC_F32 = 1, ORC_F64 = 2 };

static double load_elem(const void *base, int dtype, int64_t idx) {
    if (dtype == ORC_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype == ORC_F32) return (double)((const float *)base)[idx];
    return ((const double *)base)[idx];
}

/*
 * Run the recurrence over a packed variable-length batch.
 *
 *   q, k        [T_tot, H, d_k]  (qkv_dtype)
 *   v           [T_tot, H, d_v]  (qkv_dtype)
 *   alpha       [T_tot, H, d_k]  (gate_dtype), beta [T_tot, H] (gate_dtype)
 *   cu_seqlens  [n_seqs + 1], cu_seqlens[0] = 0, non-decreasing
 *   start_pos   [n_seqs] absolute position of each sequence's first token, or NULL
 *   init_state  [n_seqs, H, d_k, d_v] float64, or NULL for zero states
 *   o           [T_tot, H, d_v] float64 output, or NULL
 *   final_state [n_seqs, H, d_k, d_v] float64 output, or NULL
 *   snap_req    [n_req, 2] pairs (seq, ordinal); snap_out [n_req, H, d_k, d_v]
 *               receives the requested snapshots (entries never reached stay
 *               untouched); both may be NULL when n_req = 0
 *   heads       only heads h0 <= h < h1 are computed and written
 *
 * Returns 0, or -1 on an argument error.  Work is split over (sequence, head)
 * pairs with OpenMP; pairs are independent.
 */
int kda_oracle_run(int32_t n_seqs, int32_t H, int32_t d_k, int32_t d_v,
                   int32_t qkv_dtype, const void *q, const void *k, const void *v,
                   int32_t gate_dtype, const void *alpha, const void *beta,
                   const int32_t *cu_seqlens, const int32_t *start_pos,
                   const double *init_state, double scale,
                   double *o, double *final_state,
                   int32_t snap_interval, int64_t n_req, const int32_t *snap_req,
                   double *snap_out, int32_t h0, int32_t h1)
{
    if (n_seqs < 0 || H <= 0 || d_k <= 0 || d_v <= 0 || h0 < 0 || h1 > H || h0 > h1)
        return -1;
    if (qkv_dtype < ORC_BF16 || qkv_dtype > ORC_F64) return -1;
    if (gate_dtype != ORC_F32 && gate_dtype != ORC_F64) return -1;
    if (n_req > 0 && (snap_req == NULL || snap_out == NULL || snap_interval <= 0)) return -1;
    for (int32_t s = 0; s < n_seqs; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;

    const int64_t n_pairs = (int64_t)n_seqs * (h1 - h0);
    const int64_t state_sz = (int64_t)d_k * d_v;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t pair = 0; pair < n_pairs; ++pair) {
        const int32_t seq = (int32_t)(pair / (h1 - h0));
        const int32_t h = h0 + (int32_t)(pair % (h1 - h0));
        double *S = (double *)malloc(sizeof(double) * (size_t)state_sz);
        double *kt = (double *)malloc(sizeof(double) * (size_t)(2 * d_k + 2 * d_v));
        if (!S || !kt) { free(S); free(kt); bad |= 1; continue; }
        double *qt = kt + d_k, *vt = qt + d_k, *acc = vt + d_v;

        if (init_state)
            memcpy(S, init_state + ((int64_t)seq * H + h) * state_sz,
                   sizeof(double) * (size_t)state_sz);
        else
            memset(S, 0, sizeof(double) * (size_t)state_sz);

        const int64_t t_begin = cu_seqlens[seq], t_end = cu_seqlens[seq + 1];
        const int64_t pos0 = start_pos ? start_pos[seq] : 0;
        for (int64_t t = t_begin; t < t_end; ++t) {
            const int64_t row = t * H + h;
            for (int32_t i = 0; i < d_k; ++i) {
                kt[i] = load_elem(k, qkv_dtype, row * d_k + i);
                qt[i] = load_elem(q, qkv_dtype, row * d_k + i);
            }
            for (int32_t j = 0; j < d_v; ++j) {
                vt[j] = load_elem(v, qkv_dtype, row * d_v + j);
                acc[j] = 0.0;
            }
            const double b = load_elem(beta, gate_dtype, row);

            /* S' = Diag(alpha) S ;  acc = S'^T k */
            for (int32_t i = 0; i < d_k; ++i) {
                const double a = load_elem(alpha, gate_dtype, row * d_k + i);
                double *Si = S + (int64_t)i * d_v;
                for (int32_t j = 0; j < d_v; ++j) {
                    Si[j] = a * Si[j];
                    acc[j] = acc[j] + kt[i] * Si[j];
                }
            }
            /* u = beta (v - S'^T k) */
            for (int32_t j = 0; j < d_v; ++j) acc[j] = b * (vt[j] - acc[j]);
            /* S = S' + k u^T ;  o = scale * S^T q */
            double *ot = o ? o + row * d_v : NULL;
            if (ot)
                for (int32_t j = 0; j < d_v; ++j) ot[j] = 0.0;
            for (int32_t i = 0; i < d_k; ++i) {
                double *Si = S + (int64_t)i * d_v;
                for (int32_t j = 0; j < d_v; ++j) {
                    Si[j] = Si[j] + kt[i] * acc[j];
                    if (ot) ot[j] = ot[j] + qt[i] * Si[j];
                }
            }
            if (ot)
                for (int32_t j = 0; j < d_v; ++j) ot[j] = scale * ot[j];

            /* snapshot when the absolute position after this token is a multiple */
            const int64_t p = pos0 + (t - t_begin) + 1;
            if (n_req > 0 && p % snap_interval == 0) {
                const int64_t ord = p / snap_interval - 1;
                for (int64_t r = 0; r < n_req; ++r)
                    if (snap_req[2 * r] == seq && snap_req[2 * r + 1] == ord)
                        memcpy(snap_out + (r * H + h) * state_sz, S,
                               sizeof(double) * (size_t)state_sz);
            }
        }
        if (final_state)
            memcpy(final_state + ((int64_t)seq * H + h) * state_sz, S,
                   sizeof(double) * (size_t)state_sz);
        free(S);
        free(kt);
    }
    return bad ? -1 : 0;
}

/* Number of OpenMP threads the oracle runs on (reported with CPU timings). */
int kda_oracle_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
