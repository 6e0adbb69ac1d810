/*
 * kda.h -- C ABI of the GB300 (sm_103a) KDA library, libkda.so.
 *
 * KDA (Kimi Delta Attention) is the linear-attention layer that makes up most of
 * Kimi K3's layers.  Per head it keeps one fixed-size recurrent state
 * S in R^{d_k x d_v} (fp32 here) that is updated in place for every token
 * ("Kimi K3 Tech Intro", section 2.1; the vLLM Kimi K3 launch post, "Kimi Delta
 * Attention" paragraph).  The update is the gated delta rule with a
 * per-channel decay alpha_t in (0,1)^{d_k} and a write strength beta_t in (0,1):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * The library has two modes: a chunked prefill over a packed variable-length
 * batch that writes state snapshots every snap_interval tokens and can resume
 * from one ("Kimi K3 Tech Intro", sections 2.2-2.4: the 256-token prefix-match
 * unit, copy-on-write reuse of a cached state), and a batched single-token
 * decode step that updates states in place ("Kimi K3 Tech Intro", section 4.1,
 * the fused KDA decode kernel).  Two copy calls move states between the
 * block-indexed state pool and contiguous buffers (copy-on-write, section 2.3).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise, owned
 *    by the caller.  The library never allocates device memory; the only
 *    scratch is the caller's workspace (prefill).
 *  - Layouts are row-major with the last index contiguous:
 *      q, k   [T, H, d_k]      v, o  [T, H, d_v]       (T = tokens, H = heads)
 *      alpha  [T, H, d_k] fp32 beta  [T, H] fp32
 *      state pool [n_slots, H, d_k, d_v] fp32: one slot holds the H states of
 *      one sequence at one position.
 *    q, k, v, o share one element type (kda_dtype_t).  Device pointers must be
 *    16-byte aligned.
 *  - Supported shapes: d_k == d_v in {64, 128}; chunk == 64; snap_interval == 256.
 *    Anything else returns KDA_ERR_UNSUPPORTED.  Every prefill runs the chunked
 *    form (the block-matrix form of the yunthe.com "Kimi K3 open-source
 *    practice" page, FlashKDA paragraph): bf16 inputs with d = 128 on tensor
 *    cores (bf16 operands, fp32 accumulation and fp32 state), fp32 inputs and
 *    d = 64 with the same chunk algorithm in fp32 SIMT arithmetic.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and run on the current CUDA device.  Argument errors that
 *    the host can see come back synchronously, before anything is launched.  A
 *    failed launch returns KDA_ERR_CUDA.  Bad indices that only the device can
 *    see (a slot outside the pool, a start position that is not a multiple of
 *    snap_interval, a decreasing cu_seqlens, a snapshot ordinal beyond the
 *    table) never trap: the kernel skips that work and sets a bit in a per-device
 *    status word that kda_check_status() reports.
 *  - Copy-on-write is the caller's job, as in the pages' design (section 2.3):
 *    a state that other requests still share must be copied to a private slot
 *    (kda_snapshot_gather / kda_snapshot_restore) before a call that writes it,
 *    and a snapshot written by a call must not be read by another sequence of
 *    the same call (reuse waits for the next step, section 2.4).  Decode slots
 *    must be distinct; the library does not check this.
 *
 * Every function returns a kda_status_t; kda_status_string() names it and
 * kda_last_error() gives a one-line description of the last failure on the
 * calling host thread.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 1

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null pointer, negative count, misaligned pointer, small workspace */
    KDA_ERR_UNSUPPORTED = 2,   /* shape or dtype outside the supported set */
    KDA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    KDA_ERR_DEVICE_STATUS = 4, /* kda_check_status: a kernel flagged bad indices */
    KDA_ERR_TIMEOUT = 5,       /* kda_check_status: the stream did not drain in time */
    KDA_ERR_NO_MEMORY = 6      /* host memory for a host-side structure could not be allocated */
} kda_status_t;

typedef enum {
    KDA_BF16 = 0, /* q, k, v, o stored as bfloat16 */
    KDA_FP32 = 1  /* q, k, v, o stored as float */
} kda_dtype_t;

/* Bits of the device status word (kda_device_status). */
#define KDA_DEV_BAD_SLOT      0x1u /* init / snapshot / decode / copy slot outside [0, n_slots) */
#define KDA_DEV_BAD_START     0x2u /* start_pos < 0 or not a multiple of snap_interval */
#define KDA_DEV_BAD_SEQLENS   0x4u /* cu_seqlens decreasing, or past total_tokens */
#define KDA_DEV_BAD_ORDINAL   0x8u /* snapshot ordinal >= snap_table_stride */
#define KDA_DEV_WAIT_TIMEOUT  0x10u /* a kernel gave up waiting on its own copies / MMAs (about 1 s) */
#define KDA_DEV_BAD_ACCEPT    0x20u /* kda_decode_commit: an accepted count outside [0, n_tokens] */

/*
 * Chunked prefill over a packed variable-length batch.
 *
 * Sequence s owns tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 of the packed
 * tensors.  Its first token sits at absolute position start_pos[s] (0 when
 * start_pos is NULL), which must be a multiple of snap_interval: a resume starts
 * at a snapshot boundary ("Kimi K3 Tech Intro", section 2.4: the scheduler stops
 * at a hash boundary).  Its initial states are pool slot init_slot[s] (all H
 * heads), or zero when init_slot is NULL or init_slot[s] == -1.
 *
 * After the token that ends at absolute position p, for every p that is a
 * positive multiple of snap_interval, the H states are written to pool slot
 * snap_table[s * snap_table_stride + p / snap_interval - 1] unless that entry is
 * -1 (snapshot ordinals are absolute, so a resumed sequence continues the
 * numbering of the run it resumes).  snap_table may be NULL (no snapshots).
 * The states after each sequence's last token go to final_state
 * [n_seqs, H, d_k, d_v] fp32 unless it is NULL; an empty sequence's final
 * states are its initial states.  Outputs go to o.
 *
 * Chunks are aligned to absolute multiples of `chunk`, and every reduction has
 * a fixed order, so a resumed run reproduces a full run bit for bit.
 *
 * The workspace holds the chunk table and one record per (chunk, head) between
 * the chunk-local stage and the state carry: 74,240 bytes on the tensor-core
 * path, (4 * 64 * d + 64 * 64 + d) * 4 bytes on the fp32 SIMT path, for at most
 * total_tokens / 64 + n_seqs chunks.  kda_prefill_workspace_size gives the
 * exact figure; it is 0 only for an empty batch or invalid sizes.
 */
typedef struct kda_prefill_args {
    int32_t n_seqs;            /* >= 0 */
    int32_t n_heads;           /* H >= 1 */
    int32_t d_k;               /* 64 or 128 */
    int32_t d_v;               /* == d_k */
    int32_t chunk;             /* 64 */
    int32_t snap_interval;     /* 256 */
    int32_t dtype;             /* kda_dtype_t of q, k, v, o */
    float scale;               /* output scale (1 for the plain rule) */
    int64_t total_tokens;      /* host copy of cu_seqlens[n_seqs] */
    int64_t n_slots;           /* slots in pool (0 if pool is NULL) */
    int32_t snap_table_stride; /* entries per sequence in snap_table */
    int32_t reserved0;         /* must be 0 */
    const void *q, *k, *v;     /* [T, H, d_k], [T, H, d_k], [T, H, d_v] */
    const float *alpha;        /* [T, H, d_k], each in (0, 1] */
    const float *beta;         /* [T, H] */
    const int32_t *cu_seqlens; /* [n_seqs + 1], cu_seqlens[0] = 0, non-decreasing */
    const int32_t *start_pos;  /* [n_seqs] or NULL */
    const int32_t *init_slot;  /* [n_seqs] or NULL */
    float *pool;               /* [n_slots, H, d_k, d_v] or NULL */
    const int32_t *snap_table; /* [n_seqs, snap_table_stride] or NULL */
    void *o;                   /* [T, H, d_v] */
    float *final_state;        /* [n_seqs, H, d_k, d_v] or NULL */
    void *workspace;           /* >= kda_prefill_workspace_size(args) bytes, 256-B aligned */
    size_t workspace_bytes;
} kda_prefill_args;

/* Bytes of workspace kda_prefill_chunked needs for these arguments (only the
 * sizes are read).  Returns 0 when the sizes are invalid. */
size_t kda_prefill_workspace_size(const kda_prefill_args *args);

/* Chunked prefill; see kda_prefill_args.  `args` is a host pointer, read
 * before the call returns. */
kda_status_t kda_prefill_chunked(const kda_prefill_args *args, void *stream);

/*
 * kda_prefill_chunked with timing marks: on `stream`, records events[i] before
 * the i-th kernel of the prefill and one more after the last, for at most
 * n_events events (cudaEvent_t handles created by the caller, timing enabled).
 * *n_recorded receives the number recorded (kernels + 1) and names[i] (when
 * names is non-NULL, room for n_events entries) the static name of the kernel
 * that starts at events[i].  For measurement; the results equal those of
 * kda_prefill_chunked.
 */
kda_status_t kda_prefill_chunked_events(const kda_prefill_args *args, void *stream,
                                        void *const *events, int32_t n_events,
                                        int32_t *n_recorded, const char **names);

/*
 * kda_prefill_chunked for callers that cannot allocate device memory: the same
 * arguments (args->workspace and args->workspace_bytes are ignored), with the
 * prefill's scratch taken from a 64 MiB array in the library's own static device
 * memory, which every GPU that loads the library holds until process exit.  The
 * pages describe no counterpart to this call; it exists for serving code whose device
 * memory is all reserved up front, or that may not allocate on its latency
 * path.  Allocates nothing.  Returns KDA_ERR_UNSUPPORTED when
 * kda_prefill_workspace_size(args) exceeds 64 MiB.  In practice that is about
 * 900 (chunk, head) records on the bf16, d = 128 path (74,240 bytes each, for
 * total_tokens / 64 + n_seqs chunks times H heads): for example one 7,000-token
 * sequence with 8 heads, or 1,700 tokens with 32 heads.  The fp32 SIMT path's
 * records are twice as large.  All calls share the array: calls that overlap on
 * the GPU race on it.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) and should come before any stream capture.
 */
kda_status_t kda_prefill_chunked_noalloc(const kda_prefill_args *args, void *stream);

/*
 * One decode step for n_seqs sequences, one token each ("Kimi K3 Tech Intro",
 * section 4.1: the recurrent update of the fused decode kernel, with the state
 * updated in place).  Sequence s reads and rewrites the H states in pool slot
 * state_slot[s]:
 *     S <- (I - beta k k^T) Diag(alpha) S + beta k v^T ;  o = scale * S^T q
 * q, k [n_seqs, H, d_k]; v, o [n_seqs, H, d_v]; alpha [n_seqs, H, d_k];
 * beta [n_seqs, H]; state_slot [n_seqs] device int32.  Slots must be distinct.
 */
kda_status_t kda_decode_step(int32_t n_seqs, int32_t n_heads, int32_t d_k, int32_t d_v,
                             int32_t dtype, const void *q, const void *k, const void *v,
                             const float *alpha, const float *beta, float *pool,
                             int64_t n_slots, const int32_t *state_slot, void *o,
                             float scale, void *stream);

/*
 * One fused decode step of the whole KDA layer, after its input projection
 * ("Kimi K3 Tech Intro", section 4.1).  The step fuses the causal convolution,
 * the q/k norm, the gates, the recurrent update and the gated RMSNorm into one
 * kernel.  The convolution state and the recurrent state are updated in place
 * (section 2.1 names the two per-request states).
 *
 * Per (sequence, head), from the raw projections of one token:
 *   y_x = silu(sum_tau conv_w[h, x, tau] * [C_x, x_x][tau])  for x in q, k, v
 *                                                           (tap conv_size-1 is the token)
 *   C_x <- the last conv_size-1 raw inputs (oldest first)
 *   q = y_q / sqrt(|y_q|^2 + 1e-6),  k likewise,  v = y_v
 *   alpha = exp(-softplus(a)),  beta = sigmoid(b)
 *   S <- Diag(alpha) S + k (beta (v - (Diag(alpha) S)^T k))^T,   o = S^T q
 *   y = norm_w[h] * o / sqrt(mean(o^2) + norm_eps) * sigmoid(g)
 * The pages name these steps but not their forms; the forms above are this
 * library's reading (width-4 depthwise convolution with SiLU, L2 q/k norm,
 * sigmoid-gated RMSNorm).
 *
 * Layouts (device, row-major):
 *   xq, xk, xv, a, g  bf16 [n_seqs, H, d];  b bf16 [n_seqs, H]
 *   conv_w fp32 [H, 3, conv_size, d] (q, k, v);  norm_w fp32 [H, d]
 *   pool fp32 [n_slots, H, d, d];  conv_state bf16 [n_slots, H, 3, conv_size-1, d]
 *   state_slot int32 [n_seqs] (distinct);  y bf16 [n_seqs, H, d]
 * Supported: d in {64, 128}, conv_size == 4, reserved0 == 0.  Anything else
 * returns KDA_ERR_UNSUPPORTED / KDA_ERR_INVALID_ARG.  A slot outside the pool
 * sets KDA_DEV_BAD_SLOT and skips the sequence.
 */
typedef struct {
    int32_t n_seqs, n_heads, d, conv_size;
    float norm_eps;
    int32_t reserved0;
    int64_t n_slots;
    const void *xq, *xk, *xv, *a, *b, *g;
    const float *conv_w, *norm_w;
    float *pool;
    void *conv_state;
    const int32_t *state_slot;
    void *y;
} kda_fused_decode_args;

kda_status_t kda_decode_fused(const kda_fused_decode_args *args, void *stream);

/*
 * Speculative decoding, step one: verify n_tokens candidate tokens per sequence
 * ("Kimi K3 Tech Intro", section 6: a draft model proposes 7 tokens, the target
 * model checks them in one step and keeps the accepted prefix).  For every
 * (sequence, head) the state pool[state_slot[i]] is read, not written.  The
 * call runs the candidate tokens t = 0 .. n_tokens-1 through a private copy and
 * writes, for each t:
 *   - o[i, t]: scale S_t^T q_t, where S_t is the state after token t;
 *   - u[i, t]: beta_t (v_t - (Diag(alpha_t) S_{t-1})^T k_t), the update vector
 *     that kda_decode_commit() applies.
 * Token t of sequence i therefore sees the earlier candidates of i, as in n_tokens
 * consecutive decode steps.
 * Layouts (device, row-major): q, k, alpha [n_seqs, n_tokens, H, d_k];
 * v, o, u [n_seqs, n_tokens, H, d_v]; beta [n_seqs, n_tokens, H];
 * state_slot [n_seqs] int32.  o has the element type of q, k, v; u is fp32,
 * caller-owned scratch.
 * Errors:
 *   - n_tokens outside [1, 16], and the unsupported shapes of kda_decode_step,
 *     return an error status;
 *   - a slot outside the pool sets KDA_DEV_BAD_SLOT and skips the sequence.
 */
kda_status_t kda_decode_verify(int32_t n_seqs, int32_t n_tokens, int32_t n_heads, int32_t d_k, int32_t d_v,
                               int32_t dtype, const void *q, const void *k, const void *v,
                               const float *alpha, const float *beta, const float *pool,
                               int64_t n_slots, const int32_t *state_slot, void *o, float *u,
                               float scale, void *stream);

/*
 * Speculative decoding, step two: commit the accepted tokens.  For sequence i,
 * the call applies the updates of its first n_accept[i] candidate tokens to
 * pool[state_slot[i]] in place:
 *     S <- Diag(alpha_t) S + k_t u_t^T,   t = 0 .. n_accept[i]-1,
 * where u comes from the kda_decode_verify() call on the same tokens.  The
 * result is the state after the accepted tokens: the rejected ones leave no
 * trace, and n_accept[i] == 0 leaves the state untouched.  One read and one
 * write per state.
 * Inputs: k, alpha [n_seqs, n_tokens, H, d_k]; u [n_seqs, n_tokens, H, d_v]
 * fp32; n_accept [n_seqs] device int32 in [0, n_tokens].  Slots must be
 * distinct.
 * Errors: a count outside that range sets KDA_DEV_BAD_ACCEPT and a bad slot
 * sets KDA_DEV_BAD_SLOT; either skips the sequence.
 */
kda_status_t kda_decode_commit(int32_t n_seqs, int32_t n_tokens, int32_t n_heads, int32_t d_k, int32_t d_v,
                               int32_t dtype, const void *k, const float *alpha, const float *u,
                               const int32_t *n_accept, float *pool, int64_t n_slots,
                               const int32_t *state_slot, void *stream);

/*
 * Copy n pool slots out to a contiguous buffer: dst[i] = pool[slots[i]]
 * (H x d_k x d_v fp32 each; slots[i] == -1 writes zeros).  The private copy of
 * copy-on-write reuse ("Kimi K3 Tech Intro", section 2.3); bit-exact.
 */
kda_status_t kda_snapshot_gather(const float *pool, int64_t n_slots, const int32_t *slots,
                                 int32_t n, int32_t n_heads, int32_t d_k, int32_t d_v,
                                 float *dst, void *stream);

/*
 * Copy n contiguous states into pool slots: pool[slots[i]] = src[i]
 * (slots[i] == -1 skips entry i).  Target slots must be distinct; bit-exact.
 */
kda_status_t kda_snapshot_restore(const float *src, float *pool, int64_t n_slots,
                                  const int32_t *slots, int32_t n, int32_t n_heads,
                                  int32_t d_k, int32_t d_v, void *stream);

/*
 * Wait for `stream` to drain (at most timeout_ms milliseconds; <= 0 waits
 * without limit), then read and clear the current device's status word.
 * Returns KDA_OK, KDA_ERR_DEVICE_STATUS (bits in *bits_out when non-NULL),
 * KDA_ERR_TIMEOUT (the word is left untouched) or KDA_ERR_CUDA.  Calls on
 * several streams of one device share the word.  Only `stream` is drained: a
 * library kernel still running on another stream can set a bit between the
 * read and the clear, and that bit is lost.  For an exact account, check once
 * the device's other streams have drained as well.
 */
kda_status_t kda_check_status(void *stream, int32_t timeout_ms, uint32_t *bits_out);

/* Name of a status code (static string). */
const char *kda_status_string(kda_status_t status);

/* One-line description of the last failure on this host thread (static storage). */
const char *kda_last_error(void);

/* KDA_ABI_VERSION of the loaded library. */
int32_t kda_abi_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all host threads).  A diagnostic for counting launches in a timed region. */
uint64_t kda_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
