// Shared definitions of the chunked prefill (chunk 64; the tensor-core stages take
// bf16 with d_k = d_v = 128, the SIMT stages of chunk_simt.cu the rest).
//
// The chunked form ("block-matrix" form of the yunthe.com "Kimi K3 open-source
// practice" page, FlashKDA paragraph) of the gated delta rule, for a chunk of
// C = 64 tokens r = 0..C-1 entering with state S (d_k x d_v), where
// g_r = sum_{tau <= r} log alpha_tau per channel (never formed: every factor
// below is a product of alphas over a token range):
//   A_rs  = beta_r sum_c k_rc k_sc exp(g_rc - g_sc)            (s < r)
//   P_rs  =        sum_c q_rc k_sc exp(g_rc - g_sc)            (s <= r)
//   T     = (I + A)^-1
//   W     = T diag(beta) (Gamma * K),  U~ = T diag(beta) V,  Gamma_r = exp(g_r)
//   U     = U~ - W S
//   O     = (Gamma * Q) S + P U
//   S'    = Diag(gamma) S + Kbar^T U,  Kbar_s = exp(g_{C-1} - g_s) * k_s,
//           gamma = exp(g_{C-1})
// Stage one (chunk_local) computes everything that does not involve S for all
// chunks in parallel and writes one record per (chunk, head); stage two
// (chunk_recur) carries S through the chunks of each (sequence, head).
//
// Record of one (chunk, head): bf16 tiles in the 128-byte swizzled layout of
// tc05.cuh, each a [rows x 64] tile (one 128-byte row per row index):
//   W    [c][t]  = W_tc       (128 rows c = key channel, t = token)
//   Q    [c][t]  = Gamma_tc q_tc
//   K    [c][t]  = Kbar_tc
//   U    [j][t]  = U~_tj      (128 rows j = value channel)
//   P    [s][t]  = P_ts       (64 rows s)
//   gam  [c]     fp32 gamma
#pragma once

#include "kda_common.cuh"
#include "tc05.cuh"

namespace kda {

constexpr int kD = 128;        // d_k = d_v of the chunked path
constexpr int kC = 64;         // chunk length
constexpr uint32_t kRecW = 0;
constexpr uint32_t kRecQ = 16384;
constexpr uint32_t kRecK = 32768;
constexpr uint32_t kRecU = 49152;
constexpr uint32_t kRecP = 65536;
constexpr uint32_t kRecG = 73728;
constexpr uint32_t kRecBytes = 74240;       // 72.5 KiB, a multiple of 256

// Smallest alpha-product over at most 16 tokens that the diagonal sub-blocks
// factor through a reference token: the factors and their inverses then stay
// within [2^-100, 2^100], so bf16 operands neither overflow nor flush.  A chunk
// of some head below it is recomputed token by token (chain flagged).
constexpr float kGuardMin = 7.888609052210118e-31f;   // 2^-100

// Long chains split into segments at absolute positions that are multiples of
// kSegTokens.  The carry over a chunk is affine in the state, S' = A_c S + B_c,
// so a segment's map (A, B) comes from running its chunks from the identity
// with U~ = 0 (A) and from zero (B); a scan gives every segment's initial state,
// then all segments run in parallel.
// 57,344 tokens = 896 chunks: a 2^20-token sequence of 8 heads splits into 19
// segments, 152 chains, one per SM of a 152-SM GB300, and its longest chain is
// 896 chunks (65,536-token segments gave 128 chains of 1,024 chunks).
constexpr int64_t kSegTokens = 57344;
constexpr int64_t kSegChunks = kSegTokens / kC;

// Upper bound on the segments of a batch (and on the scratch entries of split
// ones): a sequence of L tokens has at most L / kSegTokens + 2.
__host__ __device__ inline int64_t max_segments(int64_t total_tokens, int64_t n_seqs) {
    return total_tokens / kSegTokens + 2 * n_seqs + 1;
}

// The carry kernel's passes.
enum CarryMode : int32_t {
    kCarryPlain = 0,    // every sequence as one chain (no segments)
    kCarryMap = 1,      // segments of split sequences: identity start, U~ = 0, writes A
    kCarryOffset = 2,   // segments of split sequences: zero start, writes B
    kCarryFinal = 3,    // every segment: outputs, snapshots, final state
    kCarryTailMap = 4,  // the last kTailChunks chunks before each segment boundary: identity
                        // start, U~ = 0; a boundary whose tail map is not exactly zero is
                        // marked for the full map / offset / scan
};

// Chunks of the tail window before a segment boundary.  When the carry over the
// window maps every state to exactly zero (the gates forgot it), the state at the
// boundary is the window run from zero: the offset pass runs over the window
// only and no segment map is needed.
constexpr int64_t kTailChunks = 2;

struct ChunkLaunch {
    kda_prefill_args a;
    int32_t* chunk_base;   // [n_seqs + 1]: first chunk of each sequence, total at [n_seqs]
    int4* chunk_info;      // [max_chunks]: {first packed token, tokens (<= 64), sequence, 0}
    uint8_t* records;      // [max_chunks * H] records (kRecBytes each, or simt_record_bytes(d))
    int64_t max_chunks;
    uint32_t* exact_count;   // items listed in exact_items (zeroed by the meta kernel)
    int64_t* exact_items;    // [max_chunks * H]: items whose P, W, U~ chunk_exact_kernel rewrites
    uint32_t* status;
    // segments (used when split is set)
    int32_t split;         // nonzero: sequences of >= 2 kSegTokens tokens are split
    int32_t mode;          // CarryMode of this carry launch
    int4* seg_info;        // [max_segs]: {sequence, first chunk within it, chunks, scratch index or -1}
    int32_t* seg_count;    // [1 + n_seqs + 1]: segments, then each sequence's first segment (and total)
    float* seg_state;      // [scratch, H, 3, kD, kD]: A, B, initial state of each split segment
    int32_t* seg_slow;     // [scratch, H]: for the boundary at the start of a split segment
                           // (not its sequence's first), nonzero = its tail map is not zero
    int64_t max_segs;
};

// Sequence checks shared by the prefill kernels; true when the sequence is usable.
__device__ __forceinline__ bool seq_valid(const kda_prefill_args& a, int seq, int64_t* t_begin,
                                          int64_t* t_end, int64_t* pos0, int32_t* init,
                                          uint32_t* bad_bits) {
    const int64_t b = a.cu_seqlens[seq], e = a.cu_seqlens[seq + 1];
    *bad_bits = 0;
    if (e < b || e > a.total_tokens || b < 0) {
        *bad_bits = KDA_DEV_BAD_SEQLENS;
        return false;
    }
    const int64_t p = a.start_pos ? a.start_pos[seq] : 0;
    if (p < 0 || p % a.snap_interval != 0) {
        *bad_bits = KDA_DEV_BAD_START;
        return false;
    }
    const int32_t s = a.init_slot ? a.init_slot[seq] : -1;
    if (s < -1 || (s >= 0 && (int64_t)s >= a.n_slots)) {
        *bad_bits = KDA_DEV_BAD_SLOT;
        return false;
    }
    *t_begin = b;
    *t_end = e;
    *pos0 = p;
    *init = s;
    return true;
}

cudaError_t launch_chunk_meta(const ChunkLaunch& p, cudaStream_t s);
cudaError_t launch_chunk_local(const ChunkLaunch& p, cudaStream_t s);
cudaError_t launch_chunk_exact(const ChunkLaunch& p, cudaStream_t s);
cudaError_t launch_chunk_recur(const ChunkLaunch& p, cudaStream_t s);
cudaError_t launch_segment_meta(const ChunkLaunch& p, cudaStream_t s);
cudaError_t launch_segment_scan(const ChunkLaunch& p, cudaStream_t s);

// The same two stages in fp32 SIMT arithmetic (chunk_simt.cu): fp32 q/k/v, or d = 64.
size_t simt_record_bytes(int d);
cudaError_t launch_simt_local(const ChunkLaunch& p, cudaStream_t s);
cudaError_t launch_simt_recur(const ChunkLaunch& p, cudaStream_t s);

}  // namespace kda
