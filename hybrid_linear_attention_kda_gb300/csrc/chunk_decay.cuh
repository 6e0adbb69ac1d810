// Exact intra-chunk decay factors in fp32 SIMT arithmetic, shared by the SIMT
// chunk-local kernel and the tensor-core chunk-local kernel's path for chunks
// whose gates leave its operand range.
//
// The intra-chunk products of the chunked form (the block-matrix form of the
// yunthe.com "Kimi K3 open-source practice" page, FlashKDA paragraph) need, for
// every token pair s <= r of a 64-token chunk and every key channel c,
//     f_rsc = prod_{s < tau <= r} alpha_tau,c      (= exp(g_rc - g_sc))
//   A_rs = beta_r sum_c k_rc k_sc f_rsc   (s < r),   P_rs = sum_c q_rc k_sc f_rsc   (s <= r).
// Every factor here is a product of alphas in (0, 1], so none overflows, an
// underflow is the true value, and alpha = 0 gives exact zeros; nothing is
// divided and no logarithm is taken, so there is no cancellation.  The chunk is
// cut into four 16-token groups; per channel:
//     pin[t]  = prod alpha over [16 b(t), t]          (group start to t)
//     pout[t] = prod alpha over (t, 16 b(t) + 15]     (after t to group end)
//     btot[b] = prod alpha over group b
// so a pair in different groups takes pout[s] * btot[between] * pin[r]; a pair
// in one group multiplies its at most 15 alphas directly.
#pragma once

#include <stdint.h>

namespace kda {

constexpr int kDecayCB = 16;            // channels per block
constexpr int kDecayLd = kDecayCB + 1;  // padded row

struct DecayBlock {
    float al[64][kDecayLd];     // alpha (1 past the chunk's tokens)
    float k[64][kDecayLd];      // k, q as fp32 (0 past the chunk's tokens)
    float q[64][kDecayLd];
    float pin[64][kDecayLd];
    float pout[64][kDecayLd];
    float btot[4][kDecayLd];
};

// pin, pout and btot from al; threads tid = 0 .. nthreads-1 of the block take
// part (64 (channel, group) walks).  The caller synchronises before and after.
__device__ __forceinline__ void decay_tables(DecayBlock& D, int tid, int nthreads) {
    for (int e = tid; e < kDecayCB * 4; e += nthreads) {
        const int c = e % kDecayCB, b = e / kDecayCB;
        float p = 1.f;
        for (int i = 0; i < 16; ++i) {
            p *= D.al[16 * b + i][c];
            D.pin[16 * b + i][c] = p;
        }
        D.btot[b][c] = p;
        float q = 1.f;
        for (int i = 15; i >= 0; --i) {
            D.pout[16 * b + i][c] = q;
            q *= D.al[16 * b + i][c];
        }
    }
}

// prod alpha_c over (s, r], s <= r
__device__ __forceinline__ float pair_decay(const DecayBlock& D, int r, int s, int c) {
    const int br = r >> 4, bs = s >> 4;
    if (br == bs) {
        float f = 1.f;
        for (int t = s + 1; t <= r; ++t) f *= D.al[t][c];
        return f;
    }
    float f = D.pout[s][c] * D.pin[r][c];
    for (int b = bs + 1; b < br; ++b) f *= D.btot[b][c];
    return f;
}

// prod alpha_c over [0, t] (chunk prefix) and over (t, 63] (chunk suffix)
__device__ __forceinline__ float prefix_decay(const DecayBlock& D, int t, int c) {
    float f = D.pin[t][c];
    for (int b = 0; b < (t >> 4); ++b) f *= D.btot[b][c];
    return f;
}
__device__ __forceinline__ float suffix_decay(const DecayBlock& D, int t, int c) {
    float f = D.pout[t][c];
    for (int b = (t >> 4) + 1; b < 4; ++b) f *= D.btot[b][c];
    return f;
}

// Adds this block's channels to the A and P sums of the 16 pairs (r, cs + 4 m),
// m = 0..15, of one thread (without beta; A for s < r, P for s <= r).
__device__ __forceinline__ void accumulate_ap(const DecayBlock& D, int r, int cs, float (&accA)[16],
                                              float (&accP)[16]) {
#pragma unroll 1
    for (int c = 0; c < kDecayCB; ++c) {
        const float kr = D.k[r][c], qr = D.q[r][c];
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int s = cs + 4 * m;
            if (s <= r) {
                const float e = pair_decay(D, r, s, c) * D.k[s][c];
                accP[m] = fmaf(qr, e, accP[m]);
                accA[m] = fmaf(kr, e, accA[m]);
            }
        }
    }
}

}  // namespace kda
