// Hierarchy-aware segsum for one chunk of Q = 32 * NW tokens.
//
// "GPU Hierarchy Meets Structured Matrices" (abstract): the 1-semiseparable
// decay mask L_ij = exp(seg(i, j)), seg(i, j) = sum_{k=j+1..i} l_k, is split
// into 1-SS diagonal blocks (one per warp) and rank-one off-diagonal blocks,
// built from warp-level scans and cross-warp aggregation, with no prefix
// subtraction.
//
// One thread owns one row i = 32 w + lane of the chunk (warp w of the row
// group).  All sums are in the log2 domain (l already scaled by log2 e), so
// the mask is 2^seg.
//
//   diagonal block w:   d[c] = seg(i, 32w + c), c <= lane, a running sum
//                       grown leftwards from the diagonal (d[lane] = 0).
//   block suffix:       colS[j] = seg(end_r, j) for j in block r: the running
//                       sums of block r's last row (lane 31 of warp r).
//   block total:        tot[r] = colS[32 r] + l_{32 r}.
//   row offsets:        R[w-1] = d[0] + l_{32 w};  R[r-1] = R[r] + tot[r];
//                       R[r] = seg(i, end_r).
//   off-diagonal:       seg(i, j) = R[r] + colS[j] (j in block r < w); in the
//                       linear domain the block is the rank-one product
//                       2^R[r] * 2^colS[j].
//   chunk prefix:       p_i = R[0] + tot[0] = sum_{k=0..i} l_k.
//   chunk suffix:       s_j = seg(Q-1, j).
//
// Monotone by construction: every longer range is formed from a shorter
// range's computed value plus further terms <= 0, along one path, and fp
// rounding is monotone, so in fp32 exactly seg(i, j) <= seg(i, j+1),
// seg(i+1, j) <= seg(i, j) and seg <= 0.  (Two rows that meet at column c
// add the same terms in the same order from there on; rows of adjacent warps
// meet through tot, which is the earlier block's last-row value plus one more
// term.)  A -inf log-decay (document start) propagates as -inf, never NaN:
// nothing is subtracted.
#pragma once
#include <cuda_runtime.h>

namespace ssd {

template <int NW>
struct SegsumShared {
    alignas(16) float ell[32 * NW];    // input: log2-domain log-decays of the chunk
    float colS[32 * NW];   // seg(end of j's block, j)
    float tot[NW];         // block totals
    float rlast[NW];       // R[r] of the chunk's last row, r < NW - 1
    float tau;             // p of the chunk's last row (whole-chunk total)
};

template <int NW>
struct SegsumRow {
    float d[32];   // diagonal-block segsums, valid for c <= lane
    float R[NW];   // row offsets into earlier blocks, valid for r < w
    float p;       // chunk prefix through row i
};

__device__ __forceinline__ float ex2_approx(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Phase 1: the diagonal 1-SS block of row i; the block's last row publishes
// its column suffixes and the block total.  Needs sh.ell complete (barrier
// before), and a barrier over the row group after.
template <int NW>
__device__ __forceinline__ void segsum_phase1(SegsumShared<NW>& sh, SegsumRow<NW>& row, int w,
                                              int lane) {
    // the block's log-decays, read once (broadcast) into registers
    float e[32];
    const float4* src = reinterpret_cast<const float4*>(sh.ell + 32 * w);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 v = src[q];
        e[4 * q] = v.x;
        e[4 * q + 1] = v.y;
        e[4 * q + 2] = v.z;
        e[4 * q + 3] = v.w;
    }
    float r = 0.f;
    row.d[31] = 0.f;
#pragma unroll
    for (int c = 30; c >= 0; --c) {
        if (c < lane) r += e[c + 1];
        row.d[c] = r;
    }
    if (lane == 31) {
#pragma unroll
        for (int c = 0; c < 32; ++c) sh.colS[32 * w + c] = row.d[c];
        sh.tot[w] = row.d[0] + e[0];
    }
}

// Phase 2: row offsets R[] and the chunk prefix p; the chunk's last row
// publishes its offsets (for the chunk suffixes) and the chunk total.
// Needs the phase-1 barrier; a barrier after before chunk_suffix().
template <int NW>
__device__ __forceinline__ void segsum_phase2(SegsumShared<NW>& sh, SegsumRow<NW>& row, int w,
                                              int lane) {
    float acc = row.d[0] + sh.ell[32 * w];   // sum_{k=32w..i}
#pragma unroll
    for (int r = NW - 1; r >= 0; --r) {
        if (r < w) {
            row.R[r] = acc;
            acc = acc + sh.tot[r];
        } else {
            row.R[r] = 0.f;
        }
    }
    row.p = acc;
    if (w == NW - 1 && lane == 31) {
#pragma unroll
        for (int r = 0; r < NW; ++r) sh.rlast[r] = row.R[r];
        sh.tau = acc;
    }
}

// s_j = seg(Q-1, j) for column j (after the phase-2 barrier).
template <int NW>
__device__ __forceinline__ float segsum_chunk_suffix(const SegsumShared<NW>& sh, int j) {
    const int r = j >> 5;
    return (r == NW - 1) ? sh.colS[j] : sh.rlast[r] + sh.colS[j];
}

}  // namespace ssd
