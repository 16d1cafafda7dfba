// Hierarchy-aware segsum for one chunk of Q = 32 * NW tokens, in two forms
// that share one hierarchy:
//
//   log domain     seg(i, j) = sum_{k=j+1..i} l_k          (SIMT kernel: exp2 of seg)
//   linear domain  L(i, j)   = prod_{k=j+1..i} a_k, a_k = 2^{l_k}
//                                                            (tensor-core kernel: L itself)
//
// "GPU Hierarchy Meets Structured Matrices" (abstract): the 1-semiseparable
// decay mask is split into 1-SS diagonal blocks (one per warp) and rank-one
// off-diagonal blocks, built from per-warp scans and cross-warp aggregation,
// with no prefix subtraction.  l is already scaled by log2 e, so the mask is
// 2^seg.  One thread owns one row i = 32 w + lane of the chunk (warp w of the
// row group).  In the log domain "+" combines ranges; in the linear domain
// "*" does, and each a_k costs one exp2 per token instead of one per entry.
//
//   diagonal block w:   d[c] = range (32w + c, i], c <= lane, a running
//                       combination grown leftwards from the diagonal
//                       (d[lane] = identity).
//   block suffix:       col[j] = range (j, end_r] for j in block r: the running
//                       values of block r's last row (lane 31 of warp r).
//   block total:        tot[r] = col[32 r] (+) l_{32 r}.
//   row offsets:        R[w-1] = d[0] (+) l_{32 w};  R[r-1] = R[r] (+) tot[r];
//                       R[r] = range (end_r, i].
//   off-diagonal:       entry (i, j) = R[r] (+) col[j] for j in block r < w:
//                       in the linear domain the block is the rank-one product
//                       of a row factor and a column factor.
//   chunk prefix:       p_i = R[0] (+) tot[0] = range [0, i].
//   chunk suffix:       s_j = range (j, Q-1] = rlast[r] (+) col[j].
//
// Monotone by construction, in either domain.  Every operand combined into a
// range is <= 0 (log) or in [0, 1] (linear), and rounding is monotone, so a
// combination never moves a value up.  Row order, seg(i, j) <= seg(i, j+1):
// each longer range is formed from the shorter one's computed value (within a
// block, across a block edge through R, and across rank-one blocks because
// R[r-1] = R[r] (+) tot[r] with tot[r] <= identity).  Column order,
// seg(i+1, j) <= seg(i, j): rows i and i+1 start one step apart and then
// combine the same terms in the same order, and combining the same term with
// two ordered values keeps them ordered; rows of adjacent warps meet through
// tot, which is bit for bit the earlier block's last-row value combined with
// one more term, exactly what the later row's offset is built from.  A -inf
// log-decay (document start) gives -inf (log) or an exact 0 (linear), never
// NaN: nothing is subtracted.
#pragma once
#include <cuda_runtime.h>

namespace ssd {

__device__ __forceinline__ float ex2_approx(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// ============================================================== log domain

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
    // the running sum takes -0 (an exact no-op) instead of a term past the
    // diagonal, so its dependent chain is one add per column
    float r = 0.f;
    row.d[31] = 0.f;
#pragma unroll
    for (int c = 30; c >= 0; --c) {
        r += (c < lane) ? e[c + 1] : -0.f;
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

// seg(i, j) of the calling thread's row i = 32 w + lane, any column j
// (compile-time block index r and column c within it; -inf above the diagonal).
template <int NW>
__device__ __forceinline__ float segsum_entry(const SegsumShared<NW>& sh, const SegsumRow<NW>& row, int w,
                                              int lane, int r, int c) {
    if (r < w) return row.R[r] + sh.colS[32 * r + c];
    if (r == w) return (c <= lane) ? row.d[c] : -INFINITY;
    return -INFINITY;
}

// =========================================================== linear domain

template <int NW>
struct alignas(16) SegsumLinShared {
    alignas(16) float a[32 * NW];      // input: a_k = 2^{l_k} (exactly 0 at a document start)
    alignas(16) float colL[32 * NW];   // L(end of j's block, j)
    float totL[NW];                    // block totals L(end_r, start_r - 1) = prod over block r
    float rlastL[NW];                  // row factors of the chunk's last row, r < NW - 1
    float tauL;                        // 2^{whole-chunk total}
};

template <int NW>
struct SegsumLinRow {
    float wl[32];                      // L(i, 32 w + c) for c <= lane, 0 above the diagonal
    float rf[NW > 1 ? NW - 1 : 1];     // L(i, end of block r) for r < w: the rank-one row factors
    float pe;                          // 2^{p_i}: prod_{k=0..i} a_k
};

// Phase 1: the diagonal 1-SS block, products grown leftwards from the
// diagonal; the block's last row publishes its column factors and the block
// total.  Needs sh.a complete (barrier before), a barrier after.  K
// independent chunks (of different heads) at once: their product chains
// interleave, each one multiply per column.  publish = false: the row's
// factors only (a second thread of the same row; the other publishes).
template <int NW, int K>
__device__ __forceinline__ void segsum_lin_phase1_k(SegsumLinShared<NW>* sh, SegsumLinRow<NW>* row, int w,
                                                    int lane, bool publish = true) {
    float e[K][32];
#pragma unroll
    for (int h = 0; h < K; ++h) {
        const float4* src = reinterpret_cast<const float4*>(sh[h].a + 32 * w);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 v = src[q];
            e[h][4 * q] = v.x;
            e[h][4 * q + 1] = v.y;
            e[h][4 * q + 2] = v.z;
            e[h][4 * q + 3] = v.w;
        }
    }
    // the running product takes 1 (an exact no-op) instead of a factor past the
    // diagonal, so its dependent chain is one multiply per column
    float r[K];
#pragma unroll
    for (int h = 0; h < K; ++h) r[h] = 1.f;
#pragma unroll
    for (int c = 31; c >= 0; --c) {
#pragma unroll
        for (int h = 0; h < K; ++h) {
            r[h] *= (c < lane) ? e[h][c + 1] : 1.f;
            row[h].wl[c] = (c <= lane) ? r[h] : 0.f;
        }
    }
    if (publish && lane == 31) {
#pragma unroll
        for (int h = 0; h < K; ++h) {
            float4* dst = reinterpret_cast<float4*>(sh[h].colL + 32 * w);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(row[h].wl[4 * q], row[h].wl[4 * q + 1], row[h].wl[4 * q + 2],
                                     row[h].wl[4 * q + 3]);
            sh[h].totL[w] = row[h].wl[0] * e[h][0];
        }
    }
}

template <int NW>
__device__ __forceinline__ void segsum_lin_phase1(SegsumLinShared<NW>& sh, SegsumLinRow<NW>& row, int w,
                                                  int lane, bool publish = true) {
    segsum_lin_phase1_k<NW, 1>(&sh, &row, w, lane, publish);
}

// Phase 2: the rank-one row factors and the chunk prefix; the chunk's last
// row publishes its factors (for the chunk suffixes) and the chunk total.
// Needs the phase-1 barrier; a barrier after before segsum_lin_suffix().
template <int NW>
__device__ __forceinline__ void segsum_lin_phase2(SegsumLinShared<NW>& sh, SegsumLinRow<NW>& row, int w,
                                                  int lane, bool publish = true) {
    float acc = row.wl[0] * sh.a[32 * w];   // prod_{k=32w..i} a_k
#pragma unroll
    for (int r = NW - 2; r >= 0; --r) {
        row.rf[r] = (r < w) ? acc : 0.f;
        acc *= (r < w) ? sh.totL[r] : 1.f;   // 1: an exact no-op past the row's own block
    }
    row.pe = acc;
    if (publish && w == NW - 1 && lane == 31) {
#pragma unroll
        for (int r = 0; r < NW - 1; ++r) sh.rlastL[r] = row.rf[r];
        sh.tauL = acc;
    }
}

// 2^{s_j} = L(Q-1, j) for column j (after the phase-2 barrier).
template <int NW>
__device__ __forceinline__ float segsum_lin_suffix(const SegsumLinShared<NW>& sh, int j) {
    const int r = j >> 5;
    return (r == NW - 1) ? sh.colL[j] : sh.rlastL[r] * sh.colL[j];
}

// L(i, j) of the calling thread's row: block r, column c within it.  The
// kernels apply the same factors to G (row factor) and dt (column factor)
// instead of forming L; this is the mask those factors make.
template <int NW>
__device__ __forceinline__ float segsum_lin_entry(const SegsumLinShared<NW>& sh, const SegsumLinRow<NW>& row,
                                                  int w, int r, int c) {
    if (r < w) return row.rf[r] * sh.colL[32 * r + c];
    if (r == w) return row.wl[c];
    return 0.f;
}

}  // namespace ssd
