// Backward pass of the SSD forward by recomputation (CUDA cores, fp32):
//   ssd_bwd_chunk       per (batch row, head): recompute the state entering
//                       every backward chunk, then walk the chunks backwards
//                       carrying the state's adjoint, and form every gradient
//                       of the chunk in the chunked (matrix) form
//   ssd_bwd_reduce      sums the per-head dB, dC shares over each group's
//                       heads and the per-row dA, dD shares over the batch
//
// "Parallel Scan and Hardware-Aware SSM Kernels", "Why the kernel matters more
// than the algorithm": the backward pass recomputes the states from the saved
// inputs instead of storing one per token.  Here only the state entering each
// chunk of Qb tokens is kept (P x N fp32 per chunk, in the workspace).
//
// Within a chunk (tokens i, j, t; l_t = dt_t A_h; p_i = sum_{k<=i} l_k and
// s_j = sum_{k>j} l_k within the chunk, tau = the chunk total; L_ij =
// exp(sum_{k=j+1..i} l_k) for j <= i; S_in the state entering the chunk and
// Lam the adjoint of the state leaving it), with G_ij = C_i . B_j and
// X_ij = dy_i . x_j, the reverse-mode derivatives of the recurrence are
//   v_j   = sum_{i>=j} L_ij G_ij dy_i + e^{s_j} Lam B_j       (= Lam_j B_j)
//   dx_j  = dt_j v_j + D dy_j
//   dB_j  = dt_j (sum_{i>=j} L_ij X_ij C_i + e^{s_j} Lam^T x_j)
//   dC_i  = sum_{j<=i} L_ij dt_j X_ij B_j + e^{p_i} S_in^T dy_i
//   dl_t  = <Lam_t, S_t> - dt_t x_t . v_t, where
//   <Lam_t, S_t> = sum_{j<=t<=i} L_ij dt_j X_ij G_ij + sum_{i>=t} e^{p_i} dy_i . S_in C_i
//                + sum_{j<=t} e^{s_j} dt_j x_j . Lam B_j + e^{tau} <Lam, S_in>
//   ddt_t = x_t . v_t + A dl_t,  dA += dt_t dl_t,  dD += dy_t . x_t
//   Lam  <- e^{tau} Lam + sum_i e^{p_i} dy_i C_i^T            (adjoint of S_in)
// Every sum of log-decays is a direct sum (no prefix subtraction).
//
// Packed documents are independent sequences (no state or adjoint crosses a
// boundary), so each (head, document) is its own unit, walked in chunks from
// the document's start: its first chunk enters from the document's initial
// state (or zero) and its start token's own decay applies to it; its last
// chunk leaves with the document's final-state gradient (or zero) as Lam; the
// adjoint of its first chunk's entering state is the initial state's gradient.
#include "ssd_common.cuh"
#include "ssd_kernels.h"

namespace ssd {
namespace {

constexpr int kBwdThreads = 1024;
constexpr int kBwdOwn = 8;    // state elements each thread keeps in registers (P * N <= 8192)

struct BwdSmem {
    int Qb, P, N, sx, sb, st;  // chunk, sizes, padded row strides of x, of B/S_in/Lam, of the transposes
    size_t x, dy, B, C, Sin, Lam, A1, A2, W, vx, lbx, scdy, dts, ell, ep, es, ddta, wv, uv, rv, ddv, misc, red;
    size_t xT, dyT, BT, CT, A2dtT, total;
};

// Shared-memory layout of one CTA (offsets in floats, each 16-byte aligned).
// `tiled` adds the transposed copies the register-tiled loops of the common
// head shape read as 8- and 16-byte vectors.
__host__ __device__ inline BwdSmem bwd_smem(int Qb, int P, int N, bool tiled) {
    BwdSmem s;
    s.Qb = Qb; s.P = P; s.N = N;
    s.sx = P + 1;              // odd strides: column walks hit distinct banks
    s.sb = N + 1;
    s.st = Qb + 4;
    size_t o = 0;
    auto take = [&](size_t n) { const size_t at = o; o = (o + n + 3) & ~(size_t)3; return at; };
    s.x = take((size_t)Qb * s.sx);
    s.dy = take((size_t)Qb * P);
    s.B = take((size_t)Qb * s.sb);
    s.C = take((size_t)Qb * N);
    s.Sin = take((size_t)P * s.sb);
    s.Lam = take((size_t)P * s.sb);
    s.A1 = take((size_t)Qb * Qb);       // L_ij G_ij
    s.A2 = take((size_t)Qb * Qb);       // L_ij X_ij
    s.W = take((size_t)Qb * Qb);        // L_ij dt_j X_ij G_ij
    s.vx = take((size_t)Qb * P);        // v_j[p] x_j[p]
    s.lbx = take((size_t)Qb * P);       // (Lam B_j)[p] x_j[p]
    s.scdy = take((size_t)Qb * P);      // (S_in C_i)[p] dy_i[p]
    s.dts = take(Qb);
    s.ell = take(Qb);
    s.ep = take(Qb);
    s.es = take(Qb);
    s.ddta = take(Qb);
    s.wv = take(Qb);
    s.uv = take(Qb);
    s.rv = take(Qb);
    s.ddv = take(Qb);                   // dy_t . x_t
    s.misc = take(4);                   // [0]: e^{tau} of the chunk
    s.red = take(2 * (kBwdThreads / 32));
    s.xT = s.dyT = s.BT = s.CT = s.A2dtT = 0;
    if (tiled) {
        s.xT = take((size_t)P * s.st);     // x[j][p] at [p][j]
        s.dyT = take((size_t)P * s.st);    // dy[j][p] at [p][j]
        s.BT = take((size_t)N * s.st);     // B[j][n] at [n][j]
        s.CT = take((size_t)N * s.st);     // C[j][n] at [n][j]
        s.A2dtT = take((size_t)Qb * s.st); // L_jk X_jk dt_k at [k][j]
    }
    s.total = o * sizeof(float);
    return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Inclusive prefix sum over lanes 0..lane, and inclusive suffix sum over lanes
// lane..31 (direct sums in a fixed order: no subtraction).
__device__ __forceinline__ float warp_prefix(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}
__device__ __forceinline__ float warp_suffix(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_down_sync(0xffffffffu, v, o);
        if (lane + o < 32) v += t;
    }
    return v;
}

// Block-wide sum (every thread gets the result); `red` holds one float per warp.
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kBwdThreads / 32; ++k) s += red[k];
    return s;
}

// kP, kN, kQ: compile-time P, N and chunk (0: run-time values).  The common head
// shape (64, 128, 32) runs register-tiled loops: each thread owns 8 state rows of
// one column, and the matrix products read their operands as vectors, so a shared-
// memory load feeds 2 to 4 multiply-adds instead of half of one.
template <typename T, int kP, int kN, int kQ>
__global__ void __launch_bounds__(kBwdThreads) ssd_bwd_chunk(BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    constexpr bool kT = kP == 64 && kN == 128 && kQ == 32;
    const int Qb = kQ ? kQ : a.Qb, P = kP ? kP : a.P, N = kN ? kN : a.N, H = a.H, G = a.G;
    const BwdSmem L = bwd_smem(Qb, P, N, kT);
    const int PN = P * N;
    float* xs = sm + L.x;
    float* dys = sm + L.dy;
    float* Bs = sm + L.B;
    float* Cs = sm + L.C;
    float* Sin = sm + L.Sin;
    float* Lam = sm + L.Lam;
    float* A1 = sm + L.A1;
    float* A2 = sm + L.A2;
    float* Wm = sm + L.W;
    float* vx = sm + L.vx;
    float* lbx = sm + L.lbx;
    float* scdy = sm + L.scdy;
    float* dts = sm + L.dts;
    float* ell = sm + L.ell;
    float* ep = sm + L.ep;
    float* es = sm + L.es;
    float* ddta = sm + L.ddta;
    float* wv = sm + L.wv;
    float* uv = sm + L.uv;
    float* rv = sm + L.rv;
    float* ddv = sm + L.ddv;
    float* misc = sm + L.misc;
    float* red = sm + L.red;
    float* xT = sm + L.xT;
    float* dyT = sm + L.dyT;
    float* BT = sm + L.BT;
    float* CT = sm + L.CT;
    float* A2dtT = sm + L.A2dtT;

    const int tid = threadIdx.x;
    const int64_t Lseq = a.L;
    const bool docs = a.cu != nullptr;
    // units: (batch row, head) = b * H + h, or with packed documents (head,
    // document) = h * ndocs + d (batch 1), documents being independent sequences
    const int64_t unit = blockIdx.x;
    const int h = (int)(docs ? unit / a.ndocs : unit % H);
    const int d = docs ? (int)(unit % a.ndocs) : 0;
    const int64_t b = docs ? 0 : unit / H;
    const int g = h / (H / G);
    const float Ah = a.A[h];
    const float Dh = a.D ? a.D[h] : 0.f;
    const T* x = static_cast<const T*>(a.x);
    const T* Bg = static_cast<const T*>(a.B);
    const T* Cg = static_cast<const T*>(a.C);
    const T* dy = static_cast<const T*>(a.dy);
    // the unit's tokens [T0, T1): the row, or the document (offsets clamped to the row)
    auto clamp_t = [&](int64_t v, int64_t lo) { return v < lo ? lo : (v > Lseq ? Lseq : v); };
    int64_t T0 = 0, T1 = Lseq;
    if (docs) {
        T0 = clamp_t(__ldg(a.cu + d), 0);
        T1 = clamp_t(__ldg(a.cu + d + 1), T0);
    }
    const int nchunks = (int)((T1 - T0 + Qb - 1) / Qb);
    // chunk-entry states: ceil(L / Qb) (+ ndocs with documents) slots per row or, with
    // documents, per head; a document's slots follow those of the documents before it
    const int nch_max = (int)((Lseq + Qb - 1) / Qb) + (docs ? a.ndocs : 0);
    int64_t off = 0;
    if (docs) {
        float part = 0.f;   // (chunk counts: integers, exact in fp32 below 2^24)
        for (int k = tid; k < d; k += kBwdThreads) {
            const int64_t s0 = clamp_t(__ldg(a.cu + k), 0), s1 = clamp_t(__ldg(a.cu + k + 1), s0);
            part += (float)((s1 - s0 + Qb - 1) / Qb);
        }
        off = (int64_t)block_sum(part, sm + L.red);
        if (unit == 0) check_cu_seqlens(a.cu, a.ndocs, Lseq, a.ws, tid, kBwdThreads);   // the call's offsets
        if (off + nchunks > nch_max) {
            // only offsets that break their contract (reported by the check above) get here
            if (tid == 0) {
                a.ws_dA[unit] = 0.f;
                a.ws_dD[unit] = 0.f;
            }
            return;
        }
    }
    float* ckpt = a.ws_ckpt + ((size_t)(docs ? h : unit) * nch_max + off) * PN;
    const size_t si = docs ? (size_t)d * H + h : (size_t)unit;   // state index: initial states, dfin, dinit

    // token row k of this chunk: x / dy row, B / C row (zeros past the end)
    auto xrow = [&](int64_t t) { return x + ((size_t)(b * Lseq + t) * H + h) * P; };
    auto dyrow = [&](int64_t t) { return dy + ((size_t)(b * Lseq + t) * H + h) * P; };
    auto bcoff = [&](int64_t t) { return ((size_t)(b * Lseq + t) * G + g) * N; };
    // the state elements this thread owns: (p, n) of its r-th element
    const int own_n = kT ? (tid & 127) : 0, own_p0 = kT ? (tid >> 7) * 8 : 0;
    auto own = [&](int r) -> int { return kT ? (own_p0 + r) * N + own_n : tid + kBwdThreads * r; };

    // ------------------------------------------------------------ phase 1
    // forward over the chunks: the state entering each chunk, kept in the workspace
    float S[kBwdOwn];
#pragma unroll
    for (int r = 0; r < kBwdOwn; ++r) {
        const int e = own(r);
        S[r] = (e < PN && a.init) ? a.init[si * PN + e] : 0.f;
    }
    for (int c = 0; c < nchunks; ++c) {
        const int64_t t0 = T0 + (int64_t)c * Qb;
        const int64_t t1 = (t0 + Qb < T1) ? t0 + Qb : T1;
#pragma unroll
        for (int r = 0; r < kBwdOwn; ++r) {
            const int e = own(r);
            if (e < PN) ckpt[(size_t)c * PN + e] = S[r];
        }
        __syncthreads();   // the previous chunk's tile reads are done
        for (int k = tid; k < Qb * P; k += kBwdThreads) {
            const int i = k / P, p = k - i * P;
            const float v = (t0 + i < t1) ? Elem<T>::load(xrow(t0 + i) + p) : 0.f;
            if (kT) dys[i * P + p] = v;    // x rows, 16-byte aligned (the dy buffer is free here)
            else xs[i * L.sx + p] = v;
        }
        for (int k = tid; k < Qb * N; k += kBwdThreads) {
            const int i = k / N, n = k - i * N;
            Bs[i * L.sb + n] = (t0 + i < t1) ? Elem<T>::load(Bg + bcoff(t0 + i) + n) : 0.f;
        }
        if constexpr (kT) {
            if (tid < 32) {   // warp 0, lane = token: suffix sums by shuffles
                const float d = (t0 + tid < t1) ? a.dt[(size_t)(b * Lseq + t0 + tid) * H + h] : 0.f;
                const float l = d * Ah;
                const float nxt = __shfl_down_sync(0xffffffffu, l, 1);
                const float sfx = warp_suffix(tid < 31 ? nxt : 0.f);   // s_t: the log-decays after t
                es[tid] = expf(sfx) * d;          // the weight of token t's input in the chunk's end state
                const float tau = __shfl_sync(0xffffffffu, l + sfx, 0);
                if (tid == 0) red[0] = expf(tau);
            }
        } else {
            if (tid < Qb) {
                const float d = (t0 + tid < t1) ? a.dt[(size_t)(b * Lseq + t0 + tid) * H + h] : 0.f;
                dts[tid] = d;
                ell[tid] = d * Ah;
            }
            __syncthreads();
            if (tid < Qb) {
                float s = 0.f;                          // s_t: the log-decays after t in the chunk
                for (int k = tid + 1; k < Qb; ++k) s += ell[k];
                es[tid] = expf(s) * dts[tid];           // the weight of token t's input in the chunk's end state
            }
            if (tid == 0) {
                float tau = 0.f;
                for (int k = 0; k < Qb; ++k) tau += ell[k];
                red[0] = expf(tau);
            }
        }
        __syncthreads();
        const float etau = red[0];
        if constexpr (kT) {
#pragma unroll
            for (int r = 0; r < kBwdOwn; ++r) S[r] *= etau;
#pragma unroll 4
            for (int j = 0; j < Qb; ++j) {
                const float w = es[j], bv = Bs[j * L.sb + own_n];
                const float4 x0 = *reinterpret_cast<const float4*>(dys + j * P + own_p0);
                const float4 x1 = *reinterpret_cast<const float4*>(dys + j * P + own_p0 + 4);
                S[0] = fmaf(w * x0.x, bv, S[0]);
                S[1] = fmaf(w * x0.y, bv, S[1]);
                S[2] = fmaf(w * x0.z, bv, S[2]);
                S[3] = fmaf(w * x0.w, bv, S[3]);
                S[4] = fmaf(w * x1.x, bv, S[4]);
                S[5] = fmaf(w * x1.y, bv, S[5]);
                S[6] = fmaf(w * x1.z, bv, S[6]);
                S[7] = fmaf(w * x1.w, bv, S[7]);
            }
        } else {
#pragma unroll
            for (int r = 0; r < kBwdOwn; ++r) {
                const int e = own(r);
                if (e < PN) {
                    const int p = e / N, n = e - p * N;
                    float acc = etau * S[r];
#pragma unroll 8
                    for (int j = 0; j < Qb; ++j) acc = fmaf(es[j] * xs[j * L.sx + p], Bs[j * L.sb + n], acc);
                    S[r] = acc;
                }
            }
        }
    }

    // ------------------------------------------------------------ phase 2
    // backward over the chunks, carrying Lam (the adjoint of the state leaving the chunk)
    float Lr[kBwdOwn];
#pragma unroll
    for (int r = 0; r < kBwdOwn; ++r) {
        const int e = own(r);
        Lr[r] = (e < PN && a.dfin) ? a.dfin[si * PN + e] : 0.f;   // the final state's adjoint
    }
    float dA_acc = 0.f, dD_acc = 0.f;    // thread 0's running sums
    for (int c = nchunks - 1; c >= 0; --c) {
        const int64_t t0 = T0 + (int64_t)c * Qb;
        const int64_t t1 = (t0 + Qb < T1) ? t0 + Qb : T1;
        __syncthreads();   // the previous chunk's shared-memory reads are done
        for (int k = tid; k < Qb * P; k += kBwdThreads) {
            const int i = k / P, p = k - i * P;
            const bool ok = t0 + i < t1;
            const float xv = ok ? Elem<T>::load(xrow(t0 + i) + p) : 0.f;
            const float dv = ok ? Elem<T>::load(dyrow(t0 + i) + p) : 0.f;
            xs[i * L.sx + p] = xv;
            dys[i * P + p] = dv;
            if (kT) {
                xT[p * L.st + i] = xv;
                dyT[p * L.st + i] = dv;
            }
        }
        for (int k = tid; k < Qb * N; k += kBwdThreads) {
            const int i = k / N, n = k - i * N;
            const bool ok = t0 + i < t1;
            const float bv = ok ? Elem<T>::load(Bg + bcoff(t0 + i) + n) : 0.f;
            const float cv = ok ? Elem<T>::load(Cg + bcoff(t0 + i) + n) : 0.f;
            Bs[i * L.sb + n] = bv;
            Cs[i * N + n] = cv;
            if (kT) {
                BT[n * L.st + i] = bv;
                CT[n * L.st + i] = cv;
            }
        }
        float kdot = 0.f;   // this thread's share of <Lam, S_in>
#pragma unroll
        for (int r = 0; r < kBwdOwn; ++r) {
            const int e = own(r);
            if (e < PN) {
                const int p = e / N, n = e - p * N;
                const float sv = ckpt[(size_t)c * PN + e];
                Sin[p * L.sb + n] = sv;
                Lam[p * L.sb + n] = Lr[r];
                kdot = fmaf(Lr[r], sv, kdot);
            }
        }
        if (tid < Qb) {
            const float d = (t0 + tid < t1) ? a.dt[(size_t)(b * Lseq + t0 + tid) * H + h] : 0.f;
            dts[tid] = d;
            ell[tid] = d * Ah;
        }
        const float K = block_sum(kdot, red);   // (contains a barrier: the tiles are visible)
        if constexpr (kT) {
            if (tid < 32) {   // warp 0, lane = token: prefix and suffix sums by shuffles
                const float l = ell[tid];
                const float pfx = warp_prefix(l);                                  // p_t
                const float nxt = __shfl_down_sync(0xffffffffu, l, 1);
                const float sfx = warp_suffix(tid < 31 ? nxt : 0.f);               // s_t
                ep[tid] = expf(pfx);
                es[tid] = expf(sfx);
                const float tau = __shfl_sync(0xffffffffu, l + sfx, 0);
                if (tid == 0) misc[0] = expf(tau);
            }
        } else {
            if (tid < Qb) {
                float pfx = 0.f, sfx = 0.f;
                for (int k = 0; k <= tid; ++k) pfx += ell[k];
                for (int k = tid + 1; k < Qb; ++k) sfx += ell[k];
                ep[tid] = expf(pfx);
                es[tid] = expf(sfx);
            }
            if (tid == 0) {
                float tau = 0.f;
                for (int k = 0; k < Qb; ++k) tau += ell[k];
                misc[0] = expf(tau);
            }
        }
        // pair quantities (i, j): L_ij by a direct sum, G_ij, X_ij
        for (int q = tid; q < Qb * Qb; q += kBwdThreads) {
            const int i = q / Qb, j = q - i * Qb;
            float a1 = 0.f, a2 = 0.f, w = 0.f;
            float seg = 0.f;
            if constexpr (kT) {   // a warp holds row i, lane = j: seg = sum_{k=j+1..i} l_k by shuffles
                seg = warp_suffix((j + 1 <= i) ? ell[j + 1] : 0.f);
            } else {
                for (int k = j + 1; k <= i; ++k) seg += ell[k];
            }
            if (j <= i) {
                const float Lij = expf(seg);
                float gij = 0.f, xij = 0.f;
                if constexpr (kT) {   // row i as broadcast vectors, column j from the transposes
#pragma unroll 4
                    for (int n = 0; n < 128; n += 4) {
                        const float4 cc = *reinterpret_cast<const float4*>(Cs + i * 128 + n);
                        gij = fmaf(cc.x, BT[(n + 0) * L.st + j], gij);
                        gij = fmaf(cc.y, BT[(n + 1) * L.st + j], gij);
                        gij = fmaf(cc.z, BT[(n + 2) * L.st + j], gij);
                        gij = fmaf(cc.w, BT[(n + 3) * L.st + j], gij);
                    }
#pragma unroll 4
                    for (int p = 0; p < 64; p += 4) {
                        const float4 dd = *reinterpret_cast<const float4*>(dys + i * 64 + p);
                        xij = fmaf(dd.x, xT[(p + 0) * L.st + j], xij);
                        xij = fmaf(dd.y, xT[(p + 1) * L.st + j], xij);
                        xij = fmaf(dd.z, xT[(p + 2) * L.st + j], xij);
                        xij = fmaf(dd.w, xT[(p + 3) * L.st + j], xij);
                    }
                } else {
#pragma unroll 8
                    for (int n = 0; n < N; ++n) gij = fmaf(Cs[i * N + n], Bs[j * L.sb + n], gij);
#pragma unroll 8
                    for (int p = 0; p < P; ++p) xij = fmaf(dys[i * P + p], xs[j * L.sx + p], xij);
                }
                a1 = Lij * gij;
                a2 = Lij * xij;
                w = a1 * dts[j] * xij;
            }
            A1[q] = a1;
            A2[q] = a2;
            Wm[q] = w;
            if (kT) A2dtT[j * L.st + i] = a2 * dts[j];
        }
        __syncthreads();
        const float etau = misc[0];
        if constexpr (kT) {
            // dx and the per-token dot products of ddt.  Threads 0-511: Lam B_j and v_j for
            // (p, rows j0 .. j0 + 3); threads 512-1023: S_in C_j for the same tiles.
            {
                const int half = tid >> 9, tt = tid & 511;
                const int p = tt & 63, j0 = (tt >> 6) * 4;
                const float* M = half ? Sin : Lam;
                const float* V = half ? CT : BT;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                for (int n = 0; n < 128; ++n) {
                    const float m = M[p * L.sb + n];
                    const float4 vv = *reinterpret_cast<const float4*>(V + n * L.st + j0);
                    acc[0] = fmaf(m, vv.x, acc[0]);
                    acc[1] = fmaf(m, vv.y, acc[1]);
                    acc[2] = fmaf(m, vv.z, acc[2]);
                    acc[3] = fmaf(m, vv.w, acc[3]);
                }
                if (half == 0) {
                    float v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) v[u] = es[j0 + u] * acc[u];
#pragma unroll 4
                    for (int i = j0; i < 32; ++i) {
                        const float4 aa = *reinterpret_cast<const float4*>(A1 + i * 32 + j0);   // 0 where j > i
                        const float d = dys[i * 64 + p];
                        v[0] = fmaf(aa.x, d, v[0]);
                        v[1] = fmaf(aa.y, d, v[1]);
                        v[2] = fmaf(aa.z, d, v[2]);
                        v[3] = fmaf(aa.w, d, v[3]);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int j = j0 + u, q = j * 64 + p;
                        const float xv = xs[j * L.sx + p], dv = dys[j * 64 + p];
                        vx[q] = v[u] * xv;
                        lbx[q] = acc[u] * xv;
                        if (t0 + j < t1)
                            Elem<T>::store(static_cast<T*>(a.dx) + ((size_t)(b * Lseq + t0 + j) * H + h) * 64 + p,
                                           fmaf(dts[j], v[u], Dh * dv));
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int j = j0 + u;
                        scdy[j * 64 + p] = acc[u] * dys[j * 64 + p];
                    }
                }
            }
            // this head's shares of dB (threads 0-511) and dC (threads 512-1023):
            // thread = (n, eight rows j0 .. j0 + 7)
            {
                const int half = tid >> 9, tt = tid & 511;
                const int n = tt & 127, j0 = (tt >> 7) * 8;
                const float* M = half ? Sin : Lam;
                const float* V = half ? dyT : xT;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int p = 0; p < 64; ++p) {
                    const float m = M[p * L.sb + n];
                    const float4 v0 = *reinterpret_cast<const float4*>(V + p * L.st + j0);
                    const float4 v1 = *reinterpret_cast<const float4*>(V + p * L.st + j0 + 4);
                    acc[0] = fmaf(m, v0.x, acc[0]);
                    acc[1] = fmaf(m, v0.y, acc[1]);
                    acc[2] = fmaf(m, v0.z, acc[2]);
                    acc[3] = fmaf(m, v0.w, acc[3]);
                    acc[4] = fmaf(m, v1.x, acc[4]);
                    acc[5] = fmaf(m, v1.y, acc[5]);
                    acc[6] = fmaf(m, v1.z, acc[6]);
                    acc[7] = fmaf(m, v1.w, acc[7]);
                }
                float r[8];
                if (half == 0) {   // dB_j = dt_j (e^{s_j} Lam^T x_j + sum_{i>=j} L_ij X_ij C_i)
#pragma unroll
                    for (int u = 0; u < 8; ++u) r[u] = es[j0 + u] * acc[u];
#pragma unroll 4
                    for (int i = j0; i < 32; ++i) {   // A2[i][j] = 0 where j > i
                        const float4 a0 = *reinterpret_cast<const float4*>(A2 + i * 32 + j0);
                        const float4 a1 = *reinterpret_cast<const float4*>(A2 + i * 32 + j0 + 4);
                        const float cv = Cs[i * 128 + n];
                        r[0] = fmaf(a0.x, cv, r[0]);
                        r[1] = fmaf(a0.y, cv, r[1]);
                        r[2] = fmaf(a0.z, cv, r[2]);
                        r[3] = fmaf(a0.w, cv, r[3]);
                        r[4] = fmaf(a1.x, cv, r[4]);
                        r[5] = fmaf(a1.y, cv, r[5]);
                        r[6] = fmaf(a1.z, cv, r[6]);
                        r[7] = fmaf(a1.w, cv, r[7]);
                    }
                } else {           // dC_j = e^{p_j} S_in^T dy_j + sum_{k<=j} L_jk dt_k X_jk B_k
#pragma unroll
                    for (int u = 0; u < 8; ++u) r[u] = ep[j0 + u] * acc[u];
#pragma unroll 4
                    for (int k = 0; k < j0 + 8; ++k) {   // A2[j][k] = 0 where k > j
                        const float4 a0 = *reinterpret_cast<const float4*>(A2dtT + k * L.st + j0);
                        const float4 a1 = *reinterpret_cast<const float4*>(A2dtT + k * L.st + j0 + 4);
                        const float bv = Bs[k * L.sb + n];
                        r[0] = fmaf(a0.x, bv, r[0]);
                        r[1] = fmaf(a0.y, bv, r[1]);
                        r[2] = fmaf(a0.z, bv, r[2]);
                        r[3] = fmaf(a0.w, bv, r[3]);
                        r[4] = fmaf(a1.x, bv, r[4]);
                        r[5] = fmaf(a1.y, bv, r[5]);
                        r[6] = fmaf(a1.z, bv, r[6]);
                        r[7] = fmaf(a1.w, bv, r[7]);
                    }
                }
                float* out = half ? a.ws_dC : a.ws_dB;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + u;
                    if (t0 + j < t1)
                        out[((size_t)(b * Lseq + t0 + j) * H + h) * 128 + n] = half ? r[u] : dts[j] * r[u];
                }
            }
        } else {
            // dx, and the per-token dot products of ddt
            for (int q = tid; q < Qb * P; q += kBwdThreads) {
                const int j = q / P, p = q - j * P;
                float lb = 0.f;
#pragma unroll 8
                for (int n = 0; n < N; ++n) lb = fmaf(Lam[p * L.sb + n], Bs[j * L.sb + n], lb);
                float v = es[j] * lb;
#pragma unroll 8
                for (int i = j; i < Qb; ++i) v = fmaf(A1[i * Qb + j], dys[i * P + p], v);
                const float xv = xs[j * L.sx + p];
                vx[q] = v * xv;
                lbx[q] = lb * xv;
                float sc = 0.f;   // (S_in C_j)[p], for the row j as an output row
#pragma unroll 8
                for (int n = 0; n < N; ++n) sc = fmaf(Sin[p * L.sb + n], Cs[j * N + n], sc);
                scdy[q] = sc * dys[j * P + p];
                if (t0 + j < t1)
                    Elem<T>::store(static_cast<T*>(a.dx) + ((size_t)(b * Lseq + t0 + j) * H + h) * P + p,
                                   fmaf(dts[j], v, Dh * dys[j * P + p]));
            }
            // this head's shares of dB and dC
            for (int q = tid; q < Qb * N; q += kBwdThreads) {
                const int j = q / N, n = q - j * N;
                if (t0 + j >= t1) continue;
                float lx = 0.f, sd = 0.f;
#pragma unroll 8
                for (int p = 0; p < P; ++p) {
                    lx = fmaf(Lam[p * L.sb + n], xs[j * L.sx + p], lx);
                    sd = fmaf(Sin[p * L.sb + n], dys[j * P + p], sd);
                }
                float db = es[j] * lx;
#pragma unroll 8
                for (int i = j; i < Qb; ++i) db = fmaf(A2[i * Qb + j], Cs[i * N + n], db);
                float dc = ep[j] * sd;
#pragma unroll 8
                for (int k = 0; k <= j; ++k) dc = fmaf(A2[j * Qb + k] * dts[k], Bs[k * L.sb + n], dc);
                const size_t o = ((size_t)(b * Lseq + t0 + j) * H + h) * N + n;
                a.ws_dB[o] = dts[j] * db;
                a.ws_dC[o] = dc;
            }
        }
        __syncthreads();
        // per-token reductions (warp w takes tokens w, w + 32, ...)
        {
            const int w = tid >> 5, lane = tid & 31;
            for (int t = w; t < Qb; t += kBwdThreads / 32) {
                float s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f, s5 = 0.f;
                for (int p = lane; p < P; p += 32) {
                    s1 += vx[t * P + p];
                    s2 += lbx[t * P + p];
                    s3 += scdy[t * P + p];
                    s5 = fmaf(dys[t * P + p], xs[t * L.sx + p], s5);
                }
                for (int i = t + lane; i < Qb; i += 32)
                    for (int j = 0; j <= t; ++j) s4 += Wm[i * Qb + j];
                s1 = warp_sum(s1);
                s2 = warp_sum(s2);
                s3 = warp_sum(s3);
                s4 = warp_sum(s4);
                s5 = warp_sum(s5);
                if (lane == 0) {
                    ddv[t] = s5;
                    ddta[t] = s1;
                    wv[t] = es[t] * dts[t] * s2;
                    uv[t] = ep[t] * s3;
                    rv[t] = s4;
                }
            }
        }
        __syncthreads();
        if constexpr (kT) {
            if (tid < 32) {   // warp 0, lane = token
                const int t = tid;
                const float U = warp_suffix(uv[t]), V = warp_prefix(wv[t]);
                const float dl = rv[t] + U + V + etau * K - dts[t] * ddta[t];
                if (t0 + t < t1) a.ddt[(size_t)(b * Lseq + t0 + t) * H + h] = fmaf(Ah, dl, ddta[t]);
                const float da = warp_sum(dts[t] * dl), dd = warp_sum(ddv[t]);
                dA_acc += da;
                dD_acc += dd;
            }
        } else {
            if (tid < Qb) {
                const int t = tid;
                float U = 0.f, V = 0.f;
                for (int i = t; i < Qb; ++i) U += uv[i];
                for (int j = 0; j <= t; ++j) V += wv[j];
                const float dl = rv[t] + U + V + etau * K - dts[t] * ddta[t];
                if (t0 + t < t1) a.ddt[(size_t)(b * Lseq + t0 + t) * H + h] = fmaf(Ah, dl, ddta[t]);
                // thread 0 sums these in token order below
                ddta[t] = dts[t] * dl;
            }
            __syncthreads();
            if (tid == 0) {
                for (int t = 0; t < Qb; ++t) {
                    dA_acc += ddta[t];
                    dD_acc += ddv[t];
                }
            }
        }
        // Lam becomes the adjoint of the state entering this chunk
        if constexpr (kT) {
#pragma unroll
            for (int r = 0; r < kBwdOwn; ++r) Lr[r] *= etau;
#pragma unroll 4
            for (int i = 0; i < 32; ++i) {
                const float w = ep[i], cv = Cs[i * 128 + own_n];
                const float4 d0 = *reinterpret_cast<const float4*>(dys + i * 64 + own_p0);
                const float4 d1 = *reinterpret_cast<const float4*>(dys + i * 64 + own_p0 + 4);
                Lr[0] = fmaf(w * d0.x, cv, Lr[0]);
                Lr[1] = fmaf(w * d0.y, cv, Lr[1]);
                Lr[2] = fmaf(w * d0.z, cv, Lr[2]);
                Lr[3] = fmaf(w * d0.w, cv, Lr[3]);
                Lr[4] = fmaf(w * d1.x, cv, Lr[4]);
                Lr[5] = fmaf(w * d1.y, cv, Lr[5]);
                Lr[6] = fmaf(w * d1.z, cv, Lr[6]);
                Lr[7] = fmaf(w * d1.w, cv, Lr[7]);
            }
        } else {
#pragma unroll
            for (int r = 0; r < kBwdOwn; ++r) {
                const int e = own(r);
                if (e < PN) {
                    const int p = e / N, n = e - p * N;
                    float acc = etau * Lr[r];
#pragma unroll 8
                    for (int i = 0; i < Qb; ++i) acc = fmaf(ep[i] * dys[i * P + p], Cs[i * N + n], acc);
                    Lr[r] = acc;
                }
            }
        }
    }
    // Lr is the adjoint of the state entering the unit: the initial state's gradient
    if (a.dinit) {
#pragma unroll
        for (int r = 0; r < kBwdOwn; ++r) {
            const int e = own(r);
            if (e < PN) a.dinit[si * PN + e] = Lr[r];
        }
    }
    if (tid == 0) {
        a.ws_dA[unit] = dA_acc;
        a.ws_dD[unit] = dD_acc;
    }
}

// dB, dC (batch, L, G, N) = sums over each group's heads of the per-head shares
// (fp32, or bf16 from the tensor-core backward), in fp32; dA, dD (H) = sums over
// the batch rows.  Fixed summation order.
template <typename T, typename S>
__global__ void __launch_bounds__(256) ssd_bwd_reduce(BwdArgs a) {
    const S* shB = reinterpret_cast<const S*>(a.ws_dB);
    const S* shC = reinterpret_cast<const S*>(a.ws_dC);
    const int64_t total = a.batch * a.L * a.G * a.N;
    const int hpg = a.H / a.G;
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < total; k += (int64_t)gridDim.x * blockDim.x) {
        const int n = (int)(k % a.N);
        const int64_t rest = k / a.N;
        const int g = (int)(rest % a.G);
        const int64_t bt = rest / a.G;   // b * L + t
        float sb = 0.f, sc = 0.f;
        for (int hh = 0; hh < hpg; ++hh) {
            const size_t o = ((size_t)bt * a.H + g * hpg + hh) * a.N + n;
            sb += Elem<S>::load(shB + o);
            sc += Elem<S>::load(shC + o);
        }
        Elem<T>::store(static_cast<T*>(a.dB) + k, sb);
        Elem<T>::store(static_cast<T*>(a.dC) + k, sc);
    }
    if (blockIdx.x == 0) {
        for (int h = threadIdx.x; h < a.H; h += blockDim.x) {
            float sa = 0.f, sd = 0.f;
            const int ns = a.nsplit > 0 ? a.nsplit : 1;   // (one share per unit: row, head, split)
            for (int64_t b = 0; b < a.batch; ++b)
                for (int sp = 0; sp < ns; ++sp) {
                    sa += a.ws_dA[(b * a.H + h) * ns + sp];
                    sd += a.ws_dD[(b * a.H + h) * ns + sp];
                }
            a.dA[h] = sa;
            if (a.dD) a.dD[h] = sd;
        }
    }
}

// The same sums over 16-byte vectors of the shares (8 bf16 or 4 fp32 elements per
// thread, N a multiple of that), the heads of a group four loads at a time: enough
// bytes in flight for the share stream, which the scalar form left at about 0.6 of
// the HBM bandwidth.  Every element still sums its heads in order, so the results
// are the scalar form's, bit for bit.
template <typename S>
__device__ __forceinline__ void add_vec(float* acc, uint4 v) {
    if constexpr (sizeof(S) == 2) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc[2 * q] += __uint_as_float(w[q] << 16);
            acc[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
        }
    } else {
        acc[0] += __uint_as_float(v.x);
        acc[1] += __uint_as_float(v.y);
        acc[2] += __uint_as_float(v.z);
        acc[3] += __uint_as_float(v.w);
    }
}

template <typename T, int V>
__device__ __forceinline__ void store_vec(T* dst, const float* v) {
#pragma unroll
    for (int e = 0; e < V; ++e) Elem<T>::store(dst + e, v[e]);
}

template <typename T, typename S>
__global__ void __launch_bounds__(256) ssd_bwd_reduce_vec(BwdArgs a) {
    constexpr int V = 16 / (int)sizeof(S);
    const S* shB = reinterpret_cast<const S*>(a.ws_dB);
    const S* shC = reinterpret_cast<const S*>(a.ws_dC);
    const int NV = a.N / V;
    const int64_t total = a.batch * a.L * a.G * NV;
    const int hpg = a.H / a.G;
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < total; k += (int64_t)gridDim.x * blockDim.x) {
        const int nv = (int)(k % NV);
        const int64_t rest = k / NV;
        const int g = (int)(rest % a.G);
        const int64_t bt = rest / a.G;   // b * L + t
        const size_t o0 = ((size_t)bt * a.H + (size_t)g * hpg) * a.N + (size_t)nv * V;
        float sb[V], sc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) sb[e] = sc[e] = 0.f;
#pragma unroll 4
        for (int hh = 0; hh < hpg; ++hh) {
            const uint4 vb = __ldcs(reinterpret_cast<const uint4*>(shB + o0 + (size_t)hh * a.N));
            const uint4 vc = __ldcs(reinterpret_cast<const uint4*>(shC + o0 + (size_t)hh * a.N));
            add_vec<S>(sb, vb);
            add_vec<S>(sc, vc);
        }
        const size_t oo = ((size_t)bt * a.G + g) * a.N + (size_t)nv * V;
        store_vec<T, V>(static_cast<T*>(a.dB) + oo, sb);
        store_vec<T, V>(static_cast<T*>(a.dC) + oo, sc);
    }
    if (blockIdx.x == 0) {
        for (int h = threadIdx.x; h < a.H; h += blockDim.x) {
            float sa = 0.f, sd = 0.f;
            const int ns = a.nsplit > 0 ? a.nsplit : 1;   // (one share per unit: row, head, split)
            for (int64_t b = 0; b < a.batch; ++b)
                for (int sp = 0; sp < ns; ++sp) {
                    sa += a.ws_dA[(b * a.H + h) * ns + sp];
                    sd += a.ws_dD[(b * a.H + h) * ns + sp];
                }
            a.dA[h] = sa;
            if (a.dD) a.dD[h] = sd;
        }
    }
}

}  // namespace

static bool bwd_tiled(int Qb, int P, int N) { return P == 64 && N == 128 && Qb == 32; }

size_t bwd_smem_bytes(int Qb, int P, int N) { return bwd_smem(Qb, P, N, bwd_tiled(Qb, P, N)).total; }

int bwd_chunk(int P, int N, size_t smem_limit) {
    if (P * N > kBwdThreads * kBwdOwn) return 0;
    if (P == 64 && N == 128 && bwd_smem_bytes(32, P, N) <= smem_limit) return 32;   // the tiled loops
    for (int Qb = 64; Qb >= 8; Qb >>= 1)
        if (bwd_smem_bytes(Qb, P, N) <= smem_limit) return Qb;
    return 0;
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t st) {
    const size_t smem = bwd_smem_bytes(a.Qb, a.P, a.N);
    const bool mamba_shape = bwd_tiled(a.Qb, a.P, a.N);
    auto k1 = a.dtype == SSD_BF16 ? (mamba_shape ? ssd_bwd_chunk<__nv_bfloat16, 64, 128, 32>
                                                 : ssd_bwd_chunk<__nv_bfloat16, 0, 0, 0>)
                                  : (mamba_shape ? ssd_bwd_chunk<float, 64, 128, 32> : ssd_bwd_chunk<float, 0, 0, 0>);
    cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // (units: rows x heads, or heads x documents)
    k1<<<(unsigned)(a.cu ? (int64_t)a.H * a.ndocs : a.batch * a.H), kBwdThreads, smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_bwd_reduce(a, st);
}

cudaError_t launch_bwd_reduce(const BwdArgs& a, cudaStream_t st) {
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int64_t total = a.batch * a.L * a.G * a.N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)nsm * 8) blocks = (int64_t)nsm * 8;
    if (blocks < 1) blocks = 1;
    // 16-byte vectors of the shares when N holds whole ones (the shares start on
    // 256-byte boundaries and dB, dC on 16-byte ones)
    const int V = a.shares_bf16 ? 8 : 4;
    if (a.N % V == 0) {
        const int64_t nvec = a.batch * a.L * a.G * (a.N / V);
        const int64_t vblocks = (nvec + 255) / 256 < 1 ? 1 : (nvec + 255) / 256;
        auto kv = a.dtype == SSD_BF16 ? (a.shares_bf16 ? ssd_bwd_reduce_vec<__nv_bfloat16, __nv_bfloat16>
                                                       : ssd_bwd_reduce_vec<__nv_bfloat16, float>)
                                      : ssd_bwd_reduce_vec<float, float>;
        kv<<<(unsigned)vblocks, 256, 0, st>>>(a);
        return cudaGetLastError();
    }
    auto k2 = a.dtype == SSD_BF16
                  ? (a.shares_bf16 ? ssd_bwd_reduce<__nv_bfloat16, __nv_bfloat16> : ssd_bwd_reduce<__nv_bfloat16, float>)
                  : ssd_bwd_reduce<float, float>;
    k2<<<(unsigned)blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ssd
