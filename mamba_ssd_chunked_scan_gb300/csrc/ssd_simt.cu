// SIMT (CUDA-core, fp32) kernels of libssd:
//   ssd_chunk_simt      the chunked SSD forward for any supported shape and
//                       dtype, fp32 arithmetic throughout (the fp32 path)
//   ssd_split_scan      composes split aggregates into incoming states
//   ssd_segsum_dump_k   both forms of the hierarchy-aware segsum routine on
//                       their own (the log-domain form this file's forward
//                       kernel uses, the linear-domain form of ssd_tc.cu)
//
// The chunked form follows "State Space Duality and Mamba-2", "The SSD Block
// Decomposition Algorithm": per chunk the diagonal block ((C B^T) o L) X, the
// chunk state summary, the inter-chunk state passing, and the chunk state
// projection C * state (with the decay from the chunk start to the row, which
// the 1-SS matrix entry M_ij = C_i^T (prod_{k=j+1..i} a_k) B_j implies).
// Packed documents cut a chunk into segments that never mix: each segment
// starts from the carried state (when it continues a document) or from the
// document's initial state.
#include "ssd_common.cuh"
#include "segsum.cuh"
#include "ssd_kernels.h"

namespace ssd {

// Document of token t in a packed row: the last d with cu[d] <= t.
__device__ __forceinline__ int find_doc(const int32_t* cu, int ndocs, int64_t t) {
    int lo = 0, hi = ndocs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The segsum scratch (SegsumShared<4> at most) sits at the start of the
// dynamic shared memory, ahead of the tiles.
constexpr size_t kSegsumBytes = (sizeof(SegsumShared<4>) + 15) / 16 * 16;

size_t simt_smem_bytes(int Q, int P, int N) {
    size_t floats = (size_t)Q * P + 2 * (size_t)Q * N + (size_t)Q * Q + (size_t)P * N + 6 * (size_t)Q;
    size_t ints = 3 * (size_t)Q;
    return kSegsumBytes + floats * 4 + ints * 4 + 64;
}

// Chunk Q = 32 NW.  The decay mask comes from the hierarchy-aware segsum in
// the log domain (segsum.cuh): one thread per chunk row, exp2 of each entry.
// A document that starts at row st > 0 of the chunk gets a -inf log-decay
// there, which zeroes every mask entry that would cross into it; the decay of
// its own initial state (which the document's first token does apply) is
// 2^{seg(i, st) + l_st}.
template <typename T, int NW>
__global__ void __launch_bounds__(256) ssd_chunk_simt(FwdArgs a) {
    constexpr int Q = 32 * NW;
    extern __shared__ float4 smem4[];
    SegsumShared<NW>& sg = *reinterpret_cast<SegsumShared<NW>*>(smem4);
    float* smem = reinterpret_cast<float*>(reinterpret_cast<char*>(smem4) + kSegsumBytes);
    const int P = a.P, N = a.N, H = a.H, G = a.G;
    const int64_t L = a.L;
    float* xs = smem;                       // [Q][P]
    float* Bs = xs + Q * P;                 // [Q][N]
    float* Cs = Bs + Q * N;                 // [Q][N]
    float* M = Cs + Q * N;                  // [Q][Q]
    float* S = M + Q * Q;                   // [P][N] carried state
    float* lreal = S + P * N;               // [Q] log2-decays (no document-start -inf)
    float* dtv = lreal + Q;                 // [Q]
    float* pexp = dtv + Q;                  // [Q] decay of row i's segment-entry state
    float* wv = pexp + Q;                   // [Q] state weights of one segment end
    float* misc = wv + Q;                   // [2Q]: misc[0] = segment total
    int* segstart = (int*)(misc + 2 * Q);   // [Q] first row of row i's segment
    int* docid = segstart + Q;              // [Q] document (state index) of row i
    int* flags = docid + Q;                 // [Q] bit0: segment starts a document; bit1: row ends a document

    const int tid = threadIdx.x, nt = blockDim.x;
    const int w = tid >> 5, lane = tid & 31;   // segsum row tid (threads < Q)
    const int64_t u = blockIdx.x;
    const int s = (int)(u % a.nsplit);
    const int h = (int)((u / a.nsplit) % H);
    const int64_t b = u / ((int64_t)a.nsplit * H);
    const int g = h / (H / G);
    const int64_t t0 = (int64_t)s * a.split_len;
    const int64_t t1 = (t0 + a.split_len < L) ? t0 + a.split_len : L;
    const float A2 = a.A[h] * kLog2e;
    const float Dh = a.D ? a.D[h] : 0.f;
    const T* x = (const T*)a.x;
    const T* Bg = (const T*)a.B;
    const T* Cg = (const T*)a.C;
    T* y = (T*)a.y;
    const size_t PN = (size_t)P * N;

    // the full pass checks the call's packed-document offsets (block 0)
    if (a.cu && a.mode == kModeFull && u == 0) check_cu_seqlens(a.cu, a.ndocs, L, a.ws, tid, nt);
    // incoming state: from the split scan (slot s - 1) when this split continues a document
    for (int k = tid; k < P * N; k += nt)
        S[k] = (a.mode == kModeFull && a.nsplit > 1 && s > 0) ? a.ws_state[(u - 1) * PN + k] : 0.f;
    float tau = 0.f;  // natural-log decay applied to the split's incoming state

    for (int64_t c0 = t0; c0 < t1; c0 += Q) {
        const int n = (int)((c0 + Q < t1) ? Q : t1 - c0);
        __syncthreads();
        for (int k = tid; k < Q * P; k += nt) {
            int i = k / P, p = k % P;
            xs[k] = (i < n) ? Elem<T>::load(x + (((b * L + c0 + i) * H + h) * P + p)) : 0.f;
        }
        for (int k = tid; k < Q * N; k += nt) {
            int i = k / N, q = k % N;
            bool ok = i < n;
            int64_t off = ((b * L + c0 + i) * G + g) * N + q;
            Bs[k] = ok ? Elem<T>::load(Bg + off) : 0.f;
            Cs[k] = ok ? Elem<T>::load(Cg + off) : 0.f;
        }
        for (int i = tid; i < Q; i += nt) {
            float d = (i < n) ? a.dt[(b * L + c0 + i) * H + h] : 0.f;
            dtv[i] = d;
            const float l2 = d * A2;   // 0 past the chunk's last token
            int st = 0, doc = (int)b, fl = 0;
            if (i < n) {
                const int64_t t = c0 + i;
                if (a.cu) {
                    doc = find_doc(a.cu, a.ndocs, t);
                    const int64_t ds = a.cu[doc];
                    // (clamped to the row: offsets that break their contract keep the
                    // shared-memory indexes in bounds)
                    st = (ds > c0) ? (int)((ds - c0 < i) ? ds - c0 : i) : 0;
                    if (ds >= c0) fl |= 1;
                    if (t + 1 == a.cu[doc + 1]) fl |= 2;
                } else {
                    if (c0 == 0) fl |= 1;
                    if (t == L - 1) fl |= 2;
                }
            }
            lreal[i] = l2;
            sg.ell[i] = (st == i && i > 0) ? -INFINITY : l2;   // a document starts inside the chunk
            segstart[i] = st;
            docid[i] = doc;
            flags[i] = fl;
        }
        __syncthreads();
        SegsumRow<NW> R;
        if (tid < Q) segsum_phase1<NW>(sg, R, w, lane);
        __syncthreads();
        if (tid < Q) segsum_phase2<NW>(sg, R, w, lane);
        // (a) decay mask rows: M[i][j] = 2^{seg(i, j)} dt_j (0 before the row's
        //     segment start and above the diagonal); pexp_i for the state term
        if (tid < Q) {
            const int i = tid;
            float* Mi = M + (size_t)i * Q;
            const int st = segstart[i];
            float sst = 0.f;   // seg(i, st)
#pragma unroll
            for (int r = 0; r < NW; ++r) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int j = 32 * r + c;
                    const float sv = segsum_entry<NW>(sg, R, w, lane, r, c);
                    if (j == st) sst = sv;
                    Mi[j] = (i < n && j <= i) ? exp2f(sv) * dtv[j] : 0.f;
                }
            }
            pexp[i] = (st > 0) ? exp2f(sst + lreal[st]) : exp2f(R.p);
        }
        __syncthreads();
        // (b) times C_i . B_j
        for (int k = tid; k < n * Q; k += nt) {
            int i = k / Q, j = k % Q;
            if (j <= i && j >= segstart[i]) {
                const float* ci = Cs + (size_t)i * N;
                const float* bj = Bs + (size_t)j * N;
                float acc = 0.f;
                for (int q = 0; q < N; ++q) acc = fmaf(ci[q], bj[q], acc);
                M[(size_t)i * Q + j] *= acc;
            }
        }
        __syncthreads();
        // (c) outputs
        if (a.mode == kModeFull) {
            for (int k = tid; k < n * P; k += nt) {
                int i = k / P, p = k % P;
                const float* Mi = M + (size_t)i * Q;
                float acc = 0.f;
                for (int j = segstart[i]; j <= i; ++j) acc = fmaf(Mi[j], xs[j * P + p], acc);
                const float* ci = Cs + (size_t)i * N;
                float st = 0.f;
                if (!(flags[segstart[i]] & 1)) {
                    const float* Sp = S + (size_t)p * N;
                    for (int q = 0; q < N; ++q) st = fmaf(ci[q], Sp[q], st);
                } else if (a.init) {
                    const float* Ip = a.init + (((size_t)docid[i] * H + h) * P + p) * N;
                    for (int q = 0; q < N; ++q) st = fmaf(ci[q], Ip[q], st);
                }
                acc = fmaf(pexp[i], st, acc);
                acc = fmaf(Dh, xs[i * P + p], acc);
                Elem<T>::store(y + (((b * L + c0 + i) * H + h) * P + p), acc);
            }
        }
        // (d) states at segment ends: the chunk end (carried) and document ends
        for (int e = 0; e < n; ++e) {
            const bool chunk_end = (e == n - 1);
            const bool doc_end = (flags[e] & 2) != 0;
            if (!chunk_end && !doc_end) continue;
            const bool write_fin = doc_end && a.fin && a.mode == kModeFull;
            if (!chunk_end && !write_fin) continue;
            const int st = segstart[e];
            __syncthreads();
            if (tid == e) {
                // row e of the segsum: weights 2^{seg(e, j)} dt_j (0 before the segment)
#pragma unroll
                for (int r = 0; r < NW; ++r) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int j = 32 * r + c;
                        if (j <= e) wv[j] = exp2f(segsum_entry<NW>(sg, R, w, lane, r, c)) * dtv[j];
                    }
                }
                misc[0] = pexp[e];
            }
            __syncthreads();
            const bool starts_doc = (flags[st] & 1) != 0;
            const float decay = misc[0];
            const float* I0 = (starts_doc && a.init) ? a.init + ((size_t)docid[e] * H + h) * PN : nullptr;
            for (int k = tid; k < P * N; k += nt) {
                int p = k / N, q = k % N;
                float s0 = starts_doc ? (I0 ? I0[k] : 0.f) : S[k];
                float v = decay * s0;
                for (int j = st; j <= e; ++j) v = fmaf(wv[j] * xs[j * P + p], Bs[j * N + q], v);
                if (write_fin) a.fin[((size_t)docid[e] * H + h) * PN + k] = v;
                if (chunk_end) S[k] = v;   // each element read and written by one thread only
            }
        }
        // the split's total decay: -inf once a document starts inside it (the
        // chunk total is the segsum's, in log2, -inf past a document start)
        if (tid == 0) {
            bool restart = false;
            for (int i = 0; i < n; ++i)
                if (i == segstart[i] && (flags[i] & 1)) restart = true;
            tau = restart ? -INFINITY : tau + sg.tau * 0.6931471805599453f;
        }
    }
    if (a.mode == kModeAggregate) {
        __syncthreads();
        for (int k = tid; k < P * N; k += nt) a.ws_state[u * PN + k] = S[k];
        if (tid == 0) a.ws_tau[u] = tau;
    }
}

// Composition of split aggregates, left to right per (row, head):
// (tau_1, S_1) then (tau_2, S_2) -> (tau_1 + tau_2, exp(tau_2) S_1 + S_2).
// Slot s of a (row, head) holds the aggregate of split s (splits 0 .. nsplit-2;
// split 0's includes the caller's initial state).  In place, slot s - 1
// receives the state entering split s: slot 0 already is that of split 1, and
// S_in(s + 1) = exp(tau_s) S_in(s) + agg_s goes over agg_s in slot s.  So the
// scan reads nsplit - 1 slots and writes nsplit - 2 (nothing with two splits),
// and no slot holds the zero state of split 0 or the unneeded aggregate of
// the last split.  One thread owns 4 consecutive state elements; the loads of
// the next kScanDepth slots are issued before the current ones are combined,
// so the sequential chain waits on arithmetic, not on memory.
constexpr int kScanDepth = 8;

__global__ void ssd_split_scan(const float* __restrict__ tau, float* __restrict__ state,
                               int64_t units_bh, int nsplit, int PN) {
    const int PN4 = PN >> 2;
    const int nagg = nsplit - 1;   // slots holding aggregates
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // (no early trigger: the full pass starts as this grid's blocks exit, so it does not
    // compete for bandwidth with the scan, which is bandwidth-bound at short splits)
    pdl_wait();                    // the aggregates are complete (also on the early return)
    if (nagg < 2 || k >= units_bh * PN4) return;
    const int64_t bh = k / PN4;
    const int e4 = (int)(k % PN4);
    float4* st = reinterpret_cast<float4*>(state) + bh * nsplit * (int64_t)PN4 + e4;
    const float* tu = tau + bh * nsplit;
    float4 run = st[0];   // S_in(1)
    float4 cur[kScanDepth];
    float ct[kScanDepth];
#pragma unroll
    for (int d = 0; d < kScanDepth; ++d) {
        if (1 + d < nagg) {
            cur[d] = st[(int64_t)(1 + d) * PN4];
            ct[d] = tu[1 + d];
        }
    }
    for (int s0 = 1; s0 < nagg; s0 += kScanDepth) {
        float4 nxt[kScanDepth];
        float nt[kScanDepth];
#pragma unroll
        for (int d = 0; d < kScanDepth; ++d) {
            const int sn = s0 + kScanDepth + d;
            if (sn < nagg) {
                nxt[d] = st[(int64_t)sn * PN4];
                nt[d] = tu[sn];
            }
        }
#pragma unroll
        for (int d = 0; d < kScanDepth; ++d) {
            if (s0 + d < nagg) {
                const float e = expf(ct[d]);
                run = make_float4(fmaf(e, run.x, cur[d].x), fmaf(e, run.y, cur[d].y), fmaf(e, run.z, cur[d].z),
                                  fmaf(e, run.w, cur[d].w));
                st[(int64_t)(s0 + d) * PN4] = run;   // S_in(s0 + d + 1)
            }
        }
#pragma unroll
        for (int d = 0; d < kScanDepth; ++d) {
            cur[d] = nxt[d];
            ct[d] = nt[d];
        }
    }
}

// Reverse composition for the backward pass's splits: the adjoint of the state
// leaving split s, Lam_out(s) = e^{tau_{s+1}} Lam_out(s + 1) + V_{s+1}, from
// Lam_out(nsplit - 1) = dfin (or zero).  In place: slot s + 1 (V_{s+1})
// receives Lam_out(s), for s = nsplit - 2 down to 0.  tau: the splits' totals
// (split s at s).  The loads of the next kScanDepth slots are in flight while
// the current ones are combined.
__global__ void ssd_split_rscan(const float* __restrict__ tau, float* __restrict__ state,
                                const float* __restrict__ dfin, int64_t units_bh, int nsplit, int PN) {
    const int PN4 = PN >> 2;
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (nsplit < 2 || k >= units_bh * PN4) return;
    const int64_t bh = k / PN4;
    const int e4 = (int)(k % PN4);
    float4* st = reinterpret_cast<float4*>(state) + bh * nsplit * (int64_t)PN4 + e4;
    const float* tu = tau + bh * nsplit;
    float4 run = dfin ? reinterpret_cast<const float4*>(dfin)[bh * PN4 + e4] : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 cur[kScanDepth];
    float ct[kScanDepth];
#pragma unroll
    for (int d = 0; d < kScanDepth; ++d) {
        const int sn = nsplit - 1 - d;   // slots nsplit - 1, nsplit - 2, ..., 1
        if (sn >= 1) {
            cur[d] = st[(int64_t)sn * PN4];
            ct[d] = tu[sn];
        }
    }
    for (int s0 = nsplit - 1; s0 >= 1; s0 -= kScanDepth) {
        float4 nxt[kScanDepth];
        float nt[kScanDepth];
#pragma unroll
        for (int d = 0; d < kScanDepth; ++d) {
            const int sn = s0 - kScanDepth - d;
            if (sn >= 1) {
                nxt[d] = st[(int64_t)sn * PN4];
                nt[d] = tu[sn];
            }
        }
#pragma unroll
        for (int d = 0; d < kScanDepth; ++d) {
            const int sc = s0 - d;
            if (sc >= 1) {
                const float e = expf(ct[d]);
                run = make_float4(fmaf(e, run.x, cur[d].x), fmaf(e, run.y, cur[d].y), fmaf(e, run.z, cur[d].z),
                                  fmaf(e, run.w, cur[d].w));
                st[(int64_t)sc * PN4] = run;   // Lam_out(sc - 1)
            }
        }
#pragma unroll
        for (int d = 0; d < kScanDepth; ++d) {
            cur[d] = nxt[d];
            ct[d] = nt[d];
        }
    }
}

// Both forms of the segsum routine on rows of log2-decays: the log-domain
// seg the SIMT kernel exponentiates, and the linear-domain mask, row prefix
// and column suffix factors the tensor-core kernel multiplies in (the same
// device functions, with the same inputs a_k = ex2(l_k)).
template <int NW>
__global__ void __launch_bounds__(32 * NW) ssd_segsum_dump_k(const float* __restrict__ l2, int64_t nrows,
                                                             float* __restrict__ seg_out,
                                                             float* __restrict__ L_out,
                                                             float* __restrict__ pexp_out,
                                                             float* __restrict__ sfx_out) {
    constexpr int Q = 32 * NW;
    __shared__ SegsumShared<NW> sh;
    __shared__ SegsumLinShared<NW> shl;
    const int i = threadIdx.x, w = i >> 5, lane = i & 31;
    for (int64_t row = blockIdx.x; row < nrows; row += gridDim.x) {
        __syncthreads();
        const float l = l2[row * Q + i];
        sh.ell[i] = l;
        shl.a[i] = ex2_approx(l);
        __syncthreads();
        SegsumRow<NW> R;
        SegsumLinRow<NW> RL;
        segsum_phase1<NW>(sh, R, w, lane);
        segsum_lin_phase1<NW>(shl, RL, w, lane);
        __syncthreads();
        segsum_phase2<NW>(sh, R, w, lane);
        segsum_lin_phase2<NW>(shl, RL, w, lane);
        __syncthreads();
        if (pexp_out) pexp_out[row * Q + i] = RL.pe;
        if (sfx_out) sfx_out[row * Q + i] = segsum_lin_suffix<NW>(shl, i);
        float* so = seg_out ? seg_out + (row * Q + i) * Q : nullptr;
        float* lo = L_out ? L_out + (row * Q + i) * Q : nullptr;
#pragma unroll
        for (int r = 0; r < NW; ++r) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                if (so) so[32 * r + c] = segsum_entry<NW>(sh, R, w, lane, r, c);
                if (lo) lo[32 * r + c] = segsum_lin_entry<NW>(shl, RL, w, r, c);
            }
        }
    }
}

template <typename T, int NW>
cudaError_t launch_simt_q(const FwdArgs& a, size_t smem, int64_t grid, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(ssd_chunk_simt<T, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ssd_chunk_simt<T, NW><<<(unsigned)grid, 256, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_simt(const FwdArgs& a, cudaStream_t st) {
    const size_t smem = simt_smem_bytes(a.Q, a.P, a.N);
    const int64_t grid = a.batch * a.H * a.nsplit;
    if (a.Q != 64 && a.Q != 128) return cudaErrorInvalidValue;
    if (a.dtype == SSD_BF16)
        return a.Q == 128 ? launch_simt_q<__nv_bfloat16, 4>(a, smem, grid, st)
                          : launch_simt_q<__nv_bfloat16, 2>(a, smem, grid, st);
    return a.Q == 128 ? launch_simt_q<float, 4>(a, smem, grid, st) : launch_simt_q<float, 2>(a, smem, grid, st);
}

cudaError_t launch_split_rscan(const FwdArgs& a, const float* dfin, cudaStream_t st) {
    const int PN = a.P * a.N;
    const int64_t total = a.nsplit > 1 ? a.batch * a.H * (int64_t)(PN / 4) : 1;
    const int threads = 256;
    ssd_split_rscan<<<(unsigned)((total + threads - 1) / threads), threads, 0, st>>>(
        a.ws_tau, a.ws_state, dfin, a.batch * a.H, a.nsplit, PN);
    return cudaGetLastError();
}

cudaError_t launch_split_scan(const FwdArgs& a, cudaStream_t st) {
    const int PN = a.P * a.N;   // a multiple of 4: P * 4 bytes is a multiple of 16
    // (with two splits there is nothing to compose: one block that returns at once)
    const int64_t total = a.nsplit > 2 ? a.batch * a.H * (int64_t)(PN / 4) : 1;
    const int threads = 256;
    return launch_kernel(ssd_split_scan, (unsigned)((total + threads - 1) / threads), threads, 0, st, a.pdl != 0,
                         (const float*)a.ws_tau, a.ws_state, a.batch * a.H, a.nsplit, PN);
}

cudaError_t launch_segsum_dump(const float* l2, int64_t nrows, int chunk, float* seg, float* L, float* pexp,
                               float* sfx, cudaStream_t st) {
    const unsigned grid = (unsigned)(nrows < 4096 ? nrows : 4096);
    if (chunk == 128) ssd_segsum_dump_k<4><<<grid, 128, 0, st>>>(l2, nrows, seg, L, pexp, sfx);
    else ssd_segsum_dump_k<2><<<grid, 64, 0, st>>>(l2, nrows, seg, L, pexp, sfx);
    return cudaGetLastError();
}

}  // namespace ssd
