// SIMT (CUDA-core, fp32) kernels of libssd:
//   ssd_chunk_simt      the chunked SSD forward for any supported shape and
//                       dtype, fp32 arithmetic throughout (the fp32 path)
//   ssd_split_scan      composes split aggregates into incoming states
//   ssd_segsum_dump_k   the hierarchy-aware segsum routine on its own
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

size_t simt_smem_bytes(int Q, int P, int N) {
    size_t floats = (size_t)Q * P + 2 * (size_t)Q * N + (size_t)Q * Q + (size_t)P * N + 6 * (size_t)Q;
    size_t ints = 3 * (size_t)Q;
    return floats * 4 + ints * 4 + 64;
}

template <typename T>
__global__ void __launch_bounds__(256) ssd_chunk_simt(FwdArgs a) {
    extern __shared__ float smem[];
    const int Q = a.Q, P = a.P, N = a.N, H = a.H, G = a.G;
    const int64_t L = a.L;
    float* xs = smem;                       // [Q][P]
    float* Bs = xs + Q * P;                 // [Q][N]
    float* Cs = Bs + Q * N;                 // [Q][N]
    float* M = Cs + Q * N;                  // [Q][Q]
    float* S = M + Q * Q;                   // [P][N] carried state
    float* ell = S + P * N;                 // [Q] natural-log decays
    float* dtv = ell + Q;                   // [Q]
    float* pexp = dtv + Q;                  // [Q] exp(sum_{k=segstart..i} l_k)
    float* wv = pexp + Q;                   // [Q] state weights of one segment end
    float* misc = wv + Q;                   // [2Q]: misc[0] = segment total
    int* segstart = (int*)(misc + 2 * Q);   // [Q] first row of row i's segment
    int* docid = segstart + Q;              // [Q] document (state index) of row i
    int* flags = docid + Q;                 // [Q] bit0: segment starts a document; bit1: row ends a document

    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t u = blockIdx.x;
    const int s = (int)(u % a.nsplit);
    const int h = (int)((u / a.nsplit) % H);
    const int64_t b = u / ((int64_t)a.nsplit * H);
    const int g = h / (H / G);
    const int64_t t0 = (int64_t)s * a.split_len;
    const int64_t t1 = (t0 + a.split_len < L) ? t0 + a.split_len : L;
    const float Ah = a.A[h];
    const float Dh = a.D ? a.D[h] : 0.f;
    const T* x = (const T*)a.x;
    const T* Bg = (const T*)a.B;
    const T* Cg = (const T*)a.C;
    T* y = (T*)a.y;
    const size_t PN = (size_t)P * N;

    // incoming state: from the split scan when this split continues a document
    for (int k = tid; k < P * N; k += nt)
        S[k] = (a.mode == kModeFull && a.nsplit > 1 && s > 0) ? a.ws_state[u * PN + k] : 0.f;
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
            ell[i] = d * Ah;
            int st = 0, doc = (int)b, fl = 0;
            if (i < n) {
                const int64_t t = c0 + i;
                if (a.cu) {
                    doc = find_doc(a.cu, a.ndocs, t);
                    const int64_t ds = a.cu[doc];
                    st = (ds > c0) ? (int)(ds - c0) : 0;
                    if (ds >= c0) fl |= 1;
                    if (t + 1 == a.cu[doc + 1]) fl |= 2;
                } else {
                    if (c0 == 0) fl |= 1;
                    if (t == L - 1) fl |= 2;
                }
            }
            segstart[i] = st;
            docid[i] = doc;
            flags[i] = fl;
        }
        __syncthreads();
        // (a) decay mask rows: M[i][j] = exp(seg(i, j)) dt_j on the segment,
        //     seg grown leftwards from the diagonal; pexp_i for the state term
        for (int i = tid; i < Q; i += nt) {
            float* Mi = M + (size_t)i * Q;
            for (int j = 0; j < Q; ++j) Mi[j] = 0.f;
            if (i < n) {
                float r = 0.f;
                for (int j = i; j >= segstart[i]; --j) {
                    Mi[j] = expf(r) * dtv[j];
                    r += ell[j];
                }
                pexp[i] = expf(r);
            }
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
            if (tid == 0) {
                float r = 0.f;
                for (int j = e; j >= st; --j) {
                    wv[j] = expf(r) * dtv[j];
                    r += ell[j];
                }
                misc[0] = expf(r);
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
        // the split's total decay: -inf once a document starts inside it
        if (tid == 0) {
            bool restart = false;
            float csum = 0.f;
            for (int i = 0; i < n; ++i) {
                if (i == segstart[i] && (flags[i] & 1)) restart = true;
                csum += ell[i];
            }
            tau = restart ? -INFINITY : tau + csum;
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
// In place: slot s receives the state entering split s.
// Exclusive scan over the splits of one (row, head): the incoming state of
// split s is the composition of the aggregates of splits 0..s-1 (affine steps
// S -> exp(tau_s) S + agg_s).  One thread owns 4 consecutive state elements;
// the loads of the next kDepth splits are issued before the current ones are
// combined, so the sequential chain waits on arithmetic, not on memory.
constexpr int kScanDepth = 8;

__global__ void ssd_split_scan(const float* __restrict__ tau, float* __restrict__ state,
                               int64_t units_bh, int nsplit, int PN) {
    const int PN4 = PN >> 2;
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= units_bh * PN4) return;
    const int64_t bh = k / PN4;
    const int e4 = (int)(k % PN4);
    float4* st = reinterpret_cast<float4*>(state) + bh * nsplit * (int64_t)PN4 + e4;
    const float* tu = tau + bh * nsplit;
    float4 cur[kScanDepth];
    float ct[kScanDepth];
#pragma unroll
    for (int d = 0; d < kScanDepth; ++d) {
        if (d < nsplit) {
            cur[d] = st[(int64_t)d * PN4];
            ct[d] = tu[d];
        }
    }
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nsplit; s0 += kScanDepth) {
        float4 nxt[kScanDepth];
        float nt[kScanDepth];
#pragma unroll
        for (int d = 0; d < kScanDepth; ++d) {
            const int sn = s0 + kScanDepth + d;
            if (sn < nsplit) {
                nxt[d] = st[(int64_t)sn * PN4];
                nt[d] = tu[sn];
            }
        }
#pragma unroll
        for (int d = 0; d < kScanDepth; ++d) {
            if (s0 + d < nsplit) {
                st[(int64_t)(s0 + d) * PN4] = run;
                const float e = expf(ct[d]);
                run = make_float4(fmaf(e, run.x, cur[d].x), fmaf(e, run.y, cur[d].y), fmaf(e, run.z, cur[d].z),
                                  fmaf(e, run.w, cur[d].w));
            }
        }
#pragma unroll
        for (int d = 0; d < kScanDepth; ++d) {
            cur[d] = nxt[d];
            ct[d] = nt[d];
        }
    }
}

template <int NW>
__global__ void __launch_bounds__(32 * NW) ssd_segsum_dump_k(const float* __restrict__ l2, int64_t nrows,
                                                             float* __restrict__ seg_out,
                                                             float* __restrict__ L_out) {
    constexpr int Q = 32 * NW;
    __shared__ SegsumShared<NW> sh;
    const int i = threadIdx.x, w = i >> 5, lane = i & 31;
    for (int64_t row = blockIdx.x; row < nrows; row += gridDim.x) {
        __syncthreads();
        sh.ell[i] = l2[row * Q + i];
        __syncthreads();
        SegsumRow<NW> R;
        segsum_phase1<NW>(sh, R, w, lane);
        __syncthreads();
        segsum_phase2<NW>(sh, R, w, lane);
        float* so = seg_out ? seg_out + (row * Q + i) * Q : nullptr;
        float* lo = L_out ? L_out + (row * Q + i) * Q : nullptr;
#pragma unroll
        for (int r = 0; r < NW; ++r) {
            if (r < w) {
                const float rf = ex2_approx(R.R[r]);
#pragma unroll 8
                for (int c = 0; c < 32; ++c) {
                    const float cs = sh.colS[32 * r + c];
                    if (so) so[32 * r + c] = R.R[r] + cs;
                    if (lo) lo[32 * r + c] = rf * ex2_approx(cs);
                }
            } else if (r == w) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    if (so) so[32 * r + c] = (c <= lane) ? R.d[c] : -INFINITY;
                    if (lo) lo[32 * r + c] = (c <= lane) ? ex2_approx(R.d[c]) : 0.f;
                }
            } else {
                for (int c = 0; c < 32; ++c) {
                    if (so) so[32 * r + c] = -INFINITY;
                    if (lo) lo[32 * r + c] = 0.f;
                }
            }
        }
    }
}

cudaError_t launch_simt(const FwdArgs& a, cudaStream_t st) {
    const size_t smem = simt_smem_bytes(a.Q, a.P, a.N);
    const int64_t grid = a.batch * a.H * a.nsplit;
    if (a.dtype == SSD_BF16) {
        cudaFuncSetAttribute(ssd_chunk_simt<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        ssd_chunk_simt<__nv_bfloat16><<<(unsigned)grid, 256, smem, st>>>(a);
    } else {
        cudaFuncSetAttribute(ssd_chunk_simt<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        ssd_chunk_simt<float><<<(unsigned)grid, 256, smem, st>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_split_scan(const FwdArgs& a, cudaStream_t st) {
    const int PN = a.P * a.N;   // a multiple of 4: P * 4 bytes is a multiple of 16
    const int64_t total = a.batch * a.H * (int64_t)(PN / 4);
    const int threads = 256;
    ssd_split_scan<<<(unsigned)((total + threads - 1) / threads), threads, 0, st>>>(
        a.ws_tau, a.ws_state, a.batch * a.H, a.nsplit, PN);
    return cudaGetLastError();
}

cudaError_t launch_segsum_dump(const float* l2, int64_t nrows, int chunk, float* seg, float* L,
                               cudaStream_t st) {
    const unsigned grid = (unsigned)(nrows < 4096 ? nrows : 4096);
    if (chunk == 128) ssd_segsum_dump_k<4><<<grid, 128, 0, st>>>(l2, nrows, seg, L);
    else ssd_segsum_dump_k<2><<<grid, 64, 0, st>>>(l2, nrows, seg, L);
    return cudaGetLastError();
}

}  // namespace ssd
