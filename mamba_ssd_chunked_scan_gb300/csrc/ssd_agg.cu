// Split aggregates on the tensor cores: for each split s of a sequence and
// each head h, the state the split leaves when it starts from zero (from the
// initial state for the first split) and the split's total log-decay,
//
//   S_s = sum_{t in split} 2^{seg(end, t)} dt_t x_t B_t^T        (P x N)
//   tau_s = sum_{t in split} l_t                                  (natural log)
//
// ("GPU Hierarchy Meets Structured Matrices", abstract: the split-sequence
// algorithm; "Parallel Scan and Hardware-Aware SSM Kernels", "The scan": each
// split is one affine step S -> e^{tau} S + S_s, composed afterwards).  The
// whole split is one contraction over its tokens: S^T = B^T X~ with
// X~_t = w_t x_t, w_t = 2^{seg(end, t)} dt_t.  Its chunks are visited from
// the split's end backwards, so that w_t is the chunk's column suffix (the
// linear-domain hierarchy-aware segsum of segsum.cuh) times the running
// product of the later chunks' totals, and every chunk adds into one TMEM
// accumulator: no per-chunk state update.  Heads of one B/C group share the
// A operand B^T, so one CTA takes K in {1, 2} of them and each UMMA step is
// N = 64 K wide.
//
// Warps: 0 TMA producer (a ring of B and K x tiles, as many stages as fit),
// 1 MMA issuer, 2 TMEM owner; warpgroups 1 and 2 are scaling groups that take
// alternating chunks, one thread per chunk row: log-decays (dt loaded one
// item ahead), segsum, the scaled x rows written in place.
// The running product of the later chunks' totals passes from one group to
// the other through shared memory; group 1 writes the states at the end.
//
// Reverse mode (kRev, for the backward pass's sequence splits): the adjoint
// entering split s from its right, V_s = sum_{i in split} 2^{P_i} dy_i C_i^T
// with P_i = sum_{k=split start..i} l_k, is the same contraction with C in
// place of B, dy in place of x, the chunks visited from the split's start
// forwards and the row prefix 2^{p_i} times the running product of the
// earlier chunks' totals in place of the suffix weight (no dt factor).  It is
// formed for splits 1 .. nsplit - 1.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stddef.h>

#include <atomic>

#include "ssd_common.cuh"
#include "segsum.cuh"
#include "ssd_kernels.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

constexpr int Q = 128, P = 64, N = 128;
constexpr int kThreads = 384;
constexpr uint32_t kTileB = 32768, kTileX = 16384;
constexpr int kBarScale0 = 1;    // named barriers of scaling groups 1 and 2 (ids 1, 2)
constexpr int kBarBoth = 3;      // both scaling groups
constexpr float kLn2 = 0.6931471805599453f;

enum : uint32_t { kWhereAggEmpty = 21, kWhereAggFull = 22, kWhereAggReady = 23, kWhereAggDone = 24,
                  kWhereAggDrain = 25, kWhereAggRdy = 26 };

template <int K>
struct AggCfg {
    static constexpr uint32_t kStage = kTileB + K * kTileX;   // B (two 64-column slabs), then K x tiles
    static constexpr int kStages = K == 4 ? 2 : K == 2 ? 3 : 4; // as many stages as shared memory holds
    static constexpr uint32_t kCols = K * P < 32 ? 32 : K * P; // TMEM accumulator columns
    static constexpr size_t kSmem = 1024 + kStages * kStage;
};

struct AggSmall {
    SegsumLinShared<4> seg[2][4];   // per scaling group and head
    float lsum[2][4][4];            // per group, head and warp: sums of the log2-decays over the split
    float rin[2][4];                // running product of the later chunks' totals, by chunk parity
    uint64_t full[4], empty[4], ready[4], rdy[2], done;
    uint32_t tmem_base;
    int abort;
    int never;
};

// L2 policies: x streams through once (evicted first), while the split states stay
// for the split scan that reads them next (evicted last); without them the x
// stream pushed the states out of L2 and the scan read them back from HBM.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void tma_load_4d_hint(void* smem_dst, const CUtensorMap* tm, uint64_t* bar, int c0, int c1,
                                                 int c2, int c3, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
        "%4, %5, %6}], [%2], %7;" ::"r"(ptx::smem_u32(smem_dst)),
        "l"(tm), "r"(ptx::smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void st_hint(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

struct AggParams {
    CUtensorMap tm_x, tm_B;
    FwdArgs a;
    int nsplit_agg;   // splits that need an aggregate (all but the last)
};

__device__ __forceinline__ bool agg_wait(AggSmall& sh, const FwdArgs& a, uint64_t* bar, uint32_t parity,
                                         uint32_t where) {
    if (ptx::mbar_wait(bar, parity, &sh.abort, a.wait_iters)) return true;
    if (!*(volatile int*)&sh.abort) {
        record_error(a.ws, SSD_ERR_TIMEOUT, where);
        *(volatile int*)&sh.abort = 1;
    }
    return false;
}

__device__ __forceinline__ int find_doc_agg(const int32_t* cu, int ndocs, int64_t t) {
    int lo = 0, hi = ndocs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Two bf16 values (one 32-bit word) times f2 = (f, f), rounded back to bf16;
// the two products in one packed fp32 multiply (each lane rounds as mul.rn.f32).
__device__ __forceinline__ uint32_t scale_pair(uint32_t w, uint64_t f2) {
    float lo, hi;
    ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)), f2), lo, hi);
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int K, bool kDocs, bool kRev>
__global__ void __launch_bounds__(kThreads, 1) ssd_split_agg_tc(const __grid_constant__ AggParams prm) {
    using Cfg = AggCfg<K>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ AggSmall sh;
    const FwdArgs& a = prm.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();                                // the split scan may start on SMs this grid leaves free

    // unit: (batch row, split, group of K heads), head groups fastest so that
    // CTAs running together share B in L2
    const int nhq = a.H / K;
    const int64_t u = blockIdx.x;
    const int hq = (int)(u % nhq);
    const int64_t bs = u / nhq;
    const int s = (int)(bs % prm.nsplit_agg) + (kRev ? 1 : 0);   // (reverse mode: splits 1 ..)
    const int b = (int)(bs / prm.nsplit_agg);
    const int h0 = hq * K;
    const int g = h0 / (a.H / a.G);
    const int t0 = (int)(s * a.split_len);
    const int t1 = (int)((t0 + a.split_len < a.L) ? t0 + a.split_len : a.L);
    const int nch = (t1 - t0 + Q - 1) / Q;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::kStages; ++i) {
            ptx::mbar_init(&sh.full[i], 1);
            ptx::mbar_init(&sh.empty[i], 1);
            ptx::mbar_init(&sh.ready[i], 4);
        }
        for (int i = 0; i < 2; ++i) ptx::mbar_init(&sh.rdy[i], 1);
        ptx::mbar_init(&sh.done, 1);
        sh.abort = 0;
        sh.never = 0;
        for (int h = 0; h < 4; ++h) sh.rin[0][h] = 1.f;   // nothing after the split's last chunk
        ptx::mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&prm.tm_x);
        ptx::prefetch_tmap(&prm.tm_B);
    }
    if (warp == 2) ptx::tmem_alloc(&sh.tmem_base, Cfg::kCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tb = sh.tmem_base;
    if (threadIdx.x == 0) ptx::mbar_arrive(&sh.rdy[0]);   // the last chunk's factor (1) is ready

    if (warp == 0) {
        if (lane == 0) {
            // ============================================================ TMA producer
            int issued = 0;
            constexpr int NS = Cfg::kStages;
            const uint64_t stream_pol = l2_evict_first();
            for (int r = 0; r < (a.stall_loads ? 0 : nch); ++r) {
                const int st = r % NS;
                if (r >= NS && !agg_wait(sh, a, &sh.empty[st], ((r / NS) - 1) & 1, kWhereAggEmpty)) break;
                const int t = t0 + (kRev ? r : nch - 1 - r) * Q;   // chunks from the split's end backwards
                uint8_t* stg = sm + st * Cfg::kStage;
                ptx::mbar_expect_tx(&sh.full[st], Cfg::kStage);
                ptx::tma_load_4d(stg, &prm.tm_B, &sh.full[st], 0, g, t, b);
                ptx::tma_load_4d(stg + 16384, &prm.tm_B, &sh.full[st], 64, g, t, b);
#pragma unroll
                for (int h = 0; h < K; ++h)
                    tma_load_4d_hint(stg + kTileB + h * kTileX, &prm.tm_x, &sh.full[st], 0, h0 + h, t, b, stream_pol);
                ++issued;
            }
            for (int st = 0; st < NS && st < issued; ++st) {
                const int last = ((issued - 1 - st) / NS) * NS + st;
                if (!ptx::mbar_wait(&sh.full[st], (last / NS) & 1, &sh.never, a.wait_iters)) {
                    record_error(a.ws, SSD_ERR_TIMEOUT, kWhereAggDrain);
                    *(volatile int*)&sh.abort = 1;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ============================================================ MMA issuer
            // S^T (n rows, K x 64 p columns) += B^T X~ over the chunk's 128 tokens
            constexpr uint32_t id = ptx::idesc_bf16(128, K * P, 1, 1);
            for (int r = 0; r < nch; ++r) {
                const int st = r % Cfg::kStages;
                if (!agg_wait(sh, a, &sh.ready[st], (r / Cfg::kStages) & 1, kWhereAggReady)) break;
                ptx::tc_fence_after();
                const uint32_t stg = ptx::smem_u32(sm + st * Cfg::kStage);
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb, ptx::sdesc_sw128(stg + kk * 2048, 16384, 1024),
                                ptx::sdesc_sw128(stg + kTileB + kk * 2048, 16384, 1024), id, (r > 0 || kk > 0));
                ptx::mma_commit(&sh.empty[st]);
            }
            ptx::mma_commit(&sh.done);
        }
    } else if (warp >= 4) {
        // ================================================================ scaling groups
        const int X = (warp >> 2) - 1;            // group X takes the items r with r & 1 == X
        const int nb = kBarScale0 + X;
        const int mt = (threadIdx.x & 127);       // 0..127
        const int rb = warp & 3;
        const int i = 32 * rb + lane;             // chunk row; TMEM lane = state column n
        float A2[K], Ls[K];
#pragma unroll
        for (int h = 0; h < K; ++h) {
            A2[h] = a.A[h0 + h] * kLog2e;
            Ls[h] = 0.f;
        }
        int doc = 0;   // document cursor (packed documents), moving backwards
        if (kDocs && !kRev) doc = find_doc_agg(a.cu, a.ndocs, (int64_t)t1 - 1);
        // dt of item r for this thread's row (0 past the split), loaded one item ahead
        auto load_dt = [&](int r, float (&v)[K]) {
            const int t = t0 + (kRev ? r : nch - 1 - r) * Q;
            const bool ok = r < nch && t + i < t1;
            const float* dp = a.dt + ((size_t)b * a.L + t + i) * a.H + h0;
            if constexpr (K == 4) {
                const float4 q = ok ? __ldg(reinterpret_cast<const float4*>(dp)) : make_float4(0.f, 0.f, 0.f, 0.f);
                v[0] = q.x;
                v[1] = q.y;
                v[2] = q.z;
                v[3] = q.w;
            } else {
#pragma unroll
                for (int h = 0; h < K; ++h) v[h] = ok ? __ldg(dp + h) : 0.f;
            }
        };
        float dtn[K];
        load_dt(X, dtn);
        for (int r = X; r < nch; r += 2) {
            const int j = r >> 1;
            const int t = t0 + (kRev ? r : nch - 1 - r) * Q;
            const bool valid = t + i < t1;
            float dtv[K];
#pragma unroll
            for (int h = 0; h < K; ++h) dtv[h] = dtn[h];
            load_dt(r + 2, dtn);
            bool start = false;   // a document starts at this token (after the first)
            if (kDocs && valid) {
                if (kRev) doc = find_doc_agg(a.cu, a.ndocs, (int64_t)t + i);   // (chunks forwards)
                else
                    while (doc > 0 && __ldg(a.cu + doc) > t + i) --doc;
                start = doc > 0 && __ldg(a.cu + doc) == t + i;
            }
#pragma unroll
            for (int h = 0; h < K; ++h) {
                const float l2 = start ? -INFINITY : dtv[h] * A2[h];
                sh.seg[X][h].a[i] = ex2_approx(l2);   // 0 at a document start
                Ls[h] += l2;                          // this row's share of the split's total
            }
            ptx::named_bar(nb, 128);
            // segsum: the diagonal blocks, then the rank-one row factors (the
            // column suffixes need both; the rows themselves are not used)
            float w0[K];
            {
                SegsumLinRow<4> rows[K];
                segsum_lin_phase1_k<4, K>(sh.seg[X], rows, rb, lane);
#pragma unroll
                for (int h = 0; h < K; ++h) w0[h] = rows[h].wl[0];
            }
            ptx::named_bar(nb, 128);
            float pe[K];   // 2^{p_i}: the row prefix (reverse mode's weight)
#pragma unroll
            for (int h = 0; h < K; ++h) {
                SegsumLinRow<4> row;
                row.wl[0] = w0[h];
                segsum_lin_phase2<4>(sh.seg[X][h], row, rb, lane);
                pe[h] = row.pe;
            }
            ptx::named_bar(nb, 128);
            // the product of the later chunks' totals (from the other group); as soon
            // as every thread has read it, the product that includes this chunk's
            // total goes on to the earlier chunk's group, so the two groups' scaling
            // work overlaps
            agg_wait(sh, a, &sh.rdy[r & 1], j & 1, kWhereAggRdy);
            float R[K];
#pragma unroll
            for (int h = 0; h < K; ++h) R[h] = sh.rin[r & 1][h];
            const bool stop = ptx::named_bar_any(nb, 128, *(volatile int*)&sh.abort != 0);
            if (mt == 0 && r + 1 < nch) {
#pragma unroll
                for (int h = 0; h < K; ++h) sh.rin[(r + 1) & 1][h] = R[h] * sh.seg[X][h].tauL;
                ptx::mbar_arrive(&sh.rdy[(r + 1) & 1]);
            }
            // x~ = 2^{seg(split end, t)} dt_t x_t, written over the x rows in place
            const int st = r % Cfg::kStages;
            agg_wait(sh, a, &sh.full[st], (r / Cfg::kStages) & 1, kWhereAggFull);
            uint8_t* xs = sm + st * Cfg::kStage + kTileB;
#pragma unroll
            for (int h = 0; h < K; ++h) {
                const float wgt = kRev ? pe[h] * R[h] : segsum_lin_suffix<4>(sh.seg[X][h], i) * R[h] * dtv[h];
                const uint64_t wgt2 = ptx::f2_pack(wgt, wgt);
                uint8_t* row = xs + h * kTileX;
                uint4 v[8];   // the whole row's loads in flight before the first multiply
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = *reinterpret_cast<const uint4*>(row + sw128_off(i, 8 * q));
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    v[q].x = scale_pair(v[q].x, wgt2);
                    v[q].y = scale_pair(v[q].y, wgt2);
                    v[q].z = scale_pair(v[q].z, wgt2);
                    v[q].w = scale_pair(v[q].w, wgt2);
                    *reinterpret_cast<uint4*>(row + sw128_off(i, 8 * q)) = v[q];
                }
            }
            ptx::fence_proxy_async();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sh.ready[st]);
            if (stop) break;
        }
        // the split's total log-decay: each thread's rows, then the warps' sums
#pragma unroll
        for (int h = 0; h < K; ++h) {
            float ls = Ls[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
            if (lane == 0) sh.lsum[X][h][rb] = ls;
        }
        ptx::named_bar(kBarBoth, 256);
        if (X == 0) {
            // the split's state: TMEM lane i holds column n = i of every head's S^T
            const bool ok = ptx::mbar_wait(&sh.done, 0, &sh.never, a.wait_iters);
            if (!ok) {
                record_error(a.ws, SSD_ERR_TIMEOUT, kWhereAggDone);
                *(volatile int*)&sh.abort = 1;
            }
            ptx::tc_fence_after();
            if (ok && !*(volatile int*)&sh.abort) {
                const uint32_t lane_addr = tb + ((uint32_t)(32 * rb) << 16);
                const size_t PN = (size_t)P * N;
#pragma unroll 1
                for (int h = 0; h < K; ++h) {
                    uint32_t d0[32], d1[32];
                    ptx::tmem_load32x2(lane_addr + h * P, d0, lane_addr + h * P + 32, d1);
                    const size_t ws = ((size_t)b * a.H + h0 + h) * a.nsplit + s;
                    const float lsum = ((sh.lsum[0][h][0] + sh.lsum[0][h][1]) + (sh.lsum[0][h][2] + sh.lsum[0][h][3])) +
                                       ((sh.lsum[1][h][0] + sh.lsum[1][h][1]) + (sh.lsum[1][h][2] + sh.lsum[1][h][3]));
                    float* out = a.ws_state + ws * PN + i;
                    // the first split starts from the caller's initial state (packed
                    // documents: the first document's, d = 0 = b; a later start in the
                    // split makes its decay 2^{-inf} = 0)
                    const float* init =
                        (!kRev && s == 0 && a.init) ? a.init + ((size_t)b * a.H + h0 + h) * PN + i : nullptr;
                    if (init) {
                        // (read-only loads, so that all of them are issued before the stores)
                        const float dec = ex2_approx(lsum);
#pragma unroll
                        for (int p = 0; p < 32; ++p) {
                            d0[p] = __float_as_uint(fmaf(dec, __ldg(init + (size_t)p * N), __uint_as_float(d0[p])));
                            d1[p] = __float_as_uint(
                                fmaf(dec, __ldg(init + (size_t)(p + 32) * N), __uint_as_float(d1[p])));
                        }
                    }
                    const uint64_t keep = l2_evict_last();
#pragma unroll
                    for (int p = 0; p < 32; ++p) {
                        st_hint(out + (size_t)p * N, __uint_as_float(d0[p]), keep);
                        st_hint(out + (size_t)(p + 32) * N, __uint_as_float(d1[p]), keep);
                    }
                    if (mt == 0) a.ws_tau[ws] = lsum * kLn2;   // (reverse mode: its own tau array)
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 2) ptx::tmem_dealloc(tb, Cfg::kCols);
}

template <int K, bool kDocs, bool kRev>
cudaError_t launch_k(const AggParams& prm, int64_t grid, cudaStream_t st) {
    static std::atomic<uint8_t> ready[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!ready[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(ssd_split_agg_tc<K, kDocs, kRev>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)AggCfg<K>::kSmem);
        if (e != cudaSuccess) return e;
        ready[dev].store(1, std::memory_order_release);
    }
    ssd_split_agg_tc<K, kDocs, kRev><<<(unsigned)grid, kThreads, AggCfg<K>::kSmem, st>>>(prm);
    return cudaGetLastError();
}

template <bool kRev>
cudaError_t launch_agg(const FwdArgs& a, cudaStream_t st) {
    AggParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.a = a;
    if (prm.a.wait_iters == 0) prm.a.wait_iters = kDefaultWaitIters;
    // forwards: splits 0 .. nsplit - 2 (the last split's aggregate is never composed
    // into a later split); reverse: splits 1 .. nsplit - 1 (nothing enters split 0's
    // left side)
    prm.nsplit_agg = a.nsplit - 1;
    if (prm.nsplit_agg < 1) return cudaSuccess;
    if (!encode_4d(&prm.tm_x, a.x, P, a.H, a.L, a.batch) || !encode_4d(&prm.tm_B, a.B, N, a.G, a.L, a.batch))
        return cudaErrorInvalidValue;
    const int K = agg_heads_per_cta(a.H, a.G);
    const int64_t grid = a.batch * (int64_t)prm.nsplit_agg * (a.H / K);
    const bool docs = a.cu != nullptr;
    if (K == 2) return docs ? launch_k<2, true, kRev>(prm, grid, st) : launch_k<2, false, kRev>(prm, grid, st);
    return docs ? launch_k<1, true, kRev>(prm, grid, st) : launch_k<1, false, kRev>(prm, grid, st);
}

}  // namespace

// Heads per CTA: 2 when each group's heads come in pairs (three 64 KB stages
// in flight), else 1 (four 48 KB stages).
int agg_heads_per_cta(int H, int G) {
    const int hg = H / G;
    return (hg % 2 == 0) ? 2 : 1;
}

cudaError_t launch_agg_tc(const FwdArgs& a, cudaStream_t st) { return launch_agg<false>(a, st); }

// The reverse aggregates V_s of the backward pass: a.x = dy, a.B = C,
// a.ws_state the slots (split s in slot s of its (row, head)) and a.ws_tau the
// splits' total log-decays (split s at s, for s >= 1).
cudaError_t launch_agg_rev_tc(const FwdArgs& a, cudaStream_t st) { return launch_agg<true>(a, st); }

}  // namespace ssd
