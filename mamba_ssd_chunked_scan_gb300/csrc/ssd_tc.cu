// Tensor-core (tcgen05 / TMEM / TMA) kernel of the chunked SSD forward pass
// for the Mamba-2 head shape: chunk Q = 128, head dim P = 64, state N = 128,
// bf16 x / B / C / y, fp32 dt / A / D / states, fp32 accumulation.
//
// One CTA walks the chunks of one (batch row, head, split) unit and keeps the
// P x N state on chip between chunks ("State Space Duality and Mamba-2",
// "The SSD Block Decomposition Algorithm"; "NVIDIA Accelerates Mamba-2
// Forward Kernel with CUDA Tile": intra-block parallel, inter-block
// recurrent, state resident on chip).  Per chunk c:
//
//   G     = C B^T                        (UMMA 128x128x128 -> TMEM)
//   M     = G o L o dt                   (hierarchy-aware segsum mask, bf16 -> TMEM)
//   Ydiag = M X                          (UMMA, A operand from TMEM)
//   dS    = B^T (exp(s_j) dt_j x_j)      (UMMA, chunk state summary)
//   Yoff  = C S_in^T                     (UMMA; the row decay exp(p_i) is applied in the epilogue)
//   S     = exp(tau) S + dS              (state carried in registers)
//   y     = Ydiag + exp(p_i) Yoff + D x  (epilogue, TMA store)
//
// Warp roles (320 threads):
//   warp 0      TMA producer (two-stage ring of C, B, X tiles)
//   warp 1      TMEM owner and MMA issuer
//   warps 2-5   mask group: log-decays, segsum, scaled X tile, mask M
//   warps 6-9   state group: state update, incoming-state tile, epilogue
// One thread of each math group owns one chunk row (= TMEM lane).  The MMA
// issue order G(c), Ydiag(c), dS(c), G(c+1), Yoff(c) keeps the tensor pipe
// fed while the state group closes the state recurrence of chunk c; the Y
// accumulators are double-buffered in TMEM so the epilogue of chunk c
// overlaps the products of chunk c+1.
//
// Every wait is bounded; a wait that runs out records SSD_ERR_TIMEOUT in the
// workspace status word, and the CTA drains its copies, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <stddef.h>

#include "ssd_common.cuh"
#include "segsum.cuh"
#include "ssd_kernels.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

constexpr int Q = 128, P = 64, N = 128;
constexpr int NS = 2;                        // input stages
constexpr int kThreads = 320;
constexpr uint32_t kTileC = 0, kTileB = 32768, kTileX = 65536, kStageBytes = 81920;
constexpr uint32_t kXt = NS * kStageBytes;   // scaled X for the state summary
constexpr uint32_t kSin = kXt + 16384;       // incoming state, bf16, (n rows, p)
constexpr uint32_t kYs = kSin + 16384;       // y staging for the TMA store
constexpr uint32_t kTiles = kYs + 16384;
// TMEM columns: G | M (bf16 pairs) | dS | Ydiag[2] | Yoff[2]
constexpr uint32_t kTmG = 0, kTmM = 128, kTmDS = 192, kTmYd = 256, kTmYo = 384, kTmCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kBarMask = 1, kBarState = 2;   // named barriers of the two math groups

// codes of the wait that gave up (WsHeader::where)
enum : uint32_t {
    kWhereEmpty = 1, kWhereFull = 2, kWhereBarM = 3, kWhereYFree = 4, kWhereDsFree = 5, kWhereBarS = 6,
    kWhereMetaFree = 7, kWhereBarDS = 8, kWhereBarG = 9, kWhereMetaFull = 10, kWhereBarY = 11,
    kWhereDrain = 12
};

// Per-chunk values handed from the mask group to the state group.
struct ChunkMeta {
    alignas(16) float pexp[Q];   // 2^{p_i}: decay of the incoming state at row i
    alignas(16) float ell[Q];    // log2-decays
    alignas(16) float dtv[Q];
    int rowflag[Q];              // bit0: a document starts at this token, bit1: one ends here
    int rowdoc[Q];               // state index (document, or batch row)
    float tau;                   // whole-chunk log2-decay
};

struct TcSmall {
    SegsumShared<4> seg;
    alignas(16) float dtv[Q];      // read as float4
    alignas(16) float colfac[Q];   // read as float4
    alignas(16) float wv[Q];
    ChunkMeta meta[2];
    int doc_cursor;
    uint64_t full[NS], empty[NS];
    uint64_t barG, barM, barDS, barS, barY, dsFree, barDrain;
    uint64_t yFree[2], metaFull[2], metaFree[2];
    uint32_t tmem_base;
    int abort;
    int never;                     // stays 0: lets drain waits ignore the abort flag
};

static_assert(offsetof(TcSmall, dtv) % 16 == 0 && offsetof(TcSmall, colfac) % 16 == 0,
              "vector-loaded arrays must be 16-byte aligned");
static_assert(offsetof(TcSmall, meta) % 16 == 0 && sizeof(ChunkMeta) % 16 == 0, "meta alignment");
static_assert(offsetof(TcSmall, full) % 8 == 0, "mbarriers are 8-byte aligned");
static_assert(kTiles % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");

struct TcParams {
    CUtensorMap tm_x, tm_B, tm_C, tm_y;
    FwdArgs a;
};

__device__ __forceinline__ int find_doc_tc(const int32_t* cu, int ndocs, int64_t t) {
    int lo = 0, hi = ndocs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __noinline__ void fail(TcSmall& sh, const FwdArgs& a, uint32_t where) {
    record_error(a.ws, SSD_ERR_TIMEOUT, where);
    *(volatile int*)&sh.abort = 1;
}

// bounded wait; the first role that gives up records why and raises abort
__device__ __forceinline__ bool wait_or_fail(TcSmall& sh, const FwdArgs& a, uint64_t* bar, uint32_t parity,
                                             uint32_t where) {
    if (ptx::mbar_wait(bar, parity, &sh.abort, kWaitNs)) return true;
    if (!*(volatile int*)&sh.abort) fail(sh, a, where);
    return false;
}

// K-major operand (C or B tile, 2 slabs of 64 columns), k-step kk of 16
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk) {
    return ptx::sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
// MN-major operand with one 64-wide block (X, scaled X, incoming state), k-step kk
__device__ __forceinline__ uint64_t desc_mn1(uint32_t base, int kk) {
    return ptx::sdesc_sw128(base + kk * 2048, 8192, 1024);
}
// MN-major operand with two 64-wide blocks (B tile read as B^T), k-step kk
__device__ __forceinline__ uint64_t desc_mn2(uint32_t base, int kk) {
    return ptx::sdesc_sw128(base + kk * 2048, 16384, 1024);
}

// Final states of packed documents that end at row e < nv - 1 of a chunk:
//   S_e[p][n] = 2^{p_e} S_in[p][n] + sum_{j <= e} 2^{seg(e, j)} dt_j x_j[p] B_j[n]
// (seg grown leftwards from the diagonal; -inf log-decays at document starts
// zero the terms of earlier documents).  S_in is read from the bf16
// incoming-state tile.  Rare path, kept out of line: one thread per state
// column n = i, all 128 threads of the state group call it together.
__device__ __noinline__ void doc_end_states(TcSmall& sh, const ChunkMeta& m, const uint8_t* stg,
                                            const uint8_t* sin_tile, float* fin, int H, int h, int nv, int i) {
    const uint8_t* xt = stg + kTileX;
    const uint8_t* bt = stg + kTileB + (i >> 6) * 16384;
    for (int e = 0; e < nv - 1; ++e) {
        if (!(m.rowflag[e] & 2)) continue;
        ptx::named_bar(kBarState, 128);
        if (i == e) {
            float r = 0.f;
            for (int j = e; j >= 0; --j) {
                sh.wv[j] = ex2_approx(r) * m.dtv[j];
                r += m.ell[j];
            }
        }
        ptx::named_bar(kBarState, 128);
        const float pe = m.pexp[e];
        float* fo = fin + ((size_t)m.rowdoc[e] * H + h) * (size_t)(P * N) + i;
#pragma unroll 1
        for (int p = 0; p < P; ++p) {
            float acc = pe * __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sin_tile + sw128_off(i, p)));
#pragma unroll 4
            for (int j = 0; j <= e; ++j) {
                const float xv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(xt + sw128_off(j, p)));
                const float bv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(bt + sw128_off(j, i & 63)));
                acc = fmaf(sh.wv[j] * xv, bv, acc);
            }
            fo[(size_t)p * N] = acc;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) ssd_chunk_tc(const __grid_constant__ TcParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    TcSmall& sh = *reinterpret_cast<TcSmall*>(sm + kTiles);
    const FwdArgs& a = prm.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool full_mode = (a.mode == kModeFull);

    // unit: heads of one (row, split) are adjacent so they share B / C in L2
    const int64_t u = blockIdx.x;
    const int h = (int)(u % a.H);
    const int s = (int)((u / a.H) % a.nsplit);
    const int64_t b = u / ((int64_t)a.H * a.nsplit);
    const int64_t uw = ((b * a.H) + h) * a.nsplit + s;   // workspace slot
    const int g = h / (a.H / a.G);
    const int64_t t0 = (int64_t)s * a.split_len;
    const int64_t t1 = (t0 + a.split_len < a.L) ? t0 + a.split_len : a.L;
    const int nch = (int)((t1 - t0 + Q - 1) / Q);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            ptx::mbar_init(&sh.full[i], 1);
            ptx::mbar_init(&sh.empty[i], 3);   // MMA commit + mask group + state group
        }
        ptx::mbar_init(&sh.barG, 1);
        ptx::mbar_init(&sh.barM, 4);
        ptx::mbar_init(&sh.barDS, 1);
        ptx::mbar_init(&sh.barS, 4);
        ptx::mbar_init(&sh.barY, 1);
        ptx::mbar_init(&sh.dsFree, 4);
        ptx::mbar_init(&sh.barDrain, 1);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sh.yFree[i], 4);
            ptx::mbar_init(&sh.metaFull[i], 4);
            ptx::mbar_init(&sh.metaFree[i], 1);
        }
        sh.abort = 0;
        sh.never = 0;
        sh.doc_cursor = a.cu ? find_doc_tc(a.cu, a.ndocs, t0) : 0;
        ptx::mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&prm.tm_x);
        ptx::prefetch_tmap(&prm.tm_B);
        ptx::prefetch_tmap(&prm.tm_C);
        ptx::prefetch_tmap(&prm.tm_y);
    }
    if (warp == 1) ptx::tmem_alloc(&sh.tmem_base, kTmCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tb = sh.tmem_base;

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int st = c % NS, k = c / NS;
                if (c >= NS && !wait_or_fail(sh, a, &sh.empty[st], (k - 1) & 1, kWhereEmpty)) break;
                const int t = (int)(t0 + (int64_t)c * Q);
                uint8_t* stg = sm + st * kStageBytes;
                ptx::mbar_expect_tx(&sh.full[st], full_mode ? 81920u : 49152u);
                if (full_mode) {
                    ptx::tma_load_4d(stg + kTileC, &prm.tm_C, &sh.full[st], 0, g, t, (int)b);
                    ptx::tma_load_4d(stg + kTileC + 16384, &prm.tm_C, &sh.full[st], 64, g, t, (int)b);
                }
                ptx::tma_load_4d(stg + kTileB, &prm.tm_B, &sh.full[st], 0, g, t, (int)b);
                ptx::tma_load_4d(stg + kTileB + 16384, &prm.tm_B, &sh.full[st], 64, g, t, (int)b);
                ptx::tma_load_4d(stg + kTileX, &prm.tm_x, &sh.full[st], 0, h, t, (int)b);
                ++issued;
            }
            // drain: the last load issued into each stage has landed
            for (int st = 0; st < NS && st < issued; ++st) {
                const int last = ((issued - 1 - st) / NS) * NS + st;
                if (!ptx::mbar_wait(&sh.full[st], (last / NS) & 1, &sh.never, kWaitNs)) fail(sh, a, kWhereDrain);
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idG = ptx::idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idYd = ptx::idesc_bf16(128, 64, 0, 1);
            constexpr uint32_t idYo = ptx::idesc_bf16(128, 64, 0, 1);
            constexpr uint32_t idDS = ptx::idesc_bf16(128, 64, 1, 1);
            const uint32_t xt = ptx::smem_u32(sm + kXt), sin = ptx::smem_u32(sm + kSin);
            auto stage = [&](int c) { return ptx::smem_u32(sm + (c % NS) * kStageBytes); };
            auto issue_G = [&](int c) {
                const uint32_t stg = stage(c);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb + kTmG, desc_k(stg + kTileC, kk), desc_k(stg + kTileB, kk), idG, kk > 0);
                ptx::mma_commit(&sh.barG);
            };
            bool ok = true;
            if (nch > 0 && full_mode) {
                ok = wait_or_fail(sh, a, &sh.full[0], 0, kWhereFull);
                ptx::tc_fence_after();
                if (ok) issue_G(0);
            }
            for (int c = 0; ok && c < nch; ++c) {
                const int st = c % NS;
                const uint32_t stg = stage(c);
                if (!full_mode && !wait_or_fail(sh, a, &sh.full[st], (c / NS) & 1, kWhereFull)) break;
                if (!wait_or_fail(sh, a, &sh.barM, c & 1, kWhereBarM)) break;
                ptx::tc_fence_after();
                if (full_mode) {
                    if (c >= 2 && !wait_or_fail(sh, a, &sh.yFree[c & 1], ((c >> 1) - 1) & 1, kWhereYFree)) break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ts(tb + kTmYd + 64 * (c & 1), tb + kTmM + 8 * kk, desc_mn1(stg + kTileX, kk), idYd,
                                    kk > 0);
                }
                if (c >= 1 && !wait_or_fail(sh, a, &sh.dsFree, (c - 1) & 1, kWhereDsFree)) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb + kTmDS, desc_mn2(stg + kTileB, kk), desc_mn1(xt, kk), idDS, kk > 0);
                ptx::mma_commit(&sh.barDS);
                if (full_mode) {
                    if (c + 1 < nch) {
                        if (!wait_or_fail(sh, a, &sh.full[(c + 1) % NS], ((c + 1) / NS) & 1, kWhereFull)) break;
                        ptx::tc_fence_after();
                        issue_G(c + 1);
                    }
                    if (!wait_or_fail(sh, a, &sh.barS, c & 1, kWhereBarS)) break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ss(tb + kTmYo + 64 * (c & 1), desc_k(stg + kTileC, kk), desc_mn1(sin, kk), idYo,
                                    kk > 0);
                    ptx::mma_commit(&sh.barY);
                }
                ptx::mma_commit(&sh.empty[st]);
            }
            // drain: every MMA issued so far has completed
            ptx::mma_commit(&sh.barDrain);
            if (!ptx::mbar_wait(&sh.barDrain, 0, &sh.never, kWaitNs)) fail(sh, a, kWhereDrain);
        }
    } else if (warp < 6) {
        // ================================================================ mask group
        const int mt = threadIdx.x - 64;          // 0..127
        const int rb = warp & 3;                  // TMEM lane quarter = row block
        const int i = 32 * rb + lane;             // chunk row = TMEM lane
        const uint32_t lane_addr = tb + ((uint32_t)(32 * rb) << 16);
        const float A2 = a.A[h] * kLog2e;
        if (full_mode) {
            // the mask above the diagonal blocks is zero in every chunk: write it once
            uint32_t z[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) z[q] = 0u;
#pragma unroll
            for (int r = 1; r < 4; ++r)
                if (r > rb) ptx::tmem_st16(lane_addr + kTmM + 16 * r, z);
            ptx::tmem_st_wait();
        }
        auto load_dt = [&](int c) -> float {
            const int64_t t = t0 + (int64_t)c * Q;
            return (c < nch && t + i < t1) ? __ldg(a.dt + ((size_t)b * a.L + t + i) * a.H + h) : 0.f;
        };
        float dt_next = load_dt(0);
        for (int c = 0; c < nch; ++c) {
            const int st = c % NS, k = c / NS, mb = c & 1;
            uint8_t* stg = sm + st * kStageBytes;
            const int64_t t = t0 + (int64_t)c * Q;
            const int nv = (int)((t + Q < t1) ? Q : t1 - t);
            const float dti = dt_next;
            dt_next = load_dt(c + 1);
            if (c >= 2) wait_or_fail(sh, a, &sh.metaFree[mb], ((c >> 1) - 1) & 1, kWhereMetaFree);
            // document boundaries: walk forward from the chunk's first document
            int flag = 0, doc = (int)b;
            if (i < nv) {
                if (a.cu) {
                    int d = sh.doc_cursor;
                    while (d + 1 < a.ndocs && __ldg(a.cu + d + 1) <= t + i) ++d;
                    doc = d;
                    if (d > 0 && __ldg(a.cu + d) == t + i) flag |= 1;
                    if (t + i + 1 == __ldg(a.cu + d + 1)) flag |= 2;
                } else if (t + i == a.L - 1) {
                    flag |= 2;
                }
            }
            const float l2 = (flag & 1) ? -INFINITY : dti * A2;
            ChunkMeta& m = sh.meta[mb];
            sh.seg.ell[i] = l2;
            sh.dtv[i] = dti;
            m.ell[i] = l2;
            m.dtv[i] = dti;
            m.rowflag[i] = flag;
            m.rowdoc[i] = doc;
            ptx::named_bar(kBarMask, 128);
            if (mt == Q - 1 && a.cu) sh.doc_cursor = doc;   // the next chunk starts in (or after) this document
            SegsumRow<4> row;
            segsum_phase1<4>(sh.seg, row, rb, lane);
            ptx::named_bar(kBarMask, 128);
            segsum_phase2<4>(sh.seg, row, rb, lane);
            ptx::named_bar(kBarMask, 128);
            sh.colfac[i] = ex2_approx(sh.seg.colS[i]) * dti;
            const float xf = ex2_approx(segsum_chunk_suffix<4>(sh.seg, i)) * dti;
            m.pexp[i] = ex2_approx(row.p);
            if (mt == 0) m.tau = sh.seg.tau;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sh.metaFull[mb]);
            // scaled X (state-summary operand); its buffer and M's are free once dS(c-1) is done
            wait_or_fail(sh, a, &sh.full[st], k & 1, kWhereFull);
            if (c >= 1) wait_or_fail(sh, a, &sh.barDS, (c - 1) & 1, kWhereBarDS);
            {
                const uint8_t* xrow = stg + kTileX;
                uint8_t* xt = sm + kXt;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4*>(xrow + sw128_off(i, 8 * q));
                    uint4 o;
                    o.x = pack_bf16(bf16lo(v.x) * xf, bf16hi(v.x) * xf);
                    o.y = pack_bf16(bf16lo(v.y) * xf, bf16hi(v.y) * xf);
                    o.z = pack_bf16(bf16lo(v.z) * xf, bf16hi(v.z) * xf);
                    o.w = pack_bf16(bf16lo(v.w) * xf, bf16hi(v.w) * xf);
                    *reinterpret_cast<uint4*>(xt + sw128_off(i, 8 * q)) = o;
                }
                ptx::fence_proxy_async();
            }
            ptx::named_bar(kBarMask, 128);        // colfac complete; X tile reads done
            if (mt == 0) ptx::mbar_arrive(&sh.empty[st]);
            if (full_mode) {
                wait_or_fail(sh, a, &sh.barG, c & 1, kWhereBarG);
                ptx::tc_fence_after();
                // rank-one off-diagonal blocks r < rb: row factor x column factor
#pragma unroll 1
                for (int r = 0; r < rb; ++r) {
                    uint32_t gr[32];
                    ptx::tmem_ld32(lane_addr + kTmG + 32 * r, gr);
                    const float Rr = (r == 0) ? row.R[0] : (r == 1) ? row.R[1] : row.R[2];
                    const float rf = ex2_approx(Rr);
                    const float4* cf = reinterpret_cast<const float4*>(sh.colfac + 32 * r);
                    ptx::tmem_ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 f = cf[q];
                        pk[2 * q] = pack_bf16(__uint_as_float(gr[4 * q]) * rf * f.x,
                                              __uint_as_float(gr[4 * q + 1]) * rf * f.y);
                        pk[2 * q + 1] = pack_bf16(__uint_as_float(gr[4 * q + 2]) * rf * f.z,
                                                  __uint_as_float(gr[4 * q + 3]) * rf * f.w);
                    }
                    ptx::tmem_st16(lane_addr + kTmM + 16 * r, pk);
                }
                // 1-SS diagonal block rb: running sums from the diagonal
                {
                    uint32_t gr[32];
                    ptx::tmem_ld32(lane_addr + kTmG + 32 * rb, gr);
                    const float4* dv = reinterpret_cast<const float4*>(sh.dtv + 32 * rb);
                    ptx::tmem_ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 f = dv[q];
                        // every term computed, then masked: no divergent branches
                        float mm[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float v = __uint_as_float(gr[4 * q + e]) * ex2_approx(row.d[4 * q + e]);
                            mm[e] = (4 * q + e <= lane) ? v : 0.f;
                        }
                        const float m0 = mm[0] * f.x, m1 = mm[1] * f.y, m2 = mm[2] * f.z, m3 = mm[3] * f.w;
                        pk[2 * q] = pack_bf16(m0, m1);
                        pk[2 * q + 1] = pack_bf16(m2, m3);
                    }
                    ptx::tmem_st16(lane_addr + kTmM + 16 * rb, pk);
                }
                ptx::tmem_st_wait();
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sh.barM);
            if (ptx::named_bar_any(kBarMask, 128, *(volatile int*)&sh.abort != 0)) break;
        }
    } else {
        // ================================================================ state group
        const int mt = threadIdx.x - 192;         // 0..127
        const int rb = warp & 3;
        const int i = 32 * rb + lane;             // chunk row = TMEM lane = state column n
        const uint32_t lane_addr = tb + ((uint32_t)(32 * rb) << 16);
        const float Dh = a.D ? a.D[h] : 0.f;
        const size_t PN = (size_t)P * N;
        float S[P];
        if (full_mode && a.nsplit > 1 && s > 0) {
#pragma unroll
            for (int p = 0; p < P; ++p) S[p] = a.ws_state[uw * PN + (size_t)p * N + i];
        } else if (s == 0 && a.init && !a.cu) {
#pragma unroll
            for (int p = 0; p < P; ++p) S[p] = a.init[((size_t)b * a.H + h) * PN + (size_t)p * N + i];
        } else {
#pragma unroll
            for (int p = 0; p < P; ++p) S[p] = 0.f;
        }
        auto write_sin = [&]() {
            uint8_t* sin = sm + kSin;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint4 sv;
                sv.x = pack_bf16(S[8 * q + 0], S[8 * q + 1]);
                sv.y = pack_bf16(S[8 * q + 2], S[8 * q + 3]);
                sv.z = pack_bf16(S[8 * q + 4], S[8 * q + 5]);
                sv.w = pack_bf16(S[8 * q + 6], S[8 * q + 7]);
                *reinterpret_cast<uint4*>(sin + sw128_off(i, 8 * q)) = sv;
            }
            ptx::fence_proxy_async();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sh.barS);
        };
        if (full_mode && nch > 0) write_sin();
        float tau_split = 0.f;
        for (int c = 0; c < nch; ++c) {
            const int st = c % NS, k = c / NS, mb = c & 1;
            uint8_t* stg = sm + st * kStageBytes;
            const int64_t t = t0 + (int64_t)c * Q;
            const int nv = (int)((t + Q < t1) ? Q : t1 - t);
            wait_or_fail(sh, a, &sh.metaFull[mb], (c >> 1) & 1, kWhereMetaFull);
            const ChunkMeta& m = sh.meta[mb];
            // ---- packed documents that end inside this chunk: their final states
            if (full_mode && a.fin && a.cu) {
                bool any = false;
                for (int e = 0; e < nv - 1; ++e) any |= (m.rowflag[e] & 2) != 0;
                if (any) {
                    wait_or_fail(sh, a, &sh.full[st], k & 1, kWhereFull);
                    doc_end_states(sh, m, stg, sm + kSin, a.fin, a.H, h, nv, i);
                }
            }
            // ---- state update: S = 2^tau S + dS (TMEM lane = state column n)
            wait_or_fail(sh, a, &sh.barDS, c & 1, kWhereBarDS);
            ptx::tc_fence_after();
            {
                uint32_t ds0[32], ds1[32];
                ptx::tmem_ld32(lane_addr + kTmDS, ds0);
                ptx::tmem_ld32(lane_addr + kTmDS + 32, ds1);
                ptx::tmem_ld_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sh.dsFree);
                const float tau2 = m.tau;
                const float ed = ex2_approx(tau2);
                tau_split += tau2;
#pragma unroll
                for (int q = 0; q < 32; ++q) S[q] = fmaf(ed, S[q], __uint_as_float(ds0[q]));
#pragma unroll
                for (int q = 0; q < 32; ++q) S[32 + q] = fmaf(ed, S[32 + q], __uint_as_float(ds1[q]));
            }
            if (full_mode && a.fin && (m.rowflag[nv - 1] & 2)) {
                float* fo = a.fin + ((size_t)m.rowdoc[nv - 1] * a.H + h) * PN + i;
#pragma unroll
                for (int p = 0; p < P; ++p) fo[(size_t)p * N] = S[p];
            }
            if (full_mode) {
                // Yoff(c) has read the incoming-state tile: stage the next one, then the outputs of c
                wait_or_fail(sh, a, &sh.barY, c & 1, kWhereBarY);
                ptx::tc_fence_after();
                if (c + 1 < nch) write_sin();
                wait_or_fail(sh, a, &sh.full[st], k & 1, kWhereFull);
                if (mt == 0) ptx::bulk_wait_read0();   // the previous y store has read the staging tile
                ptx::named_bar(kBarState, 128);
                const uint8_t* xrow = stg + kTileX;
                uint8_t* ys = sm + kYs;
                const float pe = m.pexp[i];
                const uint32_t yd_addr = lane_addr + kTmYd + 64 * (c & 1);
                const uint32_t yo_addr = lane_addr + kTmYo + 64 * (c & 1);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t yd[32], yo[32];
                    ptx::tmem_ld32(yd_addr + 32 * half, yd);
                    ptx::tmem_ld32(yo_addr + 32 * half, yo);
                    ptx::tmem_ld_wait();
                    if (half == 1) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(&sh.yFree[c & 1]);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int e0 = 32 * half + 8 * q;
                        const uint4 v = *reinterpret_cast<const uint4*>(xrow + sw128_off(i, e0));
                        const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
                        uint32_t ow[4];
#pragma unroll
                        for (int w2 = 0; w2 < 4; ++w2) {
                            const int e = 8 * q + 2 * w2;
                            float y0 = fmaf(pe, __uint_as_float(yo[e]), __uint_as_float(yd[e]));
                            float y1 = fmaf(pe, __uint_as_float(yo[e + 1]), __uint_as_float(yd[e + 1]));
                            y0 = fmaf(Dh, bf16lo(xw[w2]), y0);
                            y1 = fmaf(Dh, bf16hi(xw[w2]), y1);
                            ow[w2] = pack_bf16(y0, y1);
                        }
                        *reinterpret_cast<uint4*>(ys + sw128_off(i, e0)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                }
                ptx::fence_proxy_async();
                ptx::named_bar(kBarState, 128);
                if (mt == 0) {
                    ptx::tma_store_4d(&prm.tm_y, ys, 0, h, (int)t, (int)b);
                    ptx::bulk_commit();
                }
            }
            // release the chunk's meta and input stage
            ptx::named_bar(kBarState, 128);
            if (mt == 0) {
                ptx::mbar_arrive(&sh.metaFree[mb]);
                ptx::mbar_arrive(&sh.empty[st]);
            }
            if (ptx::named_bar_any(kBarState, 128, *(volatile int*)&sh.abort != 0)) break;
        }
        if (!full_mode && !*(volatile int*)&sh.abort) {
#pragma unroll
            for (int p = 0; p < P; ++p) a.ws_state[uw * PN + (size_t)p * N + i] = S[p];
            if (mt == 0) a.ws_tau[uw] = tau_split * kLn2;
        }
        if (mt == 0) ptx::bulk_wait0();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tb, kTmCols);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// 4-D map over a (batch, L, heads_or_groups, inner) bf16 tensor; box = one
// 64-element x 128-row tile of one head (group), 128-byte swizzle.
bool encode_4d(CUtensorMap* tm, const void* base, int64_t inner, int64_t mid, int64_t L, int64_t batch) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)mid, (cuuint64_t)L, (cuuint64_t)batch};
    cuuint64_t strides[3] = {(cuuint64_t)(inner * 2), (cuuint64_t)(inner * mid * 2),
                             (cuuint64_t)(inner * mid * L * 2)};
    cuuint32_t box[4] = {64, 1, 128, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

size_t tc_smem_bytes() { return 1024 + kTiles + sizeof(TcSmall); }

bool tc_supported(int P_, int N_, int Q_, int dtype) {
    return P_ == P && N_ == N && Q_ == Q && dtype == SSD_BF16;
}

cudaError_t launch_tc(const FwdArgs& a, cudaStream_t st) {
    TcParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.a = a;
    if (!encode_4d(&prm.tm_x, a.x, P, a.H, a.L, a.batch) || !encode_4d(&prm.tm_y, a.y, P, a.H, a.L, a.batch) ||
        !encode_4d(&prm.tm_B, a.B, N, a.G, a.L, a.batch) || !encode_4d(&prm.tm_C, a.C, N, a.G, a.L, a.batch))
        return cudaErrorInvalidValue;
    const size_t smem = tc_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(ssd_chunk_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = a.batch * a.H * a.nsplit;
    ssd_chunk_tc<<<(unsigned)grid, kThreads, smem, st>>>(prm);
    return cudaGetLastError();
}

}  // namespace ssd
