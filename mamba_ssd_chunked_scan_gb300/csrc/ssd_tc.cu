// Tensor-core (tcgen05 / TMEM / TMA) kernel of the chunked SSD forward pass
// for the Mamba-2 head shape: chunk Q = 128, head dim P = 64, state N = 128,
// bf16 x / B / C / y, fp32 dt / A / D / states, fp32 accumulation.
//
// One CTA walks the chunks of one (batch row, head, split) unit and keeps the
// P x N state on chip between chunks ("State Space Duality and Mamba-2",
// "The SSD Block Decomposition Algorithm"; "NVIDIA Accelerates Mamba-2
// Forward Kernel with CUDA Tile": intra-block parallel, inter-block
// recurrent, state resident on chip).  Per chunk:
//
//   G     = C B^T                        (UMMA 128x128x128, TMEM)
//   M     = G o L o dt                   (hierarchy-aware segsum mask, bf16, TMEM)
//   Ydiag = M X                          (UMMA, A operand from TMEM)
//   Yoff  = C S_in^T                     (UMMA; row decay exp(p_i) in the epilogue)
//   dS    = B^T (exp(s_j) dt_j x_j)      (UMMA, chunk state summary)
//   y     = Ydiag + exp(p_i) Yoff + D x  (epilogue, TMA store)
//   S     = exp(tau) S + dS              (state carried in registers)
//
// Warp roles: warp 0 issues TMA loads (two-stage ring), warp 1 owns TMEM and
// issues the MMAs, warps 2-5 (one thread per chunk row = TMEM lane) do the
// segsum, the mask, the scaled X tile, the epilogue and the state update.
// Every wait is bounded; a wait that runs out records SSD_ERR_TIMEOUT in the
// workspace status word and the CTA drains its copies, frees TMEM and exits.
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
constexpr int NS = 2;                     // input stages
constexpr int kThreads = 192;
constexpr uint32_t kTileC = 0, kTileB = 32768, kTileX = 65536, kStageBytes = 81920;
constexpr uint32_t kXt = NS * kStageBytes;   // scaled X for the state summary
constexpr uint32_t kSin = kXt + 16384;       // incoming state, bf16, (n rows, p)
constexpr uint32_t kYs = kSin + 16384;       // y staging for the TMA store
constexpr uint32_t kTiles = kYs + 16384;
constexpr uint32_t kTmG = 0, kTmM = 128, kTmYd = 192, kTmYo = 256, kTmDS = 320, kTmCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr float kLn2 = 0.6931471805599453f;

// codes of the wait that gave up (WsHeader::where)
enum : uint32_t { kWhereEmpty = 1, kWhereFullMma = 2, kWhereBarM = 3, kWhereFullMath = 4, kWhereBarG = 5,
                  kWhereBarY = 6, kWhereDrain = 7 };

struct TcSmall {
    SegsumShared<4> seg;
    alignas(16) float dtv[Q];      // read as float4
    alignas(16) float colfac[Q];   // read as float4
    alignas(16) float wv[Q];
    float pexp_e;
    int rowflag[Q];     // bit0: a document starts at this token, bit1: a document ends here
    int rowdoc[Q];      // state index (document, or batch row) of this token
    uint64_t full[NS], empty[NS];
    uint64_t barG, barM, barY, barDrain;
    uint32_t tmem_base;
    int abort;
    int never;          // stays 0: lets drain waits ignore the abort flag
};

static_assert(offsetof(TcSmall, dtv) % 16 == 0 && offsetof(TcSmall, colfac) % 16 == 0,
              "vector-loaded arrays must be 16-byte aligned");
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

__device__ void fail(TcSmall& sh, const FwdArgs& a, uint32_t where) {
    record_error(a.ws, SSD_ERR_TIMEOUT, where);
    *(volatile int*)&sh.abort = 1;
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
            ptx::mbar_init(&sh.empty[i], 2);
        }
        ptx::mbar_init(&sh.barG, 1);
        ptx::mbar_init(&sh.barM, 4);
        ptx::mbar_init(&sh.barY, 1);
        ptx::mbar_init(&sh.barDrain, 1);
        sh.abort = 0;
        sh.never = 0;
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
    const volatile int* abort = &sh.abort;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int st = c % NS, k = c / NS;
                if (c >= NS && !ptx::mbar_wait(&sh.empty[st], (k - 1) & 1, abort, kWaitNs)) {
                    if (!*abort) fail(sh, a, kWhereEmpty);
                    break;
                }
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
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idG = ptx::idesc_bf16(128, 128, 0, 0);
            const uint32_t idYd = ptx::idesc_bf16(128, 64, 0, 1);
            const uint32_t idYo = ptx::idesc_bf16(128, 64, 0, 1);
            const uint32_t idDS = ptx::idesc_bf16(128, 64, 1, 1);
            const uint32_t xt = ptx::smem_u32(sm + kXt), sin = ptx::smem_u32(sm + kSin);
            for (int c = 0; c < nch; ++c) {
                const int st = c % NS, k = c / NS;
                const uint32_t stg = ptx::smem_u32(sm + st * kStageBytes);
                if (!ptx::mbar_wait(&sh.full[st], k & 1, abort, kWaitNs)) {
                    if (!*abort) fail(sh, a, kWhereFullMma);
                    break;
                }
                ptx::tc_fence_after();
                if (full_mode) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                        ptx::mma_ss(tb + kTmG, ptx::sdesc_sw128(stg + kTileC + koff, 16, 1024),
                                    ptx::sdesc_sw128(stg + kTileB + koff, 16, 1024), idG, kk > 0);
                    }
                    ptx::mma_commit(&sh.barG);
                }
                if (!ptx::mbar_wait(&sh.barM, c & 1, abort, kWaitNs)) {
                    if (!*abort) fail(sh, a, kWhereBarM);
                    break;
                }
                ptx::tc_fence_after();
                if (full_mode) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ts(tb + kTmYd, tb + kTmM + 8 * kk,
                                    ptx::sdesc_sw128(stg + kTileX + kk * 2048, 8192, 1024), idYd, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                        ptx::mma_ss(tb + kTmYo, ptx::sdesc_sw128(stg + kTileC + koff, 16, 1024),
                                    ptx::sdesc_sw128(sin + kk * 2048, 8192, 1024), idYo, kk > 0);
                    }
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb + kTmDS, ptx::sdesc_sw128(stg + kTileB + kk * 2048, 16384, 1024),
                                ptx::sdesc_sw128(xt + kk * 2048, 8192, 1024), idDS, kk > 0);
                ptx::mma_commit(&sh.barY);
                ptx::mma_commit(&sh.empty[st]);
            }
            // drain: every MMA issued so far has completed
            ptx::mma_commit(&sh.barDrain);
            if (!ptx::mbar_wait(&sh.barDrain, 0, &sh.never, kWaitNs))
                fail(sh, a, kWhereDrain);
        }
    } else {
        // ------------------------------------------------------------ math warps
        const int mt = threadIdx.x - 64;          // 0..127
        const int rb = warp & 3;                  // TMEM lane quarter = row block
        const int i = 32 * rb + lane;             // chunk row = TMEM lane = state column n
        const uint32_t lane_addr = tb + ((uint32_t)(32 * rb) << 16);
        const float A2 = a.A[h] * kLog2e;
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
        // the mask above the diagonal blocks is zero in every chunk: write it once
        if (full_mode) {
            uint32_t z[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) z[q] = 0u;
#pragma unroll
            for (int r = 1; r < 4; ++r)
                if (r > rb) ptx::tmem_st16(lane_addr + kTmM + 16 * r, z);
            ptx::tmem_st_wait();
        }
        float tau_split = 0.f;
        for (int c = 0; c < nch; ++c) {
            const int st = c % NS, k = c / NS;
            uint8_t* stg = sm + st * kStageBytes;
            const int64_t t = t0 + (int64_t)c * Q;
            const int nv = (int)((t + Q < t1) ? Q : t1 - t);
            // per-row inputs: step size, log2-decay, document boundaries
            float dti = 0.f;
            int flag = 0, doc = (int)b;
            if (i < nv) {
                dti = a.dt[((size_t)b * a.L + t + i) * a.H + h];
                if (a.cu) {
                    doc = find_doc_tc(a.cu, a.ndocs, t + i);
                    if (doc > 0 && __ldg(a.cu + doc) == t + i) flag |= 1;
                    if (t + i + 1 == __ldg(a.cu + doc + 1)) flag |= 2;
                } else if (t + i == a.L - 1) {
                    flag |= 2;
                }
            }
            const float l2 = (flag & 1) ? -INFINITY : dti * A2;
            sh.seg.ell[i] = l2;
            sh.dtv[i] = dti;
            sh.rowflag[i] = flag;
            sh.rowdoc[i] = doc;
            ptx::named_bar(1, 128);
            SegsumRow<4> row;
            segsum_phase1<4>(sh.seg, row, rb, lane);
            ptx::named_bar(1, 128);
            segsum_phase2<4>(sh.seg, row, rb, lane);
            ptx::named_bar(1, 128);
            sh.colfac[i] = ex2_approx(sh.seg.colS[i]) * dti;
            const float xf = ex2_approx(segsum_chunk_suffix<4>(sh.seg, i)) * dti;
            if (!ptx::mbar_wait(&sh.full[st], k & 1, abort, kWaitNs) && !*abort) fail(sh, a, kWhereFullMath);
            // scaled X row (state summary operand) and the incoming state (bf16)
            {
                const uint8_t* xrow = stg + kTileX;
                uint8_t* xt = sm + kXt;
                uint8_t* sin = sm + kSin;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4*>(xrow + sw128_off(i, 8 * q));
                    uint4 o;
                    o.x = pack_bf16(bf16lo(v.x) * xf, bf16hi(v.x) * xf);
                    o.y = pack_bf16(bf16lo(v.y) * xf, bf16hi(v.y) * xf);
                    o.z = pack_bf16(bf16lo(v.z) * xf, bf16hi(v.z) * xf);
                    o.w = pack_bf16(bf16lo(v.w) * xf, bf16hi(v.w) * xf);
                    *reinterpret_cast<uint4*>(xt + sw128_off(i, 8 * q)) = o;
                    uint4 sv;
                    sv.x = pack_bf16(S[8 * q + 0], S[8 * q + 1]);
                    sv.y = pack_bf16(S[8 * q + 2], S[8 * q + 3]);
                    sv.z = pack_bf16(S[8 * q + 4], S[8 * q + 5]);
                    sv.w = pack_bf16(S[8 * q + 6], S[8 * q + 7]);
                    *reinterpret_cast<uint4*>(sin + sw128_off(i, 8 * q)) = sv;
                }
                ptx::fence_proxy_async();
            }
            if (ptx::named_bar_any(1, 128, *abort != 0)) break;
            if (full_mode) {
                if (!ptx::mbar_wait(&sh.barG, c & 1, abort, kWaitNs) && !*abort) fail(sh, a, kWhereBarG);
                ptx::tc_fence_after();
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r <= rb) {
                        uint32_t gr[32];
                        ptx::tmem_ld32(lane_addr + kTmG + 32 * r, gr);
                        ptx::tmem_ld_wait();
                        uint32_t pk[16];
                        if (r < rb) {
                            const float rf = ex2_approx(row.R[r]);
                            const float4* cf = reinterpret_cast<const float4*>(sh.colfac + 32 * r);
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 f = cf[q];
                                pk[2 * q] = pack_bf16(__uint_as_float(gr[4 * q]) * rf * f.x,
                                                      __uint_as_float(gr[4 * q + 1]) * rf * f.y);
                                pk[2 * q + 1] = pack_bf16(__uint_as_float(gr[4 * q + 2]) * rf * f.z,
                                                          __uint_as_float(gr[4 * q + 3]) * rf * f.w);
                            }
                        } else {
                            const float4* dv = reinterpret_cast<const float4*>(sh.dtv + 32 * r);
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 f = dv[q];
                                const float m0 = (4 * q + 0 <= lane) ? __uint_as_float(gr[4 * q + 0]) * ex2_approx(row.d[4 * q + 0]) * f.x : 0.f;
                                const float m1 = (4 * q + 1 <= lane) ? __uint_as_float(gr[4 * q + 1]) * ex2_approx(row.d[4 * q + 1]) * f.y : 0.f;
                                const float m2 = (4 * q + 2 <= lane) ? __uint_as_float(gr[4 * q + 2]) * ex2_approx(row.d[4 * q + 2]) * f.z : 0.f;
                                const float m3 = (4 * q + 3 <= lane) ? __uint_as_float(gr[4 * q + 3]) * ex2_approx(row.d[4 * q + 3]) * f.w : 0.f;
                                pk[2 * q] = pack_bf16(m0, m1);
                                pk[2 * q + 1] = pack_bf16(m2, m3);
                            }
                        }
                        ptx::tmem_st16(lane_addr + kTmM + 16 * r, pk);
                    }
                }
                ptx::tmem_st_wait();
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sh.barM);
            // ---- epilogue: outputs of this chunk
            if (!ptx::mbar_wait(&sh.barY, c & 1, abort, kWaitNs) && !*abort) fail(sh, a, kWhereBarY);
            ptx::tc_fence_after();
            if (full_mode) {
                if (mt == 0) ptx::bulk_wait_read0();   // the previous y store has read the staging tile
                ptx::named_bar(1, 128);
                const float pe = ex2_approx(row.p);
                const uint8_t* xrow = stg + kTileX;
                uint8_t* ys = sm + kYs;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t yd[32], yo[32];
                    ptx::tmem_ld32(lane_addr + kTmYd + 32 * half, yd);
                    ptx::tmem_ld32(lane_addr + kTmYo + 32 * half, yo);
                    ptx::tmem_ld_wait();
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
                ptx::named_bar(1, 128);
                if (mt == 0) {
                    ptx::tma_store_4d(&prm.tm_y, ys, 0, h, (int)t, (int)b);
                    ptx::bulk_commit();
                }
            }
            // ---- packed documents that end inside this chunk: their final states
            if (full_mode && a.fin && a.cu) {
                for (int e = 0; e < nv - 1; ++e) {
                    if (!(sh.rowflag[e] & 2)) continue;
                    ptx::named_bar(1, 128);
                    if (i == e) {
                        // weights exp2(seg(e, j)) dt_j exactly as the mask forms them
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            if (r < rb) {
                                const float rf = ex2_approx(row.R[r]);
                                for (int cc = 0; cc < 32; ++cc) sh.wv[32 * r + cc] = rf * sh.colfac[32 * r + cc];
                            } else if (r == rb) {
#pragma unroll
                                for (int cc = 0; cc < 32; ++cc)
                                    sh.wv[32 * r + cc] = (cc <= lane) ? ex2_approx(row.d[cc]) * sh.dtv[32 * r + cc] : 0.f;
                            }
                        }
                        sh.pexp_e = ex2_approx(row.p);
                    }
                    ptx::named_bar(1, 128);
                    const float pe = sh.pexp_e;
                    const uint8_t* xt = stg + kTileX;
                    const uint8_t* bt = stg + kTileB + (i >> 6) * 16384;
                    float* fo = a.fin + ((size_t)sh.rowdoc[e] * a.H + h) * PN + i;
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        float acc = pe * S[p];
                        for (int j = 0; j <= e; ++j) {
                            const float xv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(xt + sw128_off(j, p)));
                            const float bv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(bt + sw128_off(j, i & 63)));
                            acc = fmaf(sh.wv[j] * xv, bv, acc);
                        }
                        fo[(size_t)p * N] = acc;
                    }
                }
            }
            ptx::named_bar(1, 128);   // all reads of this input stage are done
            if (mt == 0) ptx::mbar_arrive(&sh.empty[st]);
            // ---- state update: S = exp(tau) S + dS (TMEM lane = state column n)
            {
                const float tau2 = sh.seg.tau;
                const float ed = ex2_approx(tau2);
                tau_split += tau2;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t ds[32];
                    ptx::tmem_ld32(lane_addr + kTmDS + 32 * half, ds);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 32; ++q) S[32 * half + q] = fmaf(ed, S[32 * half + q], __uint_as_float(ds[q]));
                }
            }
            if (full_mode && a.fin && (sh.rowflag[nv - 1] & 2)) {
                float* fo = a.fin + ((size_t)sh.rowdoc[nv - 1] * a.H + h) * PN + i;
#pragma unroll
                for (int p = 0; p < P; ++p) fo[(size_t)p * N] = S[p];
            }
            ptx::tc_fence_before();
            if (ptx::named_bar_any(1, 128, *abort != 0)) break;
        }
        if (!full_mode && !*abort) {
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
