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
//   M     = G o L o dt + D I             (hierarchy-aware segsum mask, bf16,
//                                         written over G in TMEM; the skip
//                                         term D x rides on the diagonal)
//   Ydiag = M X                          (UMMA, A operand from TMEM)
//   dS    = B^T (exp(s_j) dt_j x_j)      (UMMA, chunk state summary)
//   Yoff  = C S_in^T                     (UMMA; the row decay exp(p_i) is applied in the epilogue)
//   S     = exp(tau) S + dS              (state carried in registers)
//   y     = Ydiag + exp(p_i) Yoff        (epilogue, TMA store)
//
// Warpgroups (512 threads; register budgets rebalanced with setmaxnreg):
//   WG0  warp 0: TMA producer; warp 1: issues dS; warp 2: issues G; warp 3: issues Ydiag
//   WG1  mask group for even chunks, WG2 mask group for odd chunks:
//        log-decays, segsum, scaled X tile, mask M, and the chunk's epilogue
//   WG3  state group: state update, incoming-state tile, issues Yoff
// Chunk c uses input stage, G/M buffer and scaled-X buffer c & 1, so the two
// mask groups work on consecutive chunks concurrently; the only serial
// dependency, the state recurrence, is a short loop through the state group.
// One thread of each math group owns one chunk row (= TMEM lane).
//
// Every wait is bounded (FwdArgs::wait_iters polls, and 2 s); a wait that
// runs out records SSD_ERR_TIMEOUT in the workspace status word, and the CTA
// drains its copies, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
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
constexpr int NMETA = 3;                     // per-chunk value buffers between the math groups
constexpr int kPersistChunks = 4;            // units of at most this many chunks run on a persistent grid
constexpr int kThreads = 512;
// setmaxnreg budgets: issue warpgroup (unit bookkeeping of the producer, MMA
// issue) and each math warpgroup
constexpr int kRegsIssue = 72, kRegsMath = 144;   // 128 * (72 + 3 * 144) = 64512 <= 65536 = 512 * 128
static_assert(128 * (kRegsIssue + 3 * kRegsMath) <= kThreads * 128, "register split must fit the launch total");
constexpr uint32_t kTileC = 0, kTileB = 32768, kTileX = 65536, kStageBytes = 81920;
constexpr uint32_t kXt = 2 * kStageBytes;    // scaled X for the state summary, two buffers
constexpr uint32_t kSin = kXt + 2 * 16384;   // incoming state, bf16, (n rows, p)
constexpr uint32_t kTiles = kSin + 16384;
// TMEM columns: G/M/Ydiag [2] (G, then M in cols 0-63 and Ydiag in 64-127) | Yoff [2] | dS |
// C init_d^T (packed documents with initial states)
constexpr uint32_t kTmGM = 0, kTmYo = 256, kTmDS = 384, kTmInit = 448, kTmCols = 512;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kBarMask0 = 1, kBarState = 3;  // named barriers: mask groups 1 and 2, state group 3

// codes of the wait that gave up (WsHeader::where)
enum : uint32_t {
    kWhereEmpty = 1, kWhereFull = 2, kWhereBarM = 3, kWhereYFree = 4, kWhereDsFree = 5, kWhereBarXt = 6,
    kWhereMetaFree = 7, kWhereBarDS = 8, kWhereBarG = 9, kWhereMetaFull = 10, kWhereBarY = 11,
    kWhereDrain = 12, kWhereBarYd = 13, kWhereBarInit = 14, kWhereBarFix = 15
};

// Per-chunk values handed from a mask group to the state group.
struct ChunkMeta {
    alignas(16) float pexp[Q];   // 2^{p_i}: decay of the incoming state at row i
    alignas(16) float ell[Q];    // log2-decays
    alignas(16) float dtv[Q];
    int rowflag[Q];              // bit0: a document starts at this token, bit1: one ends here
    int rowdoc[Q];               // state index (document, or batch row)
    float tau;                   // whole-chunk log2-decay (aggregate pass)
    float tauexp;                // 2^tau
};

// Scratch of one mask group.  The segsum runs in the linear domain (the
// hierarchy-aware routine segsum_lin_* of segsum.cuh): a_k = 2^{l_k}, exactly
// 0 at a document start, and the mask needs one exp2 per token instead of
// one per entry.
struct MaskScratch {
    SegsumLinShared<4> seg;        // a_k in, column factors, block totals, last-row factors out
    alignas(16) float dtv[Q];      // read as float4
    alignas(16) float colfac[Q];   // colL[j] dt_j, read as float4
    float totLog[4];               // block sums of the log2-decays (aggregate pass)
    int doc_cursor;
};

struct TcSmall {
    MaskScratch mask[2];
    ChunkMeta meta[NMETA];
    alignas(16) float wv[Q];
    uint64_t full[2], empty[2];
    uint64_t barG[2], barM[2], barXt[2], barYd[2], barDS[2], barY[2], yFree[2];
    uint64_t dsFree;
    uint64_t metaFull[NMETA], metaFree[NMETA];
    uint64_t drain[4];
    uint64_t barInit;              // C init_d^T of one document start is in TMEM
    uint64_t barFix[2];            // the state group has rewritten the Yoff rows of a chunk
    uint32_t startmask[4];         // per warp: rows where a document starts (state group)
    uint32_t endmask[4];           // per warp: rows e < nv - 1 where a document ends (state group)
    uint32_t evflags[4];           // per state-group warp: OR of (stale meta, a document end, a start)
    float segtot[4];               // per warp: log2-decay sum of the warp's last document segment
    float qlast, qend;             // initial-state decay at the chunk's last row / at a document end
    int dlast;                     // the document open at the chunk's last row, if it started in the chunk
    uint32_t tmem_base;
    int abort;
    int never;                     // stays 0: lets drain waits ignore the abort flag
};

static_assert(sizeof(MaskScratch) % 16 == 0, "mask scratch keeps 16-byte alignment");
static_assert(offsetof(MaskScratch, seg) % 16 == 0 && offsetof(MaskScratch, dtv) % 16 == 0 &&
                  offsetof(MaskScratch, colfac) % 16 == 0,
              "vector-accessed arrays must be 16-byte aligned");
static_assert(offsetof(TcSmall, meta) % 16 == 0 && sizeof(ChunkMeta) % 16 == 0, "meta alignment");
static_assert(offsetof(TcSmall, full) % 8 == 0, "mbarriers are 8-byte aligned");
static_assert(kTiles % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");

constexpr size_t kSmemBytes = 1024 + kTiles + sizeof(TcSmall);
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

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
__device__ __forceinline__ uint32_t pack_bf16_2(uint64_t v) {
    float lo, hi;
    ptx::f2_unpack(v, lo, hi);
    return pack_bf16(lo, hi);
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void fail(TcSmall& sh, const FwdArgs& a, uint32_t where) {
    record_error(a.ws, SSD_ERR_TIMEOUT, where);
    *(volatile int*)&sh.abort = 1;
}

// bounded wait; the first role that gives up records why and raises abort
__device__ __forceinline__ bool wait_or_fail(TcSmall& sh, const FwdArgs& a, uint64_t* bar, uint32_t parity,
                                             uint32_t where) {
    if (ptx::mbar_wait(bar, parity, &sh.abort, a.wait_iters)) return true;
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

// Final state of a packed document that ends at row e < nv - 1 of a chunk:
//   S_e = 2^{p_e} S_in + q_e init_d + D_e,   D_e^T = B^T X~,
//   X~_j = w_j x_j,  w_j = 2^{seg(e, j)} dt_j for j <= e, else 0
// (the chunk state summary's contraction with row e's decays in place of the
// chunk end's; -inf log-decays at document starts zero the terms of earlier
// documents, and 2^{p_e} = 0 once one started in the chunk).  This computes
// D_e on the tensor cores: seg(e, j) = sum_{k=j+1..e} l_k from a reverse scan
// over the rows (no prefix subtraction), X~ staged as bf16 in the
// incoming-state tile (which Yoff has finished reading), one UMMA into the
// spare TMEM columns (lane n, column p).  It also leaves in sh.qend the decay
// q_e = 2^{seg(e, st) + l_st} of d's initial state when d started in this
// chunk at row st and the call has initial states, else 0; the caller adds
// 2^{p_e} S_in (its fp32 registers) and q_e init_d.  All 128 threads of the
// state group call it together (thread i = row i).  Inlined, and only into the
// kernel instance for document events: out of line, the caller's 64-register
// state had to be saved around the call, which made every chunk slower.
__device__ __forceinline__ void doc_end_mma(TcSmall& sh, const FwdArgs& a, const ChunkMeta& m, const uint8_t* stg,
                                         uint8_t* sin_tile, uint32_t tb, int e, float A2, int i, int& init_cnt) {
    constexpr uint32_t idDS = ptx::idesc_bf16(128, 64, 1, 1);
    const int lane = i & 31, rb = i >> 5;
    // reverse inclusive scan of v_j = l_{j+1} (j < e): s_j = sum_{k=j+1..e} l_k
    float v = (i < e) ? m.ell[i + 1] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_down_sync(0xffffffffu, v, o);
        if (lane + o < 32) v = v + t;
    }
    if (lane == 0) sh.segtot[rb] = v;
    if (i == 0) sh.qend = 0.f;
    ptx::named_bar(kBarState, 128);
    for (int r = rb + 1; r < 4; ++r) v = v + sh.segtot[r];
    if (a.init && i <= e && (m.rowflag[i] & 1) && m.rowdoc[i] == m.rowdoc[e])
        sh.qend = ex2_approx(v + m.dtv[i] * A2);
    const float w = (i <= e) ? ex2_approx(v) * m.dtv[i] : 0.f;
    {
        // X~ row i = w_i x_i, in the layout of the scaled-X operand
        const uint8_t* xrow = stg + kTileX;
        const uint64_t w2 = ptx::f2_pack(w, w);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xrow + sw128_off(i, 8 * q));
            uint4 o;
            o.x = pack_bf16_2(ptx::f2_mul(ptx::f2_pack(bf16lo(xv.x), bf16hi(xv.x)), w2));
            o.y = pack_bf16_2(ptx::f2_mul(ptx::f2_pack(bf16lo(xv.y), bf16hi(xv.y)), w2));
            o.z = pack_bf16_2(ptx::f2_mul(ptx::f2_pack(bf16lo(xv.z), bf16hi(xv.z)), w2));
            o.w = pack_bf16_2(ptx::f2_mul(ptx::f2_pack(bf16lo(xv.w), bf16hi(xv.w)), w2));
            *reinterpret_cast<uint4*>(sin_tile + sw128_off(i, 8 * q)) = o;
        }
        ptx::fence_proxy_async();
    }
    ptx::named_bar(kBarState, 128);
    if (i == 0) {
        ptx::tc_fence_after();
        const uint32_t bt = ptx::smem_u32(stg + kTileB), xt = ptx::smem_u32(sin_tile);
#pragma unroll 1
        for (int kk = 0; kk < 8; ++kk) ptx::mma_ss(tb + kTmInit, desc_mn2(bt, kk), desc_mn1(xt, kk), idDS, kk > 0);
        ptx::mma_commit(&sh.barInit);
    }
    wait_or_fail(sh, a, &sh.barInit, (uint32_t)(init_cnt & 1), kWhereBarInit);
    ++init_cnt;
    ptx::tc_fence_after();
}

// Rows of a chunk in which documents with initial states start.  Row i of
// document d, which started at row st of this chunk, takes its state term
// from d's initial state, decayed from the start:
//   q_i C_i init_d^T,   q_i = 2^{sum_{k=st..i} l_k}
// (the start token applies its own decay l_st: h_st = a_st init_d + dt_st
// x_st B_st^T), where the carried state's term 2^{p_i} C_i S_in^T is 0 (the
// -inf log-decay at st is in p_i).  The state group rewrites the chunk's Yoff
// accumulator rows in TMEM to the finished state terms: 2^{p_i} Yoff_i for
// the rows before the first start, q_i C_i init_d^T after it (one UMMA per
// start into the spare TMEM columns, with init_d staged as the bf16 operand
// in the incoming-state tile, which Yoff has finished reading); the
// epilogue then adds them unscaled.  q_i comes from a segmented scan of the
// log2-decays that restarts at each start (no prefix subtraction).  Also
// leaves in sh.qlast / sh.dlast the decay and document of the initial state
// that reaches the chunk's end (dlast = -1: none).  Inlined like doc_end_mma
// (16-column pieces and 32 loads at a time beside the caller's live state):
// all 128 threads of the state group call it together (thread i =
// chunk row i = TMEM lane i).
__device__ __forceinline__ void doc_start_rows(TcSmall& sh, const FwdArgs& a, const ChunkMeta& m, uint32_t ctile,
                                            uint8_t* sin_tile, uint32_t tb, int X, float A2, int h, int nv, int i,
                                            int& init_cnt) {
    constexpr uint32_t idYo = ptx::idesc_bf16(128, 64, 0, 1);
    const int lane = i & 31, rb = i >> 5;
    const uint32_t lane_off = (uint32_t)(32 * rb) << 16;
    const uint32_t yo = tb + lane_off + kTmYo + 64 * X, scr = tb + lane_off + kTmInit;
    // (the caller has waited for this chunk's Yoff, which has read the incoming-state tile)
    // segmented inclusive scan of l within the warp, restarting at starts
    const bool st_i = i < nv && (m.rowflag[i] & 1);
    float v = (i < nv) ? (st_i ? m.dtv[i] * A2 : m.ell[i]) : 0.f;
    bool f = st_i;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float vu = __shfl_up_sync(0xffffffffu, v, o);
        const int fu = __shfl_up_sync(0xffffffffu, (int)f, o);
        if (lane >= o && !f) {
            v = vu + v;
            f = fu != 0;
        }
    }
    const uint32_t smask = __ballot_sync(0xffffffffu, st_i);
    if (lane == 31) sh.segtot[rb] = v;
    if (lane == 0) sh.startmask[rb] = smask;
    ptx::named_bar(kBarState, 128);
    // rows whose segment began in an earlier warp carry the later warps' sums
    bool has = f;
    if (!f) {
        for (int r = rb - 1; r >= 0; --r) {
            v = sh.segtot[r] + v;
            if (sh.startmask[r]) {
                has = true;
                break;
            }
        }
    }
    const float q = has ? ex2_approx(v) : 0.f;
    // rows before the first start: 2^{p_i} Yoff_i (rows after it are rewritten below)
    {
        const float pe = m.pexp[i];
#pragma unroll 1
        for (int q16 = 0; q16 < 4; ++q16) {   // 16 columns at a time (the caller's state is live)
            uint32_t r[16];
            ptx::tmem_load16(yo + 16 * q16, r);
#pragma unroll
            for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * pe);
            ptx::tmem_st16(yo + 16 * q16, r);
        }
        ptx::tmem_st_wait();
    }
    // one UMMA C init_d^T per document start, its rows merged into Yoff
#pragma unroll 1
    for (int w = 0; w < 4; ++w) {
        uint32_t mk = sh.startmask[w];
        while (mk) {
            const int st = 32 * w + __ffs(mk) - 1;
            mk &= mk - 1;
            const int d = m.rowdoc[st];
            // init_d as the (n, p) bf16 operand; thread i writes state column n = i
            // (32 loads in flight at a time: the caller's state is live)
            const float* src = a.init + ((size_t)d * a.H + h) * (size_t)(P * N) + i;
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
                float iv[32];
#pragma unroll
                for (int p = 0; p < 32; ++p) iv[p] = __ldg(src + (size_t)(32 * hp + p) * N);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4*>(sin_tile + sw128_off(i, 32 * hp + 8 * q8)) =
                        make_uint4(pack_bf16(iv[8 * q8], iv[8 * q8 + 1]), pack_bf16(iv[8 * q8 + 2], iv[8 * q8 + 3]),
                                   pack_bf16(iv[8 * q8 + 4], iv[8 * q8 + 5]),
                                   pack_bf16(iv[8 * q8 + 6], iv[8 * q8 + 7]));
            }
            ptx::fence_proxy_async();
            ptx::named_bar(kBarState, 128);
            if (i == 0) {
                ptx::tc_fence_after();
                const uint32_t sin = ptx::smem_u32(sin_tile);
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb + kTmInit, desc_k(ctile, kk), desc_mn1(sin, kk), idYo, kk > 0);
                ptx::mma_commit(&sh.barInit);
            }
            wait_or_fail(sh, a, &sh.barInit, (uint32_t)(init_cnt & 1), kWhereBarInit);
            ++init_cnt;
            ptx::tc_fence_after();
            const bool mine = has && i < nv && m.rowdoc[i] == d;
            if (__any_sync(0xffffffffu, mine)) {
#pragma unroll 1
                for (int q16 = 0; q16 < 4; ++q16) {   // 16 columns at a time
                    uint32_t sr[16], yr[16];
                    ptx::tmem_load16x2(scr + 16 * q16, sr, yo + 16 * q16, yr);
#pragma unroll
                    for (int k = 0; k < 16; ++k) yr[k] = mine ? __float_as_uint(q * __uint_as_float(sr[k])) : yr[k];
                    ptx::tmem_st16(yo + 16 * q16, yr);
                }
                ptx::tmem_st_wait();
            }
            // the spare columns and the operand tile are free for the next start
            ptx::tc_fence_before();
            ptx::named_bar(kBarState, 128);
        }
    }
    if (i == nv - 1) {
        sh.dlast = has ? m.rowdoc[i] : -1;
        sh.qlast = q;
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&sh.barFix[X]);
    ptx::named_bar(kBarState, 128);   // dlast / qlast visible to the group
}

// A unit: batch row b, split s, head h (heads of one (row, split) are adjacent
// in unit order, so CTAs that run at the same time share B and C in L2).
struct Unit {
    int b, h, g, s;
    int t0, t1, nch;   // token range of the split (tokens < 2^31, as TMA coordinates are), its chunks
    int ws;            // workspace slot of a split (a whole unit has none)
};

__device__ __forceinline__ uint32_t fdiv(uint32_t n, uint32_t m, uint32_t l) { return (__umulhi(m, n) + n) >> l; }

template <bool kFull>
__device__ __forceinline__ Unit unit_at(const FwdArgs& a, int64_t u64) {
    const uint32_t u = (uint32_t)u64;
    Unit r;
    if (a.tail_units > 0) {
        // leftover-unit plan: whole (row, head) units first (full pass only), then the
        // pieces: leftover unit t, split s at index tail_first + t * nsplit + s
        if (kFull && u < (uint32_t)a.tail_first) {
            const uint32_t bb = fdiv(u, a.divH_m, a.divH_l);
            r.h = (int)(u - bb * (uint32_t)a.H);
            r.b = (int)bb;
            r.s = 0;
            r.ws = -1;
            r.t0 = 0;
            r.t1 = (int)a.L;
        } else {
            const uint32_t v = kFull ? u - (uint32_t)a.tail_first : u;
            const uint32_t t = fdiv(v, a.divS_m, a.divS_l);
            const uint32_t unit = (uint32_t)a.tail_first + t;
            const uint32_t bb = fdiv(unit, a.divH_m, a.divH_l);
            r.h = (int)(unit - bb * (uint32_t)a.H);
            r.b = (int)bb;
            r.s = (int)(v - t * (uint32_t)a.nsplit);
            r.ws = (int)v;
            r.t0 = r.s * (int)a.split_len;
            r.t1 = (r.t0 + a.split_len < a.L) ? r.t0 + (int)a.split_len : (int)a.L;
        }
    } else {
        // unit u = (b * nsplit + s) * H + h, below 2^31 (checked by the caller of the kernel)
        const uint32_t bs = fdiv(u, a.divH_m, a.divH_l);
        const uint32_t bb = fdiv(bs, a.divS_m, a.divS_l);
        r.h = (int)(u - bs * (uint32_t)a.H);
        r.s = (int)(bs - bb * (uint32_t)a.nsplit);
        r.b = (int)bb;
        r.ws = (int)(((uint32_t)r.b * (uint32_t)a.H + (uint32_t)r.h) * (uint32_t)a.nsplit + (uint32_t)r.s);
        r.t0 = r.s * (int)a.split_len;
        r.t1 = (r.t0 + a.split_len < a.L) ? r.t0 + (int)a.split_len : (int)a.L;
    }
    r.g = (int)fdiv((uint32_t)r.h, a.divHG_m, a.divHG_l);
    r.nch = (r.t1 - r.t0 + Q - 1) / Q;
    return r;
}

// Walks this CTA's items (unit, chunk) in order.  CTA k runs the units k,
// k + gridDim.x, ...: with more units than SMs the grid is persistent (one CTA
// per SM) and the pipeline runs on across unit boundaries, instead of paying a
// CTA start and a pipeline ramp per unit.
// (U = the number of units: a.batch * a.H * a.nsplit < 2^31.)  kPersist = false:
// one unit per CTA, and the cursor never moves to another unit.
template <bool kFull, bool kPersist>
struct Cursor {
    int u, c;
    Unit un;
    __device__ void init(const FwdArgs& a) {
        u = (int)blockIdx.x;
        c = 0;
        un = unit_at<kFull>(a, u);
    }
    __device__ __forceinline__ bool valid(int U) const { return u < U; }
    __device__ __forceinline__ int t() const { return un.t0 + c * Q; }
    __device__ void next(const FwdArgs& a, int U) {
        if (++c >= un.nch) {
            c = 0;
            if (kPersist) {
                u += (int)gridDim.x;
                if (u < U) un = unit_at<kFull>(a, u);
            } else {
                u = U;
            }
        }
    }
    // two items on (a unit may be a single chunk)
    __device__ void next2(const FwdArgs& a, int U) {
        c += 2;
        if (!kPersist) {
            if (c >= un.nch) u = U;
            return;
        }
        while (c >= un.nch && u < U) {
            c -= un.nch;
            u += (int)gridDim.x;
            if (u < U) un = unit_at<kFull>(a, u);
        }
    }
};

// kFull: full pass (else the aggregate pass of a split plan); kDocs: packed
// documents (cu_seqlens).  Each combination is its own kernel, so the hot
// loops carry no run-time mode branches: the compiler would otherwise keep a
// copy of a loop body per branch, and instruction fetch is a scarce resource
// for this kernel (its warps run several different loops at once).
// kPersist: a persistent grid (one CTA per SM, each running several units),
// used for short units, whose per-CTA start and pipeline ramp would dominate.
// kEvents (with kFull and kDocs): the documents' initial or final states are
// asked for, and the document events inside chunks are handled (their code
// would otherwise cost registers in the plain packed-document kernel).
template <bool kFull, bool kDocs, bool kPersist, bool kEvents = false>
__global__ void __launch_bounds__(kThreads, 1) ssd_chunk_tc(const __grid_constant__ TcParams prm) {
    using Cursor = ssd::Cursor<kFull, kPersist>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    TcSmall& sh = *reinterpret_cast<TcSmall*>(sm + kTiles);
    const FwdArgs& a = prm.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = warp >> 2;
    constexpr bool full_mode = kFull;
    pdl_trigger();

    // items of this CTA: the chunks of units blockIdx.x, blockIdx.x + gridDim.x, ...
    const int nunits = (int)(a.batch * a.H * a.nsplit);
    int nch = 0;
    if (kPersist) {
        for (int u = (int)blockIdx.x; u < nunits; u += (int)gridDim.x) nch += unit_at<kFull>(a, u).nch;
    } else {
        nch = unit_at<kFull>(a, (int)blockIdx.x).nch;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sh.full[i], 1);
            // stage readers: dS issuer, mask group, state group (+ Ydiag and Yoff issuers)
            ptx::mbar_init(&sh.empty[i], full_mode ? 5 : 3);
            ptx::mbar_init(&sh.barG[i], 1);
            ptx::mbar_init(&sh.barM[i], 4);
            ptx::mbar_init(&sh.barXt[i], 4);
            ptx::mbar_init(&sh.barYd[i], 1);
            ptx::mbar_init(&sh.barDS[i], 1);
            ptx::mbar_init(&sh.barY[i], 1);
            ptx::mbar_init(&sh.yFree[i], 4);
        }
        ptx::mbar_init(&sh.dsFree, 4);
        for (int i = 0; i < NMETA; ++i) {
            ptx::mbar_init(&sh.metaFull[i], 4);
            ptx::mbar_init(&sh.metaFree[i], 1);
        }
        for (int i = 0; i < 4; ++i) ptx::mbar_init(&sh.drain[i], 1);
        ptx::mbar_init(&sh.barInit, 1);
        ptx::mbar_init(&sh.barFix[0], 4);
        ptx::mbar_init(&sh.barFix[1], 4);
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

    if (wg == 0) {
        ptx::regs_dec<kRegsIssue>();
        if (warp == 0 && lane == 0) {
            // ============================================================ TMA producer
            int issued = 0;
            // L2 prefetch of the item two ahead of the one being loaded (the tiles of this
            // stage's next refill), so a refill finds them in L2 instead of waiting on
            // HBM.  Longer distances (4, 6 and 10 items) measured slower: the prefetched
            // tiles of all CTAs then compete in L2 with tiles still in use.
            auto prefetch = [&](const Cursor& k) {
                if (!k.valid(nunits)) return;
                const int t = k.t(), hh = k.un.h, gg = k.un.g, bb = k.un.b;
                ptx::tma_prefetch_4d(&prm.tm_x, 0, hh, t, bb);
                ptx::tma_prefetch_4d(&prm.tm_B, 0, gg, t, bb);
                ptx::tma_prefetch_4d(&prm.tm_B, 64, gg, t, bb);
                if (full_mode) {
                    ptx::tma_prefetch_4d(&prm.tm_C, 0, gg, t, bb);
                    ptx::tma_prefetch_4d(&prm.tm_C, 64, gg, t, bb);
                }
            };
            Cursor cl, cp;                         // the item loaded, the item prefetched
            cl.init(a);
            cp.init(a);
            cp.next2(a, nunits);
            // (fault injection: no load is issued, so the waits on them run out)
            for (int c = 0; c < (a.stall_loads ? 0 : nch); ++c, cl.next(a, nunits)) {
                const int st = c & 1;
                prefetch(cp);
                cp.next(a, nunits);
                if (c >= 2 && !wait_or_fail(sh, a, &sh.empty[st], ((c >> 1) - 1) & 1, kWhereEmpty)) break;
                const int t = cl.t(), h = cl.un.h, g = cl.un.g, b = cl.un.b;
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
            for (int st = 0; st < 2 && st < issued; ++st) {
                const int last = ((issued - 1 - st) >> 1) * 2 + st;
                if (!ptx::mbar_wait(&sh.full[st], (last >> 1) & 1, &sh.never, a.wait_iters)) fail(sh, a, kWhereDrain);
            }
        } else if (warp == 1 && lane == 0) {
            // ============================================================ dS issuer
            // the chunk state summary needs only the scaled X tile, so it runs as soon
            // as that is written (ahead of the mask), which keeps the state recurrence short
            constexpr uint32_t idDS = ptx::idesc_bf16(128, 64, 1, 1);
            for (int c = 0; c < nch; ++c) {
                const int X = c & 1, j = c >> 1;
                const uint32_t stg = ptx::smem_u32(sm + X * kStageBytes);
                if (!wait_or_fail(sh, a, &sh.barXt[X], j & 1, kWhereBarXt)) break;
                if (c >= 1 && !wait_or_fail(sh, a, &sh.dsFree, (c - 1) & 1, kWhereDsFree)) break;
                ptx::tc_fence_after();
                const uint32_t xt = ptx::smem_u32(sm + kXt + 16384 * X);
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb + kTmDS, desc_mn2(stg + kTileB, kk), desc_mn1(xt, kk), idDS, kk > 0);
                ptx::mma_commit(&sh.barDS[X]);
                ptx::mma_commit(&sh.empty[X]);
            }
            ptx::mma_commit(&sh.drain[0]);
            if (!ptx::mbar_wait(&sh.drain[0], 0, &sh.never, a.wait_iters)) fail(sh, a, kWhereDrain);
        } else if (warp == 3 && lane == 0 && full_mode) {
            // ============================================================ Ydiag issuer
            constexpr uint32_t idYd = ptx::idesc_bf16(128, 64, 0, 1);
            for (int c = 0; c < nch; ++c) {
                const int X = c & 1, j = c >> 1;
                const uint32_t stg = ptx::smem_u32(sm + X * kStageBytes);
                if (!wait_or_fail(sh, a, &sh.barM[X], j & 1, kWhereBarM)) break;
                ptx::tc_fence_after();
                const uint32_t gm = tb + kTmGM + 128 * X;
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ts(gm + 64, gm + 8 * kk, desc_mn1(stg + kTileX, kk), idYd, kk > 0);
                ptx::mma_commit(&sh.barYd[X]);
                ptx::mma_commit(&sh.empty[X]);
            }
            ptx::mma_commit(&sh.drain[3]);
            if (!ptx::mbar_wait(&sh.drain[3], 0, &sh.never, a.wait_iters)) fail(sh, a, kWhereDrain);
        } else if (warp == 2 && lane == 0 && full_mode) {
            // ============================================================ G issuer
            constexpr uint32_t idG = ptx::idesc_bf16(128, 128, 0, 0);
            for (int c = 0; c < nch; ++c) {
                const int X = c & 1, j = c >> 1;
                const uint32_t stg = ptx::smem_u32(sm + X * kStageBytes);
                if (!wait_or_fail(sh, a, &sh.full[X], j & 1, kWhereFull)) break;
                // G/M buffer X is free once the epilogue of chunk c-2 has read its Ydiag
                if (j >= 1 && !wait_or_fail(sh, a, &sh.yFree[X], (j - 1) & 1, kWhereYFree)) break;
                ptx::tc_fence_after();
                const uint32_t d = tb + kTmGM + 128 * X;
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(d, desc_k(stg + kTileC, kk), desc_k(stg + kTileB, kk), idG, kk > 0);
                ptx::mma_commit(&sh.barG[X]);
            }
            ptx::mma_commit(&sh.drain[1]);
            if (!ptx::mbar_wait(&sh.drain[1], 0, &sh.never, a.wait_iters)) fail(sh, a, kWhereDrain);
        } else if (warp == 1 && kDocs && full_mode && blockIdx.x == 0) {
            // the dS issuer's idle lanes: the packed-document offsets of the call
            check_cu_seqlens(a.cu, a.ndocs, a.L, a.ws, lane - 1, 31);
        }
    } else if (wg <= 2) {
        // ================================================================ mask groups
        ptx::regs_inc<kRegsMath>();
        const int X = wg - 1;                     // this group takes chunks c with c & 1 == X
        const int nb = kBarMask0 + X;
        MaskScratch& ms = sh.mask[X];
        const int mt = threadIdx.x - 128 * wg;    // 0..127
        const int rb = warp & 3;                  // TMEM lane quarter = row block
        const int i = 32 * rb + lane;             // chunk row = TMEM lane
        const uint32_t lane_addr = tb + ((uint32_t)(32 * rb) << 16);
        auto load_dt = [&](const Cursor& k) -> float {
            if (!k.valid(nunits)) return 0.f;
            const int t = k.t();
            return (t + i < k.un.t1) ? __ldg(a.dt + ((size_t)k.un.b * a.L + t + i) * a.H + k.un.h) : 0.f;
        };
        Cursor cur;                               // this group's item
        cur.init(a);
        if (X) cur.next(a, nunits);
        float dt_next = load_dt(cur);
        int unit_prev = -1;
        int nfix = 0;                             // chunks of this group whose Yoff rows the state group rewrote
        float A2 = 0.f, Dh = 0.f;
        for (int c = X; c < nch; c += 2) {
            const int j = c >> 1, mb = c % NMETA;
            uint8_t* stg = sm + X * kStageBytes;
            const int t = cur.t(), t1 = cur.un.t1, b = cur.un.b, h = cur.un.h;
            const int nv = (int)((t + Q < t1) ? Q : t1 - t);
            const bool new_unit = cur.u != unit_prev;
            if (new_unit) {
                unit_prev = cur.u;
                A2 = a.A[h] * kLog2e;
                Dh = a.D ? a.D[h] : 0.f;
            }
            const float dti = dt_next;
            {
                Cursor cn = cur;                  // this group's next item: its dt is loaded now,
                cn.next2(a, nunits);              // a whole iteration before it is used
                dt_next = load_dt(cn);
            }
            if (c >= NMETA) wait_or_fail(sh, a, &sh.metaFree[mb], ((c / NMETA) - 1) & 1, kWhereMetaFree);
            // document boundaries: walk forward from this group's cursor
            int flag = 0, doc = (int)b;
            if (i < nv) {
                if (kDocs) {
                    // (the cursor restarts with every unit this group enters)
                    int d = new_unit ? find_doc_tc(a.cu, a.ndocs, t) : ms.doc_cursor;
                    while (d + 1 < a.ndocs && __ldg(a.cu + d + 1) <= t + i) ++d;
                    doc = d;
                    if (d > 0 && __ldg(a.cu + d) == t + i) flag |= 1;
                    if (t + i + 1 == __ldg(a.cu + d + 1)) flag |= 2;
                    // the document's initial state, which the state group reads for this
                    // chunk, on its way to L2 a chunk ahead
                    if (kEvents && (flag & 1) && a.init)
                        ptx::bulk_prefetch_l2(a.init + ((size_t)d * a.H + h) * (P * N), P * N * 4);
                } else if (t + i == a.L - 1) {
                    flag |= 2;
                }
            }
            const float l2 = (flag & 1) ? -INFINITY : dti * A2;
            ChunkMeta& m = sh.meta[mb];
            ms.seg.a[i] = ex2_approx(l2);         // 0 at a document start
            ms.dtv[i] = dti;
            m.ell[i] = l2;
            m.dtv[i] = dti;
            m.rowflag[i] = flag;
            m.rowdoc[i] = doc;
            if (!full_mode) {
                float ls = l2;                     // block sum of the log-decays (the split's tau)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
                if (lane == 0) ms.totLog[rb] = ls;
            }
            // packed documents with initial states: when one starts in this chunk, the
            // state group rewrites the chunk's Yoff rows, which the epilogue adds unscaled
            bool fix = false;
            if (kEvents)
                fix = ptx::named_bar_any(nb, 128, (flag & 1) != 0) && a.init != nullptr;
            else
                ptx::named_bar(nb, 128);
            if (kDocs && mt == Q - 1) ms.doc_cursor = doc;   // later chunks start in (or after) this document
            SegsumLinRow<4> row;
            segsum_lin_phase1<4>(ms.seg, row, rb, lane);   // the diagonal 1-SS block
            ptx::named_bar(nb, 128);
            segsum_lin_phase2<4>(ms.seg, row, rb, lane);   // rank-one row factors, chunk prefix
            // the y store of chunk c-2 (staged in this group's scaled-X buffer) has read it
            if (mt == 0 && j >= 1) ptx::bulk_wait_read0();
            ptx::named_bar(nb, 128);
            ms.colfac[i] = ms.seg.colL[i] * dti;
            const float xf = segsum_lin_suffix<4>(ms.seg, i) * dti;   // 2^{s_i} dt_i
            const float pe = row.pe;
            m.pexp[i] = pe;
            if (mt == 0) {
                m.tauexp = ms.seg.tauL;
                if (!full_mode) m.tau = (ms.totLog[0] + ms.totLog[1]) + (ms.totLog[2] + ms.totLog[3]);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sh.metaFull[mb]);
            // scaled X (state-summary operand): buffer X is free once dS(c-2) is done
            wait_or_fail(sh, a, &sh.full[X], j & 1, kWhereFull);
            if (j >= 1) wait_or_fail(sh, a, &sh.barDS[X], (j - 1) & 1, kWhereBarDS);
            {
                const uint8_t* xrow = stg + kTileX;
                uint8_t* xt = sm + kXt + 16384 * X;
                const uint64_t xf2 = ptx::f2_pack(xf, xf);
#pragma unroll 2
                for (int q = 0; q < 8; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4*>(xrow + sw128_off(i, 8 * q));
                    uint4 o;
                    o.x = pack_bf16_2(ptx::f2_mul(ptx::f2_pack(bf16lo(v.x), bf16hi(v.x)), xf2));
                    o.y = pack_bf16_2(ptx::f2_mul(ptx::f2_pack(bf16lo(v.y), bf16hi(v.y)), xf2));
                    o.z = pack_bf16_2(ptx::f2_mul(ptx::f2_pack(bf16lo(v.z), bf16hi(v.z)), xf2));
                    o.w = pack_bf16_2(ptx::f2_mul(ptx::f2_pack(bf16lo(v.w), bf16hi(v.w)), xf2));
                    *reinterpret_cast<uint4*>(xt + sw128_off(i, 8 * q)) = o;
                }
                ptx::fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sh.barXt[X]);   // the state summary can start
            ptx::named_bar(nb, 128);              // colfac complete; X tile reads done
            if (mt == 0) ptx::mbar_arrive(&sh.empty[X]);
            if (full_mode) {
                // M is written over G (block r of M occupies G columns already consumed)
                wait_or_fail(sh, a, &sh.barG[X], j & 1, kWhereBarG);
                ptx::tc_fence_after();
                const uint32_t gm = lane_addr + kTmGM + 128 * X;
                // rank-one off-diagonal blocks r < rb: row factor x column factor
#pragma unroll 1
                for (int r = 0; r < rb; ++r) {
                    uint32_t gr[32];
                    ptx::tmem_load32(gm + 32 * r, gr);
                    const float rf = (r == 0) ? row.rf[0] : (r == 1) ? row.rf[1] : row.rf[2];
                    const uint64_t rf2 = ptx::f2_pack(rf, rf);
                    const float4* cf = reinterpret_cast<const float4*>(ms.colfac + 32 * r);
                    uint32_t pk[16];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 f = cf[q];
                        const uint64_t g01 = ptx::f2_pack(__uint_as_float(gr[4 * q]), __uint_as_float(gr[4 * q + 1]));
                        const uint64_t g23 =
                            ptx::f2_pack(__uint_as_float(gr[4 * q + 2]), __uint_as_float(gr[4 * q + 3]));
                        pk[2 * q] = pack_bf16_2(ptx::f2_mul(ptx::f2_mul(g01, rf2), ptx::f2_pack(f.x, f.y)));
                        pk[2 * q + 1] = pack_bf16_2(ptx::f2_mul(ptx::f2_mul(g23, rf2), ptx::f2_pack(f.z, f.w)));
                    }
                    ptx::tmem_st16(gm + 16 * r, pk);
                }
                // 1-SS diagonal block rb (products grown from the diagonal, 0 above it), plus D
                // on the diagonal
                {
                    uint32_t gr[32];
                    ptx::tmem_load32(gm + 32 * rb, gr);
                    const float4* dv = reinterpret_cast<const float4*>(ms.dtv + 32 * rb);
                    uint32_t pk[16];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 f = dv[q];
                        const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                        for (int e = 0; e < 4; e += 2) {
                            const int col = 4 * q + e;
                            const uint64_t gw = ptx::f2_mul(
                                ptx::f2_pack(__uint_as_float(gr[col]), __uint_as_float(gr[col + 1])),
                                ptx::f2_pack(row.wl[col], row.wl[col + 1]));
                            const uint64_t dd = ptx::f2_pack((col == lane) ? Dh : 0.f, (col + 1 == lane) ? Dh : 0.f);
                            pk[2 * q + e / 2] = pack_bf16_2(ptx::f2_fma(gw, ptx::f2_pack(fv[e], fv[e + 1]), dd));
                        }
                    }
                    ptx::tmem_st16(gm + 16 * rb, pk);
                }
                // above the diagonal blocks: zero (those columns held G)
                {
                    uint32_t z[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) z[q] = 0u;
#pragma unroll 1
                    for (int r = rb + 1; r < 4; ++r) ptx::tmem_st16(gm + 16 * r, z);
                }
                ptx::tmem_st_wait();
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sh.barM[X]);
            bool stop;
            if (full_mode) {
                // ---- epilogue of chunk c: y = Ydiag + 2^{p_i} Yoff  (D x is in Ydiag).
                // The rows are staged in this group's scaled-X buffer (free once dS(c)
                // is done) and written by one TMA store (rows past L are clipped).
                wait_or_fail(sh, a, &sh.barYd[X], j & 1, kWhereBarYd);
                wait_or_fail(sh, a, &sh.barY[X], j & 1, kWhereBarY);
                if (fix) {
                    wait_or_fail(sh, a, &sh.barFix[X], nfix & 1, kWhereBarFix);
                    ++nfix;
                }
                wait_or_fail(sh, a, &sh.barDS[X], j & 1, kWhereBarDS);
                ptx::tc_fence_after();
                const uint32_t yd_addr = lane_addr + kTmGM + 128 * X + 64;
                const uint32_t yo_addr = lane_addr + kTmYo + 64 * X;
                uint8_t* ys = sm + kXt + 16384 * X;
#pragma unroll 1
                for (int q8 = 0; q8 < 2; ++q8) {
                    uint32_t yd[32], yo[32];
                    ptx::tmem_load32x2(yd_addr + 32 * q8, yd, yo_addr + 32 * q8, yo);
                    if (q8 == 1) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(&sh.yFree[X]);
                    }
                    uint32_t ow[16];
                    const float ps = fix ? 1.f : pe;
                    const uint64_t pe2 = ptx::f2_pack(ps, ps);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        ow[e] = pack_bf16_2(ptx::f2_fma(
                            pe2, ptx::f2_pack(__uint_as_float(yo[2 * e]), __uint_as_float(yo[2 * e + 1])),
                            ptx::f2_pack(__uint_as_float(yd[2 * e]), __uint_as_float(yd[2 * e + 1]))));
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(ys + sw128_off(i, 32 * q8 + 8 * q)) =
                            make_uint4(ow[4 * q], ow[4 * q + 1], ow[4 * q + 2], ow[4 * q + 3]);
                }
                ptx::fence_proxy_async();
                // every row is staged (and the group's last look at the abort flag
                // this chunk: nothing after this barrier reads the group's scratch)
                stop = ptx::named_bar_any(nb, 128, *(volatile int*)&sh.abort != 0);
                if (mt == 0 && !stop) {
                    ptx::tma_store_4d(&prm.tm_y, ys, 0, h, (int)t, (int)b);
                    ptx::bulk_commit();
                }
            } else {
                stop = ptx::named_bar_any(nb, 128, *(volatile int*)&sh.abort != 0);
            }
            cur.next2(a, nunits);                 // this group's next item
            if (stop) break;
        }
        if (mt == 0) ptx::bulk_wait0();
    } else {
        // ================================================================ state group
        ptx::regs_inc<kRegsMath>();
        const int mt = threadIdx.x - 384;         // 0..127
        const int rb = warp & 3;
        const int i = 32 * rb + lane;             // TMEM lane = state column n
        const uint32_t lane_addr = tb + ((uint32_t)(32 * rb) << 16);
        const size_t PN = (size_t)P * N;
        float S[P];
        // the state entering a unit: the composed state of the earlier splits, the
        // caller's initial state, or zero
        auto enter_state = [&](const Unit& un) {
            const float* src = nullptr;
            if (full_mode && a.nsplit > 1 && un.s > 0) {
                pdl_wait();                       // the split scan (and everything before it) is complete
                src = a.ws_state + (size_t)(un.ws - 1) * PN;   // (slot s - 1)
            }
            else if (un.s == 0 && a.init) src = a.init + ((size_t)un.b * a.H + un.h) * PN;   // (documents: d = 0 = b)
#pragma unroll
            for (int p = 0; p < P; ++p) S[p] = src ? src[(size_t)p * N + i] : 0.f;
        };
        Cursor cs;
        cs.init(a);
        enter_state(cs.un);
        // incoming state as the bf16 operand of Yoff; then one thread issues Yoff(k)
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
        };
        auto issue_yoff = [&](int k) -> bool {
            constexpr uint32_t idYo = ptx::idesc_bf16(128, 64, 0, 1);
            const int Y = k & 1, jj = k >> 1;
            if (!wait_or_fail(sh, a, &sh.full[Y], jj & 1, kWhereFull)) return false;
            // Yoff buffer Y is free once the epilogue of chunk k-2 has read it
            if (jj >= 1 && !wait_or_fail(sh, a, &sh.yFree[Y], (jj - 1) & 1, kWhereYFree)) return false;
            ptx::tc_fence_after();
            const uint32_t stg = ptx::smem_u32(sm + Y * kStageBytes);
            const uint32_t sin = ptx::smem_u32(sm + kSin);
#pragma unroll 1
            for (int kk = 0; kk < 8; ++kk)
                ptx::mma_ss(tb + kTmYo + 64 * Y, desc_k(stg + kTileC, kk), desc_mn1(sin, kk), idYo, kk > 0);
            ptx::mma_commit(&sh.barY[Y]);
            ptx::mma_commit(&sh.empty[Y]);
            return true;
        };
        if (full_mode && nch > 0) {
            write_sin();
            ptx::named_bar(kBarState, 128);
            if (mt == 0) issue_yoff(0);
        }
        float tau_split = 0.f;
        int init_cnt = 0;                         // UMMAs C init_d^T issued (packed documents with initial states)
        for (int c = 0; c < nch; ++c) {
            const int X = c & 1, j = c >> 1, mb = c % NMETA;
            uint8_t* stg = sm + X * kStageBytes;
            const int t = cs.t(), t1 = cs.un.t1, h = cs.un.h;
            const size_t uw = (size_t)cs.un.ws;
            const int nv = (int)((t + Q < t1) ? Q : t1 - t);
            const bool unit_end = cs.c == cs.un.nch - 1;
            const bool meta_ok = wait_or_fail(sh, a, &sh.metaFull[mb], (c / NMETA) & 1, kWhereMetaFull);
            const ChunkMeta& m = sh.meta[mb];
            // ---- packed documents: final states of those that end inside this chunk,
            // and the state terms of the rows of those that start in it
            bool fix = false;
            if (kEvents) {
                const int fl = m.rowflag[i];       // 0 past the chunk's last row
                const float A2 = a.A[h] * kLog2e;
                const bool end_row = i < nv - 1 && (fl & 2);
                // agreed by the whole group, and only on chunk values that are
                // complete: the branches hold barriers, and after a wait that ran
                // out the values may still be changing
                const uint32_t wf = __reduce_or_sync(
                    0xffffffffu, (meta_ok ? 0u : 1u) | (end_row ? 2u : 0u) | ((fl & 1) ? 4u : 0u));
                if (lane == 0) sh.evflags[rb] = wf;
                ptx::named_bar(kBarState, 128);
                const uint32_t gf = (sh.evflags[0] | sh.evflags[1]) | (sh.evflags[2] | sh.evflags[3]);
                const bool stale = (gf & 1u) != 0;
                const bool any_end = (gf & 2u) && !stale && a.fin != nullptr;
                fix = (gf & 4u) && !stale && a.init != nullptr;
                if (any_end || fix) {
                    // Yoff(c) is complete: the incoming-state tile and the spare TMEM
                    // columns are free for the rare paths below
                    wait_or_fail(sh, a, &sh.barY[X], j & 1, kWhereBarY);
                    ptx::tc_fence_after();
                }
                if (any_end) {
                    wait_or_fail(sh, a, &sh.full[X], j & 1, kWhereFull);   // the chunk's x and B
                    const uint32_t emask = __ballot_sync(0xffffffffu, end_row);
                    if (lane == 0) sh.endmask[rb] = emask;
                    ptx::named_bar(kBarState, 128);
#pragma unroll 1
                    for (int w = 0; w < 4; ++w) {
                        uint32_t mk = sh.endmask[w];
                        while (mk) {
                            const int e = 32 * w + __ffs(mk) - 1;
                            mk &= mk - 1;
                            doc_end_mma(sh, a, m, stg, sm + kSin, tb, e, A2, i, init_cnt);
                            const float pe = m.pexp[e], qe = sh.qend;
                            const size_t so = ((size_t)m.rowdoc[e] * a.H + h) * PN + i;
                            float* fo = a.fin + so;
                            const float* src = a.init + so;
                            // in two halves of 32 columns (32 registers beside the state's 64)
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                uint32_t dv[32];
                                ptx::tmem_load32(lane_addr + kTmInit + 32 * half, dv);
                                if (qe != 0.f) {
#pragma unroll
                                    for (int p = 0; p < 32; ++p)
                                        fo[(size_t)(p + 32 * half) * N] =
                                            fmaf(qe, __ldg(src + (size_t)(p + 32 * half) * N),
                                                 fmaf(pe, S[p + 32 * half], __uint_as_float(dv[p])));
                                } else {
#pragma unroll
                                    for (int p = 0; p < 32; ++p)
                                        fo[(size_t)(p + 32 * half) * N] =
                                            fmaf(pe, S[p + 32 * half], __uint_as_float(dv[p]));
                                }
                            }
                            // the spare TMEM columns and the operand tile are free again
                            ptx::tc_fence_before();
                            ptx::named_bar(kBarState, 128);
                        }
                    }
                }
                if (fix)
                    doc_start_rows(sh, a, m, ptx::smem_u32(stg + kTileC), sm + kSin, tb, X, A2, h, nv, i, init_cnt);
            }
            // ---- state update: S = 2^tau S + dS (TMEM lane = state column n)
            wait_or_fail(sh, a, &sh.barDS[X], j & 1, kWhereBarDS);
            ptx::tc_fence_after();
            {
                uint32_t ds0[32], ds1[32];
                ptx::tmem_load32x2(lane_addr + kTmDS, ds0, lane_addr + kTmDS + 32, ds1);
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sh.dsFree);
                const float ed = m.tauexp;
                if (!full_mode) tau_split += m.tau;
                const uint64_t ed2 = ptx::f2_pack(ed, ed);
#pragma unroll
                for (int q = 0; q < 32; q += 2) {
                    const uint64_t r0 = ptx::f2_fma(ed2, ptx::f2_pack(S[q], S[q + 1]),
                                                    ptx::f2_pack(__uint_as_float(ds0[q]), __uint_as_float(ds0[q + 1])));
                    ptx::f2_unpack(r0, S[q], S[q + 1]);
                    const uint64_t r1 = ptx::f2_fma(
                        ed2, ptx::f2_pack(S[32 + q], S[33 + q]),
                        ptx::f2_pack(__uint_as_float(ds1[q]), __uint_as_float(ds1[q + 1])));
                    ptx::f2_unpack(r1, S[32 + q], S[33 + q]);
                }
            }
            if (kEvents && fix && sh.dlast >= 0) {
                // the initial state of the document open at the chunk's end, which started in it
                const float ql = sh.qlast;
                const float* src = a.init + ((size_t)sh.dlast * a.H + h) * PN + i;
#pragma unroll
                for (int p = 0; p < P; ++p) S[p] = fmaf(ql, __ldg(src + (size_t)p * N), S[p]);
            }
            if (full_mode && a.fin && (m.rowflag[nv - 1] & 2)) {
                float* fo = a.fin + ((size_t)m.rowdoc[nv - 1] * a.H + h) * PN + i;
#pragma unroll
                for (int p = 0; p < P; ++p) fo[(size_t)p * N] = S[p];
            }
            ptx::named_bar(kBarState, 128);       // meta and stage reads of chunk c are done
            if (mt == 0) {
                ptx::mbar_arrive(&sh.metaFree[mb]);
                ptx::mbar_arrive(&sh.empty[X]);
            }
            if (!full_mode && unit_end && !*(volatile int*)&sh.abort) {
                // aggregate pass: the split's state summary and total decay
#pragma unroll
                for (int p = 0; p < P; ++p) a.ws_state[uw * PN + (size_t)p * N + i] = S[p];
                if (mt == 0) a.ws_tau[uw] = tau_split * kLn2;
                tau_split = 0.f;
            }
            cs.next(a, nunits);
            if (unit_end && c + 1 < nch) enter_state(cs.un);   // the next unit starts
            if (full_mode && c + 1 < nch) {
                // Yoff(c) has read the incoming-state tile: stage S_in(c+1), issue Yoff(c+1)
                wait_or_fail(sh, a, &sh.barY[X], j & 1, kWhereBarY);
                write_sin();
                ptx::named_bar(kBarState, 128);
                if (mt == 0) issue_yoff(c + 1);
            }
            if (ptx::named_bar_any(kBarState, 128, *(volatile int*)&sh.abort != 0)) break;
        }
        if (mt == 0 && full_mode) {
            ptx::mma_commit(&sh.drain[2]);
            if (!ptx::mbar_wait(&sh.drain[2], 0, &sh.never, a.wait_iters)) fail(sh, a, kWhereDrain);
        }
    }
    pdl_wait();                                   // (the call's earlier launches end before this one)
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tb, kTmCols);
}

// Split aggregates of packed documents with initial states.  The aggregate
// passes start each split from zero (the first split from the first
// document's initial state), so the initial state of a document d > 0 that
// starts inside split s, at token st, and is still open at the split's end t1
// is added here:
//   S_s += exp(A_h sum_{t=st..t1-1} dt_t) init_d
// (the start token applies its own decay).  The split's total decay is
// already -inf there (the start resets the state).  One CTA per aggregate
// unit; dt is read with the heads' stride (neighbouring heads' CTAs share
// its sectors in L2).
constexpr int kDocInitThreads = 128;

__global__ void __launch_bounds__(kDocInitThreads) ssd_doc_init_agg(const FwdArgs a) {
    __shared__ float part[kDocInitThreads / 32];
    pdl_trigger();
    pdl_wait();                                // the split aggregates are complete
    const Unit un = unit_at<false>(a, blockIdx.x);
    if (un.s == (int)a.nsplit - 1) return;   // the last split's aggregate is never composed
    const int d = find_doc_tc(a.cu, a.ndocs, un.t1 - 1);
    const int st = __ldg(a.cu + d);
    if (d == 0 || st < un.t0) return;       // no document starts inside the split
    float sum = 0.f;
#pragma unroll 8
    for (int t = st + (int)threadIdx.x; t < un.t1; t += kDocInitThreads)
        sum += __ldg(a.dt + (size_t)t * a.H + un.h);   // packed documents: batch 1
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = sum;
    __syncthreads();
    const float tot = (part[0] + part[1]) + (part[2] + part[3]);
    const float dec = expf(__ldg(a.A + un.h) * tot);
    constexpr int PN4 = P * N / 4, kPer = PN4 / kDocInitThreads;
    float4* S = reinterpret_cast<float4*>(a.ws_state) + (size_t)un.ws * PN4 + threadIdx.x;
    const float4* I = reinterpret_cast<const float4*>(a.init) + ((size_t)d * a.H + un.h) * PN4 + threadIdx.x;
    float4 v[kPer], w[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {   // every load in flight before the first store
        v[k] = S[k * kDocInitThreads];
        w[k] = __ldg(I + k * kDocInitThreads);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k)
        S[k * kDocInitThreads] = make_float4(fmaf(dec, w[k].x, v[k].x), fmaf(dec, w[k].y, v[k].y),
                                             fmaf(dec, w[k].z, v[k].z), fmaf(dec, w[k].w, v[k].w));
}
static_assert(P * N / 4 % kDocInitThreads == 0, "whole float4 vectors per thread");
static_assert(kDocInitThreads == 128, "the reduction above sums four warps");

}  // namespace

cudaError_t launch_doc_init_agg(const FwdArgs& a, cudaStream_t st) {
    const int64_t grid = a.grid_units > 0 ? a.grid_units : a.batch * a.H * a.nsplit;
    if (grid <= 0 || !a.cu || !a.init) return cudaSuccess;
    return launch_kernel(ssd_doc_init_agg, (unsigned)grid, kDocInitThreads, 0, st, a.pdl != 0, a);
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

size_t tc_smem_bytes() { return kSmemBytes; }

bool tc_supported(int P_, int N_, int Q_, int dtype) {
    return P_ == P && N_ == N && Q_ == Q && dtype == SSD_BF16;
}

cudaError_t launch_tc(const FwdArgs& a, cudaStream_t st) {
    TcParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.a = a;
    if (prm.a.wait_iters == 0) prm.a.wait_iters = kDefaultWaitIters;
    if (!encode_4d(&prm.tm_x, a.x, P, a.H, a.L, a.batch) || !encode_4d(&prm.tm_B, a.B, N, a.G, a.L, a.batch) ||
        !encode_4d(&prm.tm_C, a.C, N, a.G, a.L, a.batch) || !encode_4d(&prm.tm_y, a.y, P, a.H, a.L, a.batch))
        return cudaErrorInvalidValue;
    const size_t smem = tc_smem_bytes();
    const bool full = a.mode == kModeFull, docs = a.cu != nullptr;
    // one CTA per unit; units of at most kPersistChunks chunks run on a persistent
    // grid of at most one CTA per SM instead
    int64_t grid = a.grid_units > 0 ? a.grid_units : a.batch * a.H * a.nsplit;
    const int nsm = device_sms();
    const bool persist = a.tail_units == 0 && (a.split_len + Q - 1) / Q <= kPersistChunks && nsm > 0 && grid > nsm;
    if (persist) grid = nsm;
    // packed documents whose initial or final states are asked for: the kernel with
    // the document events inside chunks
    const bool events = full && docs && (a.init != nullptr || a.fin != nullptr);
    void (*kern)(TcParams);
    if (events)
        kern = persist ? ssd_chunk_tc<true, true, true, true> : ssd_chunk_tc<true, true, false, true>;
    else if (persist)
        kern = full ? (docs ? ssd_chunk_tc<true, true, true> : ssd_chunk_tc<true, false, true>)
                    : (docs ? ssd_chunk_tc<false, true, true> : ssd_chunk_tc<false, false, true>);
    else
        kern = full ? (docs ? ssd_chunk_tc<true, true, false> : ssd_chunk_tc<true, false, false>)
                    : (docs ? ssd_chunk_tc<false, true, false> : ssd_chunk_tc<false, false, false>);
    // once per device and variant: the shared-memory opt-in, and the check that the
    // warpgroup register budgets fit the registers the CTA is launched with
    // (setmaxnreg.inc draws on that pool; a budget beyond it would wait forever)
    static std::atomic<uint8_t> ready[kMaxDevices][16];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::atomic<uint8_t>& rd = ready[dev][(events ? 8 : 0) | (full ? 4 : 0) | (docs ? 2 : 0) | (persist ? 1 : 0)];
    if (!rd.load(std::memory_order_acquire)) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
        const int need = kRegsIssue + 3 * kRegsMath;
        if (fa.numRegs * 4 < need) return cudaErrorInvalidConfiguration;
        rd.store(1, std::memory_order_release);
    }
    return launch_kernel(kern, (unsigned)grid, kThreads, smem, st, a.pdl != 0, prm);
}

}  // namespace ssd
