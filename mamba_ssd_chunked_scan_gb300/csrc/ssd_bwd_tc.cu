// Backward pass on the tensor cores (tcgen05 / TMEM / TMA) for the Mamba-2
// head shape: chunk Q = 128, P = 64, N = 128, bf16 x / B / C / dy / dx, fp32
// dt / A / D / states and fp32 accumulation.  The reverse-mode formulas are
// those of ssd_bwd_chunk (ssd_bwd.cu, which states them), by recomputation
// ("Parallel Scan and Hardware-Aware SSM Kernels", "Why the kernel matters
// more than the algorithm"), with every contraction one UMMA chain:
//
//   phase 1, chunks forwards:  S^T <- 2^tau S^T + B^T (w o x),  w_j = 2^{s_j} dt_j
//                              (the state entering each chunk is kept)
//   phase 2, chunks backwards (L = the decay mask of the hierarchy-aware
//   segsum, Lam = the adjoint of the state leaving the chunk):
//     G = C B^T, X = dy x^T              A1 = L o G, A2 = L o X (bf16 tiles)
//     V1 = A1^T dy, V2 = B Lam^T         v_j = V1_j + 2^{s_j} V2_j
//     SC = C S_in^T                      dx_j = dt_j v_j + D dy_j
//     dB_j = dt_j [A2^T C + (2^s o x) Lam^T]_j        (one accumulator, dt_j
//                                                      folded into both operands)
//     dC_i = [(A2 o dt) B + (2^p o dy) S_in^T]_i       (one accumulator)
//     Lam^T <- 2^tau Lam^T + C^T (2^p o dy)           (in TMEM)
//   and the per-token terms of ddt from row sums of those products and of
//   W = A1 o dt o X (its corner sums by warp transpose-reductions).
//
// One CTA of 384 threads per (batch row, head).  Warps 0-7 compute: thread
// (warp w, lane) owns chunk row (and state column) r = 32 (w % 4) + lane and
// the column half w / 4 of that row; both halves of a row run its segsum.
// Warp 8 issues: its lane 0 issues the TMA loads, the MMAs and the TMA stores,
// handed over through mbarriers, so the next chunk's loads start as soon as
// this chunk's last contraction is done (warps 9-11 only complete its
// warpgroup, whose registers go to the compute warps).  Every wait is bounded; a wait that
// runs out records SSD_ERR_TIMEOUT in the workspace status word, and the CTA
// drains its MMAs and copies, frees its TMEM and exits.
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
constexpr int kCompute = 256;                 // compute threads (warpgroups 0 and 1)
constexpr int kThreads = kCompute + 128;      // and the issue warpgroup (one lane issues)
// setmaxnreg budgets: registers are allocated per warpgroup, so the issue group
// hands its share to the compute groups
constexpr int kRegsIssue = 56, kRegsCompute = 224;   // 128 * (56 + 2 * 224) = 64512 <= 384 * 168
static_assert(128 * (kRegsIssue + 2 * kRegsCompute) <= kThreads * 168, "register split must fit the launch total");
constexpr int kBarCompute = 1;                // named barrier of the compute threads
// shared tiles (each 1024-byte aligned for the 128-byte swizzle)
constexpr uint32_t kTX = 0;           // x (row j, p); then 2^{s_j} x_j (phase 1: w_j x_j)
constexpr uint32_t kTDY = 16384;      // dy (row i, p); then 2^{p_i} dy_i
constexpr uint32_t kTB = 32768;       // B (row j, n in two 64-column slabs)
constexpr uint32_t kTC = 65536;       // C
constexpr uint32_t kTLam = 98304;     // Lam as (row n, p) bf16
constexpr uint32_t kTSin = 114688;    // S_in as (row n, p) bf16; then dx, staged for its store
constexpr uint32_t kT1 = 131072;      // A1 (row i, column j); then the dB share
constexpr uint32_t kT2 = 163840;      // A2 o dt (row i, column j); then the dC share
constexpr uint32_t kTiles = 196608;
// Phase 1 keeps two stages of (x, B): chunk c uses stage c & 1, stage 1's x in the
// S_in tile and its B in the A1 tile, so each load runs two chunks ahead.
// TMEM columns (phase 1: the state summary in columns 0-63 or 64-127, by chunk parity)
constexpr uint32_t kTmG = 0, kTmX = 128, kTmV2 = 256, kTmSC = 320, kTmV1 = 384, kTmLU = 448, kTmCols = 512;

// codes of the wait that gave up (WsHeader::where)
enum : uint32_t { kWhereLoad = 31, kWhereMma1 = 32, kWhereV1 = 33, kWhereDB = 34, kWhereDC = 35,
                  kWhereF = 36, kWhereDrain = 37, kWhereReady = 38, kWhereStores = 39 };

struct BwdTcSmall {
    SegsumLinShared<4> seg;
    alignas(16) float dts[Q];
    // per chunk parity (a chunk's token pass runs during the next chunk):
    float part[2][4][Q];    // per row block: partial corner sums of W (column half 0: t < 64, half 1: t >= 64)
    float F[2][Q];          // per row: the sum of W over column half 0
    float qv[2][4][Q];      // column half 1's partial row sums (vx, lbx, scdy, dy . x)
    float kred[2][8];       // per warp: partial <Lam, S_in>
    float red[16];
    float carry[3][4];      // warp totals of the token scans
    int docoff[12];         // per warp: chunks of the earlier documents (document units)
    uint64_t full, full1, mmaF, mma1, mma2, mmaV1, mmaDB, mmaDC, mmaLU, drain;   // loads and MMAs complete
    uint64_t rdyF, rdyA, rdyB, rdyC, rdyDB, rdyS;                   // compute warps -> issuer
    uint64_t stFreeS, stFreeT;   // the stores have read the S_in tile (dx), and the A1 / A2 tiles
    uint32_t tmem_base;
    int abort;
    int never;
};
static_assert(offsetof(BwdTcSmall, full) % 8 == 0, "mbarriers are 8-byte aligned");
constexpr size_t kSmemBytes = 1024 + kTiles + sizeof(BwdTcSmall);
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

struct BwdTcParams {
    CUtensorMap tm_x, tm_dy, tm_B, tm_C;   // loads (bf16)
    CUtensorMap tm_dx;                     // store (bf16)
    CUtensorMap tm_dB, tm_dC;              // stores of this head's shares (bf16)
    BwdArgs a;
};

// K-major operand of 128 rows with K = 128 (two 64-column slabs), k-step kk of 16
__device__ __forceinline__ uint64_t desc_k2(uint32_t base, int kk) {
    return ptx::sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
// K-major operand of 128 rows with K = 64 (one slab), k-step kk < 4
__device__ __forceinline__ uint64_t desc_k1(uint32_t base, int kk) {
    return ptx::sdesc_sw128(base + kk * 32, 16, 1024);
}
// MN-major operand, MN extent 64 (one block), k-step kk (16 rows of the tile)
__device__ __forceinline__ uint64_t desc_mn1(uint32_t base, int kk) {
    return ptx::sdesc_sw128(base + kk * 2048, 8192, 1024);
}
// MN-major operand, MN extent 128 (two 64-wide blocks, 16 KB apart), k-step kk
__device__ __forceinline__ uint64_t desc_mn2(uint32_t base, int kk) {
    return ptx::sdesc_sw128(base + kk * 2048, 16384, 1024);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// eight bf16 values times s, rounded to bf16 again
__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float s) {
    return make_uint4(pack_bf16(bf16lo(v.x) * s, bf16hi(v.x) * s), pack_bf16(bf16lo(v.y) * s, bf16hi(v.y) * s),
                      pack_bf16(bf16lo(v.z) * s, bf16hi(v.z) * s), pack_bf16(bf16lo(v.w) * s, bf16hi(v.w) * s));
}

// offset of element (row r, column j < 128) in a two-slab tile
__device__ __forceinline__ uint32_t off2(int r, int j) { return (uint32_t)(j >> 6) * 16384u + sw128_off(r, j & 63); }

__device__ __forceinline__ bool wait_bar(BwdTcSmall& sh, const BwdArgs& a, uint64_t* bar, uint32_t parity,
                                         uint32_t where) {
    if (ptx::mbar_wait(bar, parity, &sh.abort, a.wait_iters)) return true;
    if (!*(volatile int*)&sh.abort) {
        record_error(a.ws, SSD_ERR_TIMEOUT, where);
        *(volatile int*)&sh.abort = 1;
    }
    return false;
}

// one arrival per compute warp, after the warp's shared-memory writes (for the
// async proxy) and tensor-memory accesses
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
    ptx::fence_proxy_async();
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over the warp's 32 lanes of element (lane & 15) of each lane's
// 16-vector (a reduction and a transpose in 16 shuffles: each step hands half
// of the remaining elements to the partner lane, the last adds the two
// half-warps).
__device__ __forceinline__ float warp_transpose_sum16(float (&v)[16], int lane) {
#pragma unroll
    for (int h = 8; h >= 1; h >>= 1) {
        const bool up = (lane & h) != 0;
#pragma unroll
        for (int k = 0; k < h; ++k) {
            const float send = up ? v[k] : v[k + h];
            const float keep = up ? v[k + h] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, h);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// Document start (d >= 1) at token t of a packed row: its log-decay is -inf.
__device__ __forceinline__ bool doc_start_tc(const BwdArgs& a, int64_t t) {
    if (!a.cu) return false;
    int lo = 1, hi = a.ndocs - 1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int64_t v = __ldg(a.cu + mid);
        if (v == t) return true;
        if (v < t) lo = mid + 1; else hi = mid - 1;
    }
    return false;
}

// kDocu: document units (packed documents with their own states; BwdArgs::doc_units),
// a kernel instance of its own so that the whole-row and split units keep their
// register allocation.
template <bool kDocu>
__global__ void __launch_bounds__(kThreads, 1) ssd_bwd_tc(const __grid_constant__ BwdTcParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    BwdTcSmall& sh = *reinterpret_cast<BwdTcSmall*>(sm + kTiles);
    const BwdArgs& a = prm.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t s0 = ptx::smem_u32(sm);
    // unit = (b * H + h) * nsplit + s: split s of row b, head h.  A split enters
    // from the state the forward pass's split scan left in ws_sin (split 0: the
    // initial state) and leaves with the adjoint the reverse scan left in ws_lam
    // (the last split: dfin)
    const int64_t unit = blockIdx.x;
    const int nsplit = a.nsplit > 0 ? a.nsplit : 1;
    const int s = (int)(unit % nsplit);
    const int64_t bh = unit / nsplit;
    const int h = (int)(bh % a.H);
    const int b = (int)(bh / a.H);
    const int g = h / (a.H / a.G);
    const int64_t L = a.L;
    const int nch_all = (int)((L + Q - 1) / Q);
    const int cps = nsplit > 1 ? (int)(a.split_len / Q) : nch_all;   // chunks per split
    const int c0 = s * cps;                                          // this split's first chunk
    int nch = (c0 + cps < nch_all ? c0 + cps : nch_all) - c0;        // and its chunks (local c = 0 ..)
    const size_t PN = (size_t)P * N;
    float* ckpt = a.ws_ckpt + ((size_t)bh * nch_all + c0) * PN;
    // Document units (packed documents with their own states; batch 1, s = the document):
    // the document's tokens [T0, tend) in chunks from T0, entering from its initial
    // state and leaving with its final-state gradient.  The rows of its last chunk past
    // tend are padding: dt 0 (no decay, no input), their rows of the masks and of the
    // scaled dy zero, and that chunk's outputs written row by row (its tiles overlap
    // the next document's first rows).  Offsets are clamped, so invalid ones (which the
    // device check reports) keep every index in bounds.
    constexpr bool docu = kDocu;
    int64_t T0 = (int64_t)c0 * Q, tend = L;
    if (docu) {
        auto clampL = [&](int64_t v) { return v < 0 ? (int64_t)0 : v > L ? L : v; };
        T0 = clampL(__ldg(a.cu + s));
        tend = clampL(__ldg(a.cu + s + 1));
        if (tend < T0) tend = T0;
        nch = (int)((tend - T0 + Q - 1) / Q);
        // this document's first checkpoint slot: after the chunks of the head's earlier
        // documents (a block sum, completed after the barrier below)
        int part = 0;
        for (int e = (int)threadIdx.x; e < s; e += (int)blockDim.x) {
            const int64_t u0 = clampL(__ldg(a.cu + e)), u1 = clampL(__ldg(a.cu + e + 1));
            part += u1 > u0 ? (int)((u1 - u0 + Q - 1) / Q) : 0;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) sh.docoff[warp] = part;
    }

    if (threadIdx.x == 0) {
        ptx::mbar_init(&sh.full, 1);
        ptx::mbar_init(&sh.full1, 1);
        ptx::mbar_init(&sh.mmaF, 1);
        ptx::mbar_init(&sh.mma1, 1);
        ptx::mbar_init(&sh.mma2, 1);
        ptx::mbar_init(&sh.mmaV1, 1);
        ptx::mbar_init(&sh.mmaDB, 1);
        ptx::mbar_init(&sh.mmaDC, 1);
        ptx::mbar_init(&sh.mmaLU, 1);
        ptx::mbar_init(&sh.drain, 1);
        ptx::mbar_init(&sh.rdyF, 8);
        ptx::mbar_init(&sh.rdyA, 8);
        ptx::mbar_init(&sh.rdyB, 8);
        ptx::mbar_init(&sh.rdyC, 8);
        ptx::mbar_init(&sh.rdyDB, 8);
        ptx::mbar_init(&sh.rdyS, 8);
        ptx::mbar_init(&sh.stFreeS, 1);
        ptx::mbar_init(&sh.stFreeT, 1);
        sh.abort = 0;
        sh.never = 0;
        ptx::mbar_fence_init();
    }
    if (warp == 0) ptx::tmem_alloc(&sh.tmem_base, kTmCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tb = sh.tmem_base;
    if (docu) {
        int64_t off = 0;
        for (int w = 0; w < kThreads / 32; ++w) off += sh.docoff[w];
        const int64_t cap = (int64_t)nch_all + a.ndocs;   // checkpoint slots per head
        if (off + nch > cap) nch = 0;                     // (inconsistent offsets: no work)
        ckpt = a.ws_ckpt + ((size_t)h * cap + (size_t)off) * PN;
    }

    if (warp >= 8) {
        // ================================================================ issue warpgroup
        ptx::regs_dec<kRegsIssue>();
        if (warp == 8 && lane == 0) {
            ptx::prefetch_tmap(&prm.tm_x);
            ptx::prefetch_tmap(&prm.tm_dy);
            ptx::prefetch_tmap(&prm.tm_B);
            ptx::prefetch_tmap(&prm.tm_C);
            ptx::prefetch_tmap(&prm.tm_dx);
            ptx::prefetch_tmap(&prm.tm_dB);
            ptx::prefetch_tmap(&prm.tm_dC);
            // per stage: loads issued, and phases known complete (waited for by someone)
            uint32_t nissue[2] = {0, 0}, ndone[2] = {0, 0};
            auto load1 = [&](int c) {         // phase 1: x and B of chunk c, into stage c & 1
                const int st = c & 1;
                ++nissue[st];
                uint64_t* bar = st ? &sh.full1 : &sh.full;
                uint8_t* xt = sm + (st ? kTSin : kTX);
                uint8_t* bt = sm + (st ? kT1 : kTB);
                const int t0 = docu ? (int)(T0 + (int64_t)c * Q) : (c0 + c) * Q;
                ptx::mbar_expect_tx(bar, 16384u + 32768u);
                ptx::tma_load_4d(xt, &prm.tm_x, bar, 0, h, t0, b);
                ptx::tma_load_4d(bt, &prm.tm_B, bar, 0, g, t0, b);
                ptx::tma_load_4d(bt + 16384, &prm.tm_B, bar, 64, g, t0, b);
            };
            auto load2 = [&](int c) {         // phase 2: x, dy, B and C of chunk c; chunk c - 1 towards L2
                ++nissue[0];
                const int t0 = docu ? (int)(T0 + (int64_t)c * Q) : (c0 + c) * Q;
                ptx::mbar_expect_tx(&sh.full, 16384u * 2u + 32768u * 2u);
                ptx::tma_load_4d(sm + kTX, &prm.tm_x, &sh.full, 0, h, t0, b);
                ptx::tma_load_4d(sm + kTDY, &prm.tm_dy, &sh.full, 0, h, t0, b);
                ptx::tma_load_4d(sm + kTB, &prm.tm_B, &sh.full, 0, g, t0, b);
                ptx::tma_load_4d(sm + kTB + 16384, &prm.tm_B, &sh.full, 64, g, t0, b);
                ptx::tma_load_4d(sm + kTC, &prm.tm_C, &sh.full, 0, g, t0, b);
                ptx::tma_load_4d(sm + kTC + 16384, &prm.tm_C, &sh.full, 64, g, t0, b);
                if (c > 0) {
                    const int tp = t0 - Q;
                    ptx::bulk_prefetch_l2(ckpt + (size_t)(c - 1) * PN, (uint32_t)(PN * 4));
                    ptx::tma_prefetch_4d(&prm.tm_x, 0, h, tp, b);
                    ptx::tma_prefetch_4d(&prm.tm_dy, 0, h, tp, b);
                    ptx::tma_prefetch_4d(&prm.tm_B, 0, g, tp, b);
                    ptx::tma_prefetch_4d(&prm.tm_B, 64, g, tp, b);
                    ptx::tma_prefetch_4d(&prm.tm_C, 0, g, tp, b);
                    ptx::tma_prefetch_4d(&prm.tm_C, 64, g, tp, b);
                }
            };
            // ---- phase 1: the compute warps scale x once its load lands, then this
            // chunk's state summary goes to the TMEM columns of its parity
            if (nch > 0) load1(0);
            if (nch > 1) load1(1);
            for (int c = 0; c < nch; ++c) {
                const int st = c & 1;
                if (!wait_bar(sh, a, &sh.rdyF, c & 1, kWhereReady)) break;
                ++ndone[st];   // (the compute warps waited for this load before arriving)
                ptx::tc_fence_after();
                constexpr uint32_t id = ptx::idesc_bf16(128, 64, 1, 1);
                const uint32_t xt = s0 + (st ? kTSin : kTX), bt = s0 + (st ? kT1 : kTB);
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb + 64 * st, desc_mn2(bt, kk), desc_mn1(xt, kk), id, kk > 0);
                ptx::mma_commit(&sh.mmaF);
                if (!wait_bar(sh, a, &sh.mmaF, c & 1, kWhereF)) break;
                if (c + 2 < nch) load1(c + 2);   // the stage is free again
            }
            // ---- phase 2 (stage 0's barrier only)
            if (nch > 0 && !*(volatile int*)&sh.abort) load2(nch - 1);
            for (int k = 0; k < nch && !*(volatile int*)&sh.abort; ++k) {
                const int c = nch - 1 - k;
                const int t0 = docu ? (int)(T0 + (int64_t)c * Q) : (c0 + c) * Q;
                // a document's last chunk when it ends before the chunk does: the compute
                // threads write its rows (the groups stay, empty, for the counts below)
                const bool partial = docu && (int64_t)t0 + Q > tend;
                if (!wait_bar(sh, a, &sh.full, ndone[0] & 1, kWhereLoad)) break;
                ++ndone[0];
                // TMEM free: the last chunk's shares (or phase 1's state summaries) are read
                if (!wait_bar(sh, a, &sh.rdyS, k & 1, kWhereReady)) break;
                ptx::tc_fence_after();
                constexpr uint32_t idQQ = ptx::idesc_bf16(128, 128, 0, 0);
                constexpr uint32_t idQP = ptx::idesc_bf16(128, 64, 0, 1);
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb + kTmG, desc_k2(s0 + kTC, kk), desc_k2(s0 + kTB, kk), idQQ, kk > 0);
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk)
                    ptx::mma_ss(tb + kTmX, desc_k1(s0 + kTDY, kk), desc_k1(s0 + kTX, kk), idQQ, kk > 0);
                ptx::mma_commit(&sh.mma1);
                // the last chunk's stores (dB; dx | dC) have read their tiles
                if (k > 0) {
                    ptx::bulk_wait_read1();
                    ptx::mbar_arrive(&sh.stFreeS);
                    ptx::bulk_wait_read0();
                    ptx::mbar_arrive(&sh.stFreeT);
                }
                // B Lam^T and C S_in^T, once the Lam and S_in tiles are written
                if (!wait_bar(sh, a, &sh.rdyA, k & 1, kWhereReady)) break;
                ptx::tc_fence_after();
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb + kTmV2, desc_k2(s0 + kTB, kk), desc_mn1(s0 + kTLam, kk), idQP, kk > 0);
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ss(tb + kTmSC, desc_k2(s0 + kTC, kk), desc_mn1(s0 + kTSin, kk), idQP, kk > 0);
                ptx::mma_commit(&sh.mma2);
                // (L o G)^T dy; dB = (A2 o dt)^T C + (2^s o dt o x) Lam^T
                if (!wait_bar(sh, a, &sh.rdyB, k & 1, kWhereReady)) break;
                ptx::tc_fence_after();
                {
                    constexpr uint32_t idV = ptx::idesc_bf16(128, 64, 1, 1);
                    constexpr uint32_t idB1 = ptx::idesc_bf16(128, 128, 1, 1);
                    constexpr uint32_t idB2 = ptx::idesc_bf16(128, 128, 0, 0);
#pragma unroll 1
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ss(tb + kTmV1, desc_mn2(s0 + kT1, kk), desc_mn1(s0 + kTDY, kk), idV, kk > 0);
                    ptx::mma_commit(&sh.mmaV1);
#pragma unroll 1
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ss(tb + kTmG, desc_mn2(s0 + kT2, kk), desc_mn2(s0 + kTC, kk), idB1, kk > 0);
#pragma unroll 1
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_ss(tb + kTmG, desc_k1(s0 + kTX, kk), desc_k1(s0 + kTLam, kk), idB2, 1);
                    ptx::mma_commit(&sh.mmaDB);
                }
                // dC = (A2 o dt) B + (2^p o dy) S_in^T; Lam^T += C^T (2^p o dy)
                if (!wait_bar(sh, a, &sh.rdyC, k & 1, kWhereReady)) break;
                ptx::tc_fence_after();
                {
                    constexpr uint32_t idC1 = ptx::idesc_bf16(128, 128, 0, 1);
                    constexpr uint32_t idC2 = ptx::idesc_bf16(128, 128, 0, 0);
                    constexpr uint32_t idL = ptx::idesc_bf16(128, 64, 1, 1);
#pragma unroll 1
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ss(tb + kTmX, desc_k2(s0 + kT2, kk), desc_mn2(s0 + kTB, kk), idC1, kk > 0);
#pragma unroll 1
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_ss(tb + kTmX, desc_k1(s0 + kTDY, kk), desc_k1(s0 + kTSin, kk), idC2, 1);
                    ptx::mma_commit(&sh.mmaDC);
#pragma unroll 1
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ss(tb + kTmLU, desc_mn2(s0 + kTC, kk), desc_mn1(s0 + kTDY, kk), idL, 1);
                    ptx::mma_commit(&sh.mmaLU);
                }
                // every contraction of the chunk is done: its tiles take the next chunk's loads
                if (!wait_bar(sh, a, &sh.mmaLU, k & 1, kWhereDC)) break;
                if (c > 0) load2(c - 1);
                // the staged dB share, then dx and the dC share: their stores (rows past
                // the end are clipped), in three groups
                if (!wait_bar(sh, a, &sh.rdyDB, k & 1, kWhereStores)) break;
                if (!partial) {
                    ptx::tma_store_4d(&prm.tm_dB, sm + kT1, 0, h, t0, b);
                    ptx::tma_store_4d(&prm.tm_dB, sm + kT1 + 16384, 64, h, t0, b);
                }
                ptx::bulk_commit();
                if (!wait_bar(sh, a, &sh.rdyS, (k + 1) & 1, kWhereStores)) break;
                if (!partial) ptx::tma_store_4d(&prm.tm_dx, sm + kTSin, 0, h, t0, b);
                ptx::bulk_commit();
                if (!partial) {
                    ptx::tma_store_4d(&prm.tm_dC, sm + kT2, 0, h, t0, b);
                    ptx::tma_store_4d(&prm.tm_dC, sm + kT2 + 16384, 64, h, t0, b);
                }
                ptx::bulk_commit();
            }
            // drain: every MMA issued has completed, the last load issued has landed,
            // and the stores are complete
            ptx::mma_commit(&sh.drain);
            if (!ptx::mbar_wait(&sh.drain, 0, &sh.never, a.wait_iters)) record_error(a.ws, SSD_ERR_TIMEOUT, kWhereDrain);
            for (int st = 0; st < 2; ++st)
                if (nissue[st] > ndone[st] && !ptx::mbar_wait(st ? &sh.full1 : &sh.full, (nissue[st] - 1) & 1,
                                                             &sh.never, a.wait_iters))
                    record_error(a.ws, SSD_ERR_TIMEOUT, kWhereDrain);
            ptx::bulk_wait0();
        } else if (warp == 9 && blockIdx.x == 0 && a.cu) {
            // an idle warp checks the call's packed-document offsets
            check_cu_seqlens(a.cu, a.ndocs, a.L, a.ws, lane, 32);
        }
        __syncwarp();
    } else {
        // ================================================================ compute warps
        ptx::regs_inc<kRegsCompute>();
        const int rb = warp & 3, hf = warp >> 2;   // row block (TMEM lane quarter), column half
        const int r = 32 * rb + lane;              // chunk row = state column = TMEM lane
        const uint32_t lane_addr = tb + ((uint32_t)(32 * rb) << 16);
        const float A2 = a.A[h] * kLog2e;
        const float Ah = a.A[h];
        const float Dh = a.D ? a.D[h] : 0.f;
        uint32_t nfull = 0;
        auto dt_at = [&](int64_t t) { return t < (docu ? tend : L) ? __ldg(a.dt + ((size_t)b * L + t) * a.H + h) : 0.f; };
        // the chunk's log-decays into the segsum input, and dt (column half 0 writes them)
        auto decays = [&](float d, bool start) {
            if (hf == 0) {
                sh.seg.a[r] = ex2_approx(start ? -INFINITY : d * A2);   // 0 at a document start, 1 past the end
                sh.dts[r] = d;
            }
        };

        // ------------------------------------------------------------ phase 1
        // Chunk c's segsum runs while chunk c - 1's state summary is on the tensor
        // cores; then S (the state entering chunk c) is updated and kept.
        float S[32];   // S^T[n = r][p], this half's p
        {
            const float* s_in = docu  ? (a.init ? a.init + ((size_t)s * a.H + h) * PN : nullptr)
                                : s > 0 ? a.ws_sin + ((size_t)bh * nsplit + s - 1) * PN
                                        : (a.init ? a.init + (size_t)bh * PN : nullptr);
#pragma unroll
            for (int p = 0; p < 32; ++p) S[p] = s_in ? s_in[(size_t)(32 * hf + p) * N + r] : 0.f;
        }
        float etau_prev = 0.f;
        float d1_next = dt_at((docu ? T0 : (int64_t)c0 * Q) + r);   // (the split's first chunk)
        for (int c = 0; c < nch; ++c) {
            const int64_t t0 = docu ? T0 + (int64_t)c * Q : (int64_t)(c0 + c) * Q;
            const float d = d1_next;   // (loaded a chunk earlier)
            decays(d, !docu && t0 + r < L && doc_start_tc(a, t0 + r));
            d1_next = c + 1 < nch ? dt_at(t0 + Q + r) : 0.f;
            ptx::named_bar(kBarCompute, kCompute);
            SegsumLinRow<4> row;
            segsum_lin_phase1<4>(sh.seg, row, rb, lane, hf == 0);
            ptx::named_bar(kBarCompute, kCompute);
            segsum_lin_phase2<4>(sh.seg, row, rb, lane, hf == 0);
            ptx::named_bar(kBarCompute, kCompute);
            const float w = segsum_lin_suffix<4>(sh.seg, r) * d;
            const float etau = sh.seg.tauL;
            if (c > 0) {   // S <- 2^tau S + the summary of chunk c - 1
                wait_bar(sh, a, &sh.mmaF, (c - 1) & 1, kWhereF);
                ptx::tc_fence_after();
                uint32_t dd[32];
                ptx::tmem_load32(lane_addr + 64 * ((c - 1) & 1) + 32 * hf, dd);
#pragma unroll
                for (int p = 0; p < 32; ++p) S[p] = fmaf(etau_prev, S[p], __uint_as_float(dd[p]));
            }
            etau_prev = etau;
#pragma unroll
            for (int p = 0; p < 32; ++p) ckpt[(size_t)c * PN + (size_t)(32 * hf + p) * N + r] = S[p];
            wait_bar(sh, a, (c & 1) ? &sh.full1 : &sh.full, (c >> 1) & 1, kWhereLoad);
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // w_j x_j in place (row j = r, this half's p)
                uint4* px = reinterpret_cast<uint4*>(sm + ((c & 1) ? kTSin : kTX) + sw128_off(r, 32 * hf + 8 * q));
                *px = scale_bf16x8(*px, w);
            }
            warp_arrive(&sh.rdyF, lane);
        }
        // (the last chunk's summary is not needed; the issue warp waits for it before
        // phase 2's loads)
        warp_arrive(&sh.rdyS, lane);   // the state summaries are read: TMEM free for phase 2
        nfull = (uint32_t)(nch + 1) / 2;   // phase 1's uses of stage 0's barrier

        // ------------------------------------------------------------ phase 2
        // Lam^T (lane n, column p) lives in TMEM: each chunk scales it by 2^tau in
        // place and the update contraction accumulates onto it.  It starts as the
        // adjoint of the state leaving this split: dfin for the last split, else
        // the reverse scan's slot s + 1
        {
            const float* lam_out = docu ? (a.dfin ? a.dfin + ((size_t)s * a.H + h) * PN : nullptr)
                                   : s + 1 < nsplit ? a.ws_lam + ((size_t)bh * nsplit + s + 1) * PN
                                                    : (a.dfin ? a.dfin + (size_t)bh * PN : nullptr);
            uint32_t v[16];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    v[e] = __float_as_uint(lam_out ? lam_out[(size_t)(32 * hf + 16 * q + e) * N + r] : 0.f);
                ptx::tmem_st16(lane_addr + kTmLU + 32 * hf + 16 * q, v);
            }
            ptx::tmem_st_wait();
        }
        float dA_acc = 0.f, dD_acc = 0.f;
        // a chunk's per-token values, for its token pass
        struct Tok {
            float vx, lbx, scdy, ddv, es, ep, d, etau;
            int64_t t0;
            bool start, valid;
        };
        Tok prev{};
        // ddt of token t = r, dA and dD (column half 0 owns the token), from the chunk's
        // shared values in buffer pb
        auto token_pass = [&](const Tok& T, int pb) {
            const float K = ((sh.kred[pb][0] + sh.kred[pb][1]) + (sh.kred[pb][2] + sh.kred[pb][3])) +
                            ((sh.kred[pb][4] + sh.kred[pb][5]) + (sh.kred[pb][6] + sh.kred[pb][7]));
            const float vx = T.vx + sh.qv[pb][0][r], lbx = T.lbx + sh.qv[pb][1][r];
            const float scdy = T.scdy + sh.qv[pb][2][r], ddv = T.ddv + sh.qv[pb][3][r];
            // U_t = sum_{i >= t} 2^{p_i} scdy_i, V_t = sum_{j <= t} 2^{s_j} dt_j lbx_j,
            // F_t = sum_{i >= t} F_i (the rows' totals of W over column half 0)
            float u = T.ep * scdy, v = T.es * T.d * lbx, f = sh.F[pb][r];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float tu = __shfl_down_sync(0xffffffffu, u, o);
                const float tf = __shfl_down_sync(0xffffffffu, f, o);
                const float tv = __shfl_up_sync(0xffffffffu, v, o);
                if (lane + o < 32) {
                    u += tu;
                    f += tf;
                }
                if (lane >= o) v += tv;
            }
            if (hf == 0) {
                if (lane == 0) {   // the warp's totals
                    sh.carry[0][rb] = u;
                    sh.carry[2][rb] = f;
                }
                if (lane == 31) sh.carry[1][rb] = v;
            }
            ptx::named_bar(kBarCompute, kCompute);
            for (int w = rb + 1; w < 4; ++w) {
                u += sh.carry[0][w];
                f += sh.carry[2][w];
            }
            for (int w = rb - 1; w >= 0; --w) v += sh.carry[1][w];
            // corner sums: column half 0's transposed sums hold t < 64 in full; for
            // t >= 64 half 1's, plus the first-half totals F_i of the rows i >= t
            const float rv = ((sh.part[pb][0][r] + sh.part[pb][1][r]) + (sh.part[pb][2][r] + sh.part[pb][3][r])) +
                             (r >= 64 ? f : 0.f);
            // (a document start's decay is not dt A: it is 0, and so is its gradient)
            const float dl = T.start ? 0.f : rv + u + v + T.etau * K - T.d * vx;
            if (hf == 0) {
                if (T.valid) a.ddt[((size_t)b * L + T.t0 + r) * a.H + h] = fmaf(Ah, dl, vx);
                if (!docu || T.valid) {   // (document units: a padding row's dy . x is not zero)
                    dA_acc = fmaf(T.d, dl, dA_acc);
                    dD_acc += ddv;
                }
            }
        };
        float d_next = nch > 0 ? dt_at((docu ? T0 + (int64_t)(nch - 1) * Q : (int64_t)(c0 + nch - 1) * Q) + r) : 0.f;
        for (int k = 0; k < nch; ++k) {
            const int c = nch - 1 - k;
            // (the whole-row and split instance keeps its own expressions: fewer live registers)
            const int64_t t0 = docu ? T0 + (int64_t)c * Q : (int64_t)(c0 + c) * Q;
            const bool valid = t0 + r < (docu ? tend : L);
            const bool partial = docu && t0 + Q > tend;   // (its rows are written by this thread)
            const float d = d_next;   // (loaded a chunk earlier)
            const bool start = valid && !docu && doc_start_tc(a, t0 + r);
            decays(d, start);
            d_next = c > 0 ? dt_at(t0 - Q + r) : 0.f;
            ptx::named_bar(kBarCompute, kCompute);
            SegsumLinRow<4> row;
            segsum_lin_phase1<4>(sh.seg, row, rb, lane, hf == 0);
            ptx::named_bar(kBarCompute, kCompute);
            segsum_lin_phase2<4>(sh.seg, row, rb, lane, hf == 0);
            ptx::named_bar(kBarCompute, kCompute);
            // the state entering the chunk (row n = r, this half's p; written by this
            // thread in phase 1), loaded while the last chunk's stores read their tiles
            float sv[32];
            {
                const float* src = ckpt + (size_t)c * PN + (size_t)(32 * hf) * N + r;
#pragma unroll
                for (int p = 0; p < 32; ++p) sv[p] = src[(size_t)p * N];
            }
            const float es_r = segsum_lin_suffix<4>(sh.seg, r);
            const float ep_r = (docu && !valid) ? 0.f : row.pe;   // (a padding row's dy enters nothing)
            const float etau = sh.seg.tauL;
            // the last chunk's dx store has read the S_in tile
            if (k > 0) wait_bar(sh, a, &sh.stFreeS, (k - 1) & 1, kWhereStores);
            // S_in and Lam as bf16 (row n = r, this half's p) operands; <Lam, S_in>;
            // Lam^T <- 2^tau Lam^T in TMEM, once the last update contraction is done
            if (k > 0) {
                wait_bar(sh, a, &sh.mmaLU, (k - 1) & 1, kWhereDC);
                ptx::tc_fence_after();
            }
            float kdot = 0.f;
            {
                uint32_t lv[32];
                ptx::tmem_load32(lane_addr + kTmLU + 32 * hf, lv);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float lf[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        lf[e] = __uint_as_float(lv[8 * q + e]);
                        kdot = fmaf(lf[e], sv[8 * q + e], kdot);
                    }
                    *reinterpret_cast<uint4*>(sm + kTSin + sw128_off(r, 32 * hf + 8 * q)) =
                        make_uint4(pack_bf16(sv[8 * q], sv[8 * q + 1]), pack_bf16(sv[8 * q + 2], sv[8 * q + 3]),
                                   pack_bf16(sv[8 * q + 4], sv[8 * q + 5]), pack_bf16(sv[8 * q + 6], sv[8 * q + 7]));
                    *reinterpret_cast<uint4*>(sm + kTLam + sw128_off(r, 32 * hf + 8 * q)) =
                        make_uint4(pack_bf16(lf[0], lf[1]), pack_bf16(lf[2], lf[3]), pack_bf16(lf[4], lf[5]),
                                   pack_bf16(lf[6], lf[7]));
                }
                uint32_t lo[16], hi[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    lo[e] = __float_as_uint(etau * __uint_as_float(lv[e]));
                    hi[e] = __float_as_uint(etau * __uint_as_float(lv[16 + e]));
                }
                ptx::tmem_st16(lane_addr + kTmLU + 32 * hf, lo);
                ptx::tmem_st16(lane_addr + kTmLU + 32 * hf + 16, hi);
                ptx::tmem_st_wait();
            }
            warp_arrive(&sh.rdyA, lane);
            kdot = warp_sum(kdot);
            if (lane == 0) sh.kred[k & 1][warp] = kdot;
            // the last chunk's token pass, while this chunk's first contractions run
            if (k > 0) token_pass(prev, (k - 1) & 1);
            // this row's x and dy (this half's p), kept for the epilogue before the
            // tiles are rescaled
            wait_bar(sh, a, &sh.full, nfull & 1, kWhereLoad);
            ++nfull;
            uint4 xv[4], dv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                xv[q] = *reinterpret_cast<const uint4*>(sm + kTX + sw128_off(r, 32 * hf + 8 * q));
                dv[q] = *reinterpret_cast<const uint4*>(sm + kTDY + sw128_off(r, 32 * hf + 8 * q));
            }
            wait_bar(sh, a, &sh.mma1, k & 1, kWhereMma1);
            ptx::tc_fence_after();
            // the last chunk's share stores have read the A1 and A2 tiles
            if (k > 0) wait_bar(sh, a, &sh.stFreeT, (k - 1) & 1, kWhereStores);
            // ---- this half's columns of A1 = L o G and A2 o dt = L o X o dt (bf16 tiles)
            // and the corner sums of W.  Column block cb of 32: L_rj = rf[cb] colL[j]
            // below the diagonal block (rank-one), wl[j - 32 cb] in it, 0 above it.
            // Half 1's row prefixes start at 0; the token pass adds half 0's row totals.
            {
                float zrun = 0.f;
#pragma unroll 1
                for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb) {
                    const float rfc = (cb == 0) ? row.rf[0] : (cb == 1) ? row.rf[1] : row.rf[2];
                    const bool below = cb < rb, diag = cb == rb;
                    uint32_t gr[32], xr[32];
                    ptx::tmem_load32x2(lane_addr + kTmG + 32 * cb, gr, lane_addr + kTmX + 32 * cb, xr);
#pragma unroll
                    for (int q16 = 0; q16 < 2; ++q16) {
                        const int j0 = 32 * cb + 16 * q16;
                        float z[16];
                        uint32_t p1[8], p2[8];
#pragma unroll
                        for (int cc = 0; cc < 16; cc += 2) {
                            const int kx = 16 * q16 + cc;
                            // (document units: a padding row of A1 and A2 is zero; past the
                            // row's end the loads are zero-filled instead)
                            const float l0 = (docu && !valid) ? 0.f
                                             : below          ? rfc * sh.seg.colL[j0 + cc]
                                             : diag           ? row.wl[kx]
                                                              : 0.f;
                            const float l1 = (docu && !valid) ? 0.f
                                             : below          ? rfc * sh.seg.colL[j0 + cc + 1]
                                             : diag           ? row.wl[kx + 1]
                                                              : 0.f;
                            const float x0 = __uint_as_float(xr[kx]), x1 = __uint_as_float(xr[kx + 1]);
                            p1[cc / 2] = pack_bf16(l0 * __uint_as_float(gr[kx]), l1 * __uint_as_float(gr[kx + 1]));
                            p2[cc / 2] = pack_bf16(l0 * x0 * sh.dts[j0 + cc], l1 * x1 * sh.dts[j0 + cc + 1]);
                            // W from the bf16 A1 that V1 contracts: the token's own term of
                            // <Lam_t, S_t> and of dt_t x_t . v_t then cancel in dl_t
                            zrun += bf16lo(p1[cc / 2]) * sh.dts[j0 + cc] * x0;
                            z[cc] = (j0 + cc <= r) ? zrun : 0.f;
                            zrun += bf16hi(p1[cc / 2]) * sh.dts[j0 + cc + 1] * x1;
                            z[cc + 1] = (j0 + cc + 1 <= r) ? zrun : 0.f;
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            *reinterpret_cast<uint4*>(sm + kT1 + off2(r, j0 + 8 * q)) =
                                make_uint4(p1[4 * q], p1[4 * q + 1], p1[4 * q + 2], p1[4 * q + 3]);
                            *reinterpret_cast<uint4*>(sm + kT2 + off2(r, j0 + 8 * q)) =
                                make_uint4(p2[4 * q], p2[4 * q + 1], p2[4 * q + 2], p2[4 * q + 3]);
                        }
                        const float zs = warp_transpose_sum16(z, lane);
                        if (lane < 16) sh.part[k & 1][rb][j0 + lane] = zs;
                    }
                }
                if (hf == 0) sh.F[k & 1][r] = zrun;
            }
            // x row j = r, this half's p, becomes 2^{s_j} dt_j x_j (the X contraction is done)
            const float xs = es_r * d;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(sm + kTX + sw128_off(r, 32 * hf + 8 * q)) = scale_bf16x8(xv[q], xs);
            warp_arrive(&sh.rdyB, lane);
            // ---- the per-token partial products V1 does not enter (row j = r), while V1
            // runs: <(B Lam^T)_j, x_j>, <(C S_in^T)_j, dy_j> and <dy_j, x_j>
            float vx = 0.f, lbx = 0.f, scdy = 0.f, ddv = 0.f;
            uint32_t v2[32];
            wait_bar(sh, a, &sh.mma2, k & 1, kWhereMma1);
            ptx::tc_fence_after();
            {
                uint32_t sc[32];
                ptx::tmem_load32x2(lane_addr + kTmV2 + 32 * hf, v2, lane_addr + kTmSC + 32 * hf, sc);
#pragma unroll
                for (int kx = 0; kx < 32; kx += 2) {
                    const int q = kx >> 3, e = kx & 7;
                    const uint32_t xw = e == 0 ? xv[q].x : e == 2 ? xv[q].y : e == 4 ? xv[q].z : xv[q].w;
                    const uint32_t dw = e == 0 ? dv[q].x : e == 2 ? dv[q].y : e == 4 ? dv[q].z : dv[q].w;
                    const float x0 = bf16lo(xw), x1 = bf16hi(xw), y0 = bf16lo(dw), y1 = bf16hi(dw);
                    lbx = fmaf(__uint_as_float(v2[kx]), x0, fmaf(__uint_as_float(v2[kx + 1]), x1, lbx));
                    scdy = fmaf(__uint_as_float(sc[kx]), y0, fmaf(__uint_as_float(sc[kx + 1]), y1, scdy));
                    ddv = fmaf(y0, x0, fmaf(y1, x1, ddv));
                }
            }
            wait_bar(sh, a, &sh.mmaV1, k & 1, kWhereV1);
            ptx::tc_fence_after();
            // ---- dy row i = r, this half's p, becomes 2^{p_i} dy_i (V1 has read dy)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(sm + kTDY + sw128_off(r, 32 * hf + 8 * q)) = scale_bf16x8(dv[q], ep_r);
            warp_arrive(&sh.rdyC, lane);
            // ---- dx (this half's p) and <v_j, x_j>, v_j = V1_j + 2^{s_j} V2_j
            uint32_t dxo[16];
            {
                uint32_t v1[32];
                ptx::tmem_load32(lane_addr + kTmV1 + 32 * hf, v1);
#pragma unroll
                for (int kx = 0; kx < 32; kx += 2) {
                    const int q = kx >> 3, e = kx & 7;
                    const uint32_t xw = e == 0 ? xv[q].x : e == 2 ? xv[q].y : e == 4 ? xv[q].z : xv[q].w;
                    const uint32_t dw = e == 0 ? dv[q].x : e == 2 ? dv[q].y : e == 4 ? dv[q].z : dv[q].w;
                    const float x0 = bf16lo(xw), x1 = bf16hi(xw), y0 = bf16lo(dw), y1 = bf16hi(dw);
                    const float v0 = fmaf(es_r, __uint_as_float(v2[kx]), __uint_as_float(v1[kx]));
                    const float v1v = fmaf(es_r, __uint_as_float(v2[kx + 1]), __uint_as_float(v1[kx + 1]));
                    vx = fmaf(v0, x0, fmaf(v1v, x1, vx));
                    dxo[kx / 2] = pack_bf16(fmaf(d, v0, Dh * y0), fmaf(d, v1v, Dh * y1));
                }
            }
            if (hf == 1) {
                sh.qv[k & 1][0][r] = vx;
                sh.qv[k & 1][1][r] = lbx;
                sh.qv[k & 1][2][r] = scdy;
                sh.qv[k & 1][3][r] = ddv;
            }
            // ---- this head's share of dB (row j = r, this half's columns) as bf16 over
            // A1, which V1 has finished reading
            wait_bar(sh, a, &sh.mmaDB, k & 1, kWhereDB);
            ptx::tc_fence_after();
#pragma unroll 1
            for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb) {
                uint32_t v[32];
                ptx::tmem_load32(lane_addr + kTmG + 32 * cb, v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 u = make_uint4(
                        pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                        pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                        pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                        pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                    *reinterpret_cast<uint4*>(sm + kT1 + off2(r, 32 * cb + 8 * q)) = u;
                    if (partial && valid)
                        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.ws_dB) +
                                                  ((size_t)(t0 + r) * a.H + h) * N + 32 * cb + 8 * q) = u;
                }
            }
            warp_arrive(&sh.rdyDB, lane);   // staged
            // ---- dC (row i = r, this half's columns) as bf16 over A2 o dt, dx over S_in,
            // once the dC and Lam contractions are done
            wait_bar(sh, a, &sh.mmaDC, k & 1, kWhereDC);
            ptx::tc_fence_after();
#pragma unroll 1
            for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb) {
                uint32_t v[32];
                ptx::tmem_load32(lane_addr + kTmX + 32 * cb, v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 u = make_uint4(
                        pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                        pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                        pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                        pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                    *reinterpret_cast<uint4*>(sm + kT2 + off2(r, 32 * cb + 8 * q)) = u;
                    if (partial && valid)
                        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.ws_dC) +
                                                  ((size_t)(t0 + r) * a.H + h) * N + 32 * cb + 8 * q) = u;
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 u = make_uint4(dxo[4 * q], dxo[4 * q + 1], dxo[4 * q + 2], dxo[4 * q + 3]);
                *reinterpret_cast<uint4*>(sm + kTSin + sw128_off(r, 32 * hf + 8 * q)) = u;
                if (partial && valid)
                    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.dx) + ((size_t)(t0 + r) * a.H + h) * P +
                                              32 * hf + 8 * q) = u;
            }
            warp_arrive(&sh.rdyS, lane);   // staged, and this chunk's TMEM is read
            prev = Tok{vx, lbx, scdy, ddv, es_r, ep_r, d, etau, t0, start, valid};
            if (ptx::named_bar_any(kBarCompute, kCompute, *(volatile int*)&sh.abort != 0)) break;
        }
        if (nch > 0 && !*(volatile int*)&sh.abort) token_pass(prev, (nch - 1) & 1);
        // ---- the adjoint of the initial state; this unit's dA and dD shares
        if (a.dinit && (docu ? nch > 0 : s == 0) && !*(volatile int*)&sh.abort) {
            wait_bar(sh, a, &sh.mmaLU, (nch - 1) & 1, kWhereDC);
            ptx::tc_fence_after();
            uint32_t l0[32];
            ptx::tmem_load32(lane_addr + kTmLU + 32 * hf, l0);
            const size_t di = docu ? (size_t)s * a.H + h : (size_t)bh;
#pragma unroll
            for (int p = 0; p < 32; ++p) a.dinit[di * PN + (size_t)(32 * hf + p) * N + r] = __uint_as_float(l0[p]);
        }
        dA_acc = warp_sum(dA_acc);
        dD_acc = warp_sum(dD_acc);
        ptx::named_bar(kBarCompute, kCompute);
        if (lane == 0) {
            sh.red[warp] = dA_acc;
            sh.red[8 + warp] = dD_acc;
        }
        ptx::named_bar(kBarCompute, kCompute);
        if (threadIdx.x == 0) {
            a.ws_dA[unit] = (sh.red[0] + sh.red[1]) + (sh.red[2] + sh.red[3]);
            a.ws_dD[unit] = (sh.red[8] + sh.red[9]) + (sh.red[10] + sh.red[11]);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tb, kTmCols);
}

}  // namespace

bool bwd_tc_supported(int P_, int N_, int dtype) { return P_ == P && N_ == N && dtype == SSD_BF16; }

cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t st) {
    BwdTcParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.a = a;
    if (prm.a.wait_iters == 0) prm.a.wait_iters = kDefaultWaitIters;
    if (!encode_4d(&prm.tm_x, a.x, P, a.H, a.L, a.batch) || !encode_4d(&prm.tm_dy, a.dy, P, a.H, a.L, a.batch) ||
        !encode_4d(&prm.tm_B, a.B, N, a.G, a.L, a.batch) || !encode_4d(&prm.tm_C, a.C, N, a.G, a.L, a.batch) ||
        !encode_4d(&prm.tm_dx, a.dx, P, a.H, a.L, a.batch) ||
        !encode_4d(&prm.tm_dB, a.ws_dB, N, a.H, a.L, a.batch) || !encode_4d(&prm.tm_dC, a.ws_dC, N, a.H, a.L, a.batch))
        return cudaErrorInvalidValue;
    void (*kern)(BwdTcParams) = a.doc_units ? ssd_bwd_tc<true> : ssd_bwd_tc<false>;
    static std::atomic<uint8_t> ready[kMaxDevices][2];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::atomic<uint8_t>& rd = ready[dev][a.doc_units ? 1 : 0];
    if (!rd.load(std::memory_order_acquire)) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)) !=
            cudaSuccess)
            return e;
        // the warpgroup budgets must fit the registers the CTA is launched with
        // (setmaxnreg.inc draws on that pool; a budget beyond it would wait forever)
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
        if (fa.numRegs * (kThreads / 128) < kRegsIssue + 2 * kRegsCompute) return cudaErrorInvalidConfiguration;
        rd.store(1, std::memory_order_release);
    }
    kern<<<(unsigned)(a.batch * a.H * (a.nsplit > 0 ? a.nsplit : 1)), kThreads, kSmemBytes, st>>>(prm);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_bwd_reduce(a, st);
}

}  // namespace ssd
