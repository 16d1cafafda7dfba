// C ABI of libssd: argument checks, the split plan, and kernel dispatch.
// Nothing here allocates device memory; every launch is asynchronous on the
// caller's stream.
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "ssd_common.cuh"
#include "ssd_kernels.h"

using namespace ssd;

namespace ssd {

// SM count of the current device, looked up once per device and cached.
int device_sms() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();   // no device visible: clear the error it left
        return 0;
    }
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return 0;
    }
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

}  // namespace ssd

namespace {

constexpr int kSmemLimit = 227 * 1024;
constexpr int64_t kFallbackSMs = 152;   // SMs the automatic split plan assumes when no device is visible

constexpr int kStepMaxN = 512;    // dstate limit of the decode step (float4 vectors per lane)
constexpr int kStepMaxP = 2048;   // headdim limit of the decode step (shared-memory rows)

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_params(const ssd_params_t* p) {
    if (!p) return SSD_ERR_INVALID_ARG;
    if (p->batch < 1 || p->seqlen < 1 || p->nheads < 1 || p->headdim < 1 || p->dstate < 1 ||
        p->ngroups < 1)
        return SSD_ERR_INVALID_ARG;
    if (p->nheads % p->ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (p->dtype != SSD_F32 && p->dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (p->chunk != 64 && p->chunk != 128) return (p->chunk > 0) ? SSD_ERR_UNSUPPORTED : SSD_ERR_INVALID_ARG;
    if (p->split_len < 0 || (p->split_len % p->chunk) != 0) return SSD_ERR_INVALID_ARG;
    if (p->ndocs < 0) return SSD_ERR_INVALID_ARG;
    if (p->ndocs > 0 && p->batch != 1) return SSD_ERR_INVALID_ARG;
    // element counts must fit the 32-bit grid and index arithmetic
    if (p->batch * p->nheads > (int64_t)1 << 30) return SSD_ERR_UNSUPPORTED;
    // x/y rows must keep 16-byte alignment (vector and bulk copies)
    const int esz = p->dtype == SSD_BF16 ? 2 : 4;
    if ((p->headdim * esz) % 16 != 0 || (p->dstate * esz) % 16 != 0) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

// Automatic split plan (split_len = 0), for the current device's SM count S
// (152 when no device is visible).  With at least as many (row, head) units as
// SMs there is one split (the leftover-unit plan evens out the last wave).
// Otherwise each sequence is cut into n splits of at least 4 chunks:
// the smallest n in [ceil(S / units), 4 S / units] whose units fill their waves
// to at least 95 %, else the n with the best fill.  (Fewer splits means less
// boundary-state traffic; a part-empty last wave idles SMs for a whole split.)
int64_t plan_split_len(const ssd_params_t* p) {
    const int64_t L = p->seqlen;
    int64_t sl = p->split_len;
    if (sl == 0) {
        const int nsm = device_sms();
        const int64_t sms = nsm > 0 ? nsm : kFallbackSMs;   // this device's SMs
        const int64_t bh = p->batch * p->nheads;
        const int64_t nchunks = (L + p->chunk - 1) / p->chunk;
        int64_t n = 1;
        if (bh < sms) {
            const int64_t n_min = (sms + bh - 1) / bh;
            int64_t n_max = (4 * sms + bh - 1) / bh;
            if (n_max > nchunks / 4) n_max = nchunks / 4;
            if (n_max < 1) n_max = 1;
            if (n_min >= n_max) {
                n = n_max;
            } else {
                double best = -1.0;
                for (int64_t k = n_min; k <= n_max; ++k) {
                    const int64_t units = bh * k;
                    const double fill = (double)units / (double)(((units + sms - 1) / sms) * sms);
                    if (fill > best + 1e-12) {
                        best = fill;
                        n = k;
                    }
                    if (fill >= 0.95) break;
                }
            }
        }
        sl = (nchunks + n - 1) / n * p->chunk;
    }
    if (sl >= L) sl = (L + p->chunk - 1) / p->chunk * p->chunk;
    return sl;
}

int plan_nsplit(const ssd_params_t* p) {
    const int64_t sl = plan_split_len(p);
    return (int)((p->seqlen + sl - 1) / sl);
}

// SIMT kernel chunk: the caller's chunk when its shared-memory tiles fit,
// else 64 (the chunk size changes only the rounding, not the result).
int simt_chunk(const ssd_params_t* p) {
    if (simt_smem_bytes(p->chunk, p->headdim, p->dstate) <= (size_t)kSmemLimit) return p->chunk;
    if (simt_smem_bytes(64, p->headdim, p->dstate) <= (size_t)kSmemLimit) return 64;
    return 0;
}

// The tcgen05 kernel covers the Mamba-2 head shape in bf16 (with or without
// packed documents and initial states).
bool use_tc(const ssd_params_t* p) {
    if (!tc_supported(p->headdim, p->dstate, p->chunk, p->dtype)) return false;
    if (p->seqlen >= ((int64_t)1 << 31) - 256) return false;   // token indices are 32-bit TMA coordinates
    return true;
}

// Leftover-unit plan for the tensor-core kernel with one split.  One CTA runs
// one (row, head) unit, so U units on S SMs run in ceil(U / S) waves, and when
// U % S is small the last wave keeps most SMs idle for a whole unit (640 units
// on 152 SMs: the fifth wave holds 32).  Instead the T = U % S leftover units
// are cut into m pieces each ("GPU Hierarchy Meets Structured Matrices": the
// split-sequence algorithm): their split aggregates, the composition, then one
// full launch of the whole units followed by the pieces, so the last wave is
// about 1 / m of a unit long.
constexpr int64_t kTailStateBytes = (int64_t)4 << 20;

struct TailPlan {
    int T = 0, m = 0;
    int64_t split_len = 0;
};

bool plan_tail(const ssd_params_t* p, TailPlan* tp) {
    if (!tc_supported(p->headdim, p->dstate, p->chunk, p->dtype)) return false;
    if (plan_nsplit(p) != 1) return false;
    const int nsm = device_sms();
    if (nsm < 2) return false;   // no device here: no plan
    const int64_t units = p->batch * p->nheads;
    const int64_t T = units % nsm;
    const int64_t nch = (p->seqlen + p->chunk - 1) / p->chunk;
    if (units < nsm || T == 0 || nch < 4) return false;
    int64_t m = nsm / T;
    if (m > 8) m = 8;
    if (m > nch / 2) m = nch / 2;   // pieces of at least 2 chunks
    // keep the pieces' states within 4 MiB of workspace (so the library-owned
    // scratch of ssd_fwd_static_scratch covers every one-split problem)
    const int64_t state_bytes = (int64_t)p->headdim * p->dstate * 4;
    while (m >= 2 && T * m * state_bytes > kTailStateBytes) --m;
    if (m < 2) return false;
    tp->split_len = (nch + m - 1) / m * p->chunk;
    tp->m = (int)((p->seqlen + tp->split_len - 1) / tp->split_len);
    tp->T = (int)T;
    return tp->m >= 2;
}

WsLayout layout_for(const ssd_params_t* p, int ns, const TailPlan& tp) {
    if (tp.T > 0) return ws_layout(1, tp.T, p->headdim, p->dstate, tp.m);   // T * m pieces
    return ws_layout(p->batch, p->nheads, p->headdim, p->dstate, ns);
}

// Backward workspace: status header, the state entering every backward chunk,
// the per-head shares of dB and dC, and the per-row shares of dA and dD.
struct BwdLayout {
    int Qb = 0;
    bool tc = false;
    int nsplit = 1;            // sequence splits of the tensor-core backward
    int64_t split_len = 0;
    int shares = 1;            // dA / dD shares per (row, head): splits, or documents
    bool doc_units = false;    // tensor cores: packed documents with their own states as (head, document) units
    size_t ckpt = 0, dB = 0, dC = 0, dA = 0, dD = 0;
    size_t tau_f = 0, tau_r = 0, sin = 0, lam = 0;   // split aggregates, forwards and reverse
    size_t total = 0;
};

// The backward runs on the tensor cores for the bf16 Mamba-2 head shape (packed
// documents with initial states or final-state gradients, doc_states, as
// (head, document) units), and on CUDA cores otherwise.
bool bwd_use_tc(const ssd_params_t* p, bool doc_states) {
    (void)doc_states;
    return bwd_tc_supported(p->headdim, p->dstate, p->dtype) && p->seqlen < ((int64_t)1 << 31) - 256;
}

bool bwd_layout(const ssd_params_t* p, bool doc_states, BwdLayout* l) {
    if (check_params(p) != SSD_OK) return false;
    l->tc = bwd_use_tc(p, doc_states);
    l->Qb = l->tc ? kBwdTcChunk : bwd_chunk(p->headdim, p->dstate, kSmemLimit);
    if (l->Qb == 0) return false;
    const size_t bh = (size_t)p->batch * p->nheads;
    // (head, document) units, each document in chunks from its first token (one more
    // chunk per document at most): packed documents on CUDA cores, and on the tensor
    // cores those with their own states (without, they run as whole rows there)
    const bool per_doc = p->ndocs > 0 && (!l->tc || doc_states);
    l->doc_units = l->tc && per_doc;
    const size_t nch = (size_t)((p->seqlen + l->Qb - 1) / l->Qb) + (per_doc ? (size_t)p->ndocs : 0);
    const size_t PN = (size_t)p->headdim * p->dstate;
    // per-head shares of dB and dC: bf16 from the tensor-core backward, else fp32
    const size_t share_elem = l->tc ? 2 : 4;
    const size_t share = (size_t)p->batch * p->seqlen * p->nheads * p->dstate;
    // the tensor-core backward splits sequences when rows x heads leave SMs idle,
    // with the forward pass's automatic plan at its 128-token chunk; splits are
    // 4 chunks at least (the split aggregates' tensor-core kernel)
    l->nsplit = 1;
    l->split_len = p->seqlen;
    if (l->tc && !l->doc_units) {
        ssd_params_t q = *p;
        q.chunk = kBwdTcChunk;
        if (q.split_len > 0) q.split_len = (int32_t)((q.split_len + kBwdTcChunk - 1) / kBwdTcChunk * kBwdTcChunk);
        int64_t sl = plan_split_len(&q);
        if (sl < 4 * kBwdTcChunk) sl = 4 * kBwdTcChunk;
        if (sl < p->seqlen) {
            l->split_len = sl;
            l->nsplit = (int)((p->seqlen + sl - 1) / sl);
        }
    }
    const size_t ns = (size_t)l->nsplit;
    // document units give one dA / dD share per (head, document)
    l->shares = per_doc ? p->ndocs : l->nsplit;
    size_t o = sizeof(WsHeader);
    l->ckpt = o;  o = align_up(o + bh * nch * PN * sizeof(float), 256);
    l->dB = o;    o = align_up(o + share * share_elem, 256);
    l->dC = o;    o = align_up(o + share * share_elem, 256);
    l->dA = o;    o = align_up(o + bh * (size_t)l->shares * sizeof(float), 256);
    l->dD = o;    o = align_up(o + bh * (size_t)l->shares * sizeof(float), 256);
    if (ns > 1) {
        l->tau_f = o;  o = align_up(o + bh * ns * sizeof(float), 256);
        l->tau_r = o;  o = align_up(o + bh * ns * sizeof(float), 256);
        l->sin = o;    o = align_up(o + bh * ns * PN * sizeof(float), 256);
        l->lam = o;    o = align_up(o + bh * ns * PN * sizeof(float), 256);
    }
    l->total = o;
    return true;
}

}  // namespace

// ---------------------------------------------------------------------------
// Library-owned scratch for callers that cannot allocate device memory.
//
// Some callers of this library have no way to allocate device memory: a
// plugin running inside a host application that owns and budgets every
// device allocation, or a thin C caller that only holds pointers handed to it.
// ssd_fwd_static_scratch() serves them with a workspace that lives in this
// file-scope device array instead of caller memory.  Every GPU that loads the
// library keeps these bytes reserved until the process exits.
// ---------------------------------------------------------------------------
static constexpr size_t kStaticScratchBytes = (size_t)8 << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {
std::mutex g_static_mu;
void* g_static_ptr[256];   // device address of g_static_scratch, per device ordinal

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and cached.
int static_scratch_ptr(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return SSD_ERR_CUDA;
        g_static_ptr[dev] = ptr;
    }
    *out = g_static_ptr[dev];
    return SSD_OK;
}
}  // namespace

extern "C" {

const char* ssd_status_string(int s) {
    switch (s) {
        case SSD_OK: return "SSD_OK";
        case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG";
        case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED";
        case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE";
        case SSD_ERR_CUDA: return "SSD_ERR_CUDA";
        case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT";
        case SSD_ERR_DEVICE_CHECK: return "SSD_ERR_DEVICE_CHECK";
        default: return "SSD_ERR_UNKNOWN";
    }
}

size_t ssd_fwd_workspace_size(const ssd_params_t* p) {
    if (check_params(p) != SSD_OK) return 0;
    const int ns = plan_nsplit(p);
    TailPlan tp;
    plan_tail(p, &tp);
    return layout_for(p, ns, tp).total;
}

int ssd_fwd_plan(const ssd_params_t* p, int has_init, int has_final, int* launches, int* nsplits) {
    (void)has_final;
    if (check_params(p) != SSD_OK) return -1;
    const int ns = plan_nsplit(p);
    TailPlan tp;
    const bool tc = use_tc(p);
    const bool tail = tc && plan_tail(p, &tp);
    // aggregates (+ initial states of packed documents starting inside splits), composition, full pass
    const bool doc_init = tc && p->ndocs > 0 && has_init;
    if (launches) *launches = (ns > 1 || tail) ? (doc_init ? 4 : 3) : 1;
    if (nsplits) *nsplits = ns;
    return tc ? 1 : 0;
}

int ssd_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (!workspace || bytes < sizeof(WsHeader)) return SSD_ERR_WORKSPACE;
    if (cudaMemsetAsync(workspace, 0, sizeof(WsHeader), (cudaStream_t)stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    return SSD_OK;
}

int ssd_check_status_where(void* workspace, void* stream, uint32_t* where) {
    if (where) *where = 0;
    if (!workspace) return SSD_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    WsHeader h;
    if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
    if (h.status != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof(WsHeader), st) != cudaSuccess) return SSD_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
        if (where) *where = h.where;
    }
    return (int)h.status;
}

int ssd_check_status(void* workspace, void* stream) { return ssd_check_status_where(workspace, stream, nullptr); }

}  // extern "C"

namespace {

// Splits of at least this many chunks take the tensor-core aggregate kernel.
constexpr int kAggMinChunks = 4;

// Smallest wait cap the fault-injection entry point accepts: the drain waits
// share the cap and must outlast the MMAs and copies still in flight.
constexpr uint32_t kMinInjectWaitRounds = 4096;

// Events recorded around each launch of one forward call (the measurement entry
// point ssd_fwd_timed only).
constexpr int kMaxTimedLaunches = 4;
struct LaunchTimer {
    cudaEvent_t ev[2 * kMaxTimedLaunches];
    int n = 0;
};

// Fault injection for the time-out test (test aid): a wait cap and a producer
// that issues no loads.
struct FaultInject {
    uint32_t wait_iters;
    int stall_loads;
};

int fwd_impl(const ssd_params_t* p, const void* x, const float* dt, const float* A, const void* B,
             const void* C, const float* D, const float* init, const int32_t* cu, void* y,
             float* fin, void* workspace, size_t workspace_bytes, void* stream, LaunchTimer* tm,
             const FaultInject* fi = nullptr) {
    int rc = check_params(p);
    if (rc != SSD_OK) return rc;
    if (!x || !dt || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(y, 16) || !aligned(dt, 16))
        return SSD_ERR_INVALID_ARG;
    if (!aligned(A, 4) || (D && !aligned(D, 4)) || (init && !aligned(init, 16)) || (fin && !aligned(fin, 16)))
        return SSD_ERR_INVALID_ARG;
    if ((cu == nullptr) != (p->ndocs == 0)) return SSD_ERR_INVALID_ARG;
    if (cu && !aligned(cu, 4)) return SSD_ERR_INVALID_ARG;
    if ((const void*)y == x || (const void*)y == B || (const void*)y == C) return SSD_ERR_INVALID_ARG;
    const size_t need = ssd_fwd_workspace_size(p);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return SSD_ERR_WORKSPACE;

    const int ns = plan_nsplit(p);
    if (p->batch * p->nheads * ns >= ((int64_t)1 << 31)) return SSD_ERR_UNSUPPORTED;   // units are 32-bit
    TailPlan tp;
    plan_tail(p, &tp);
    const WsLayout wl = layout_for(p, ns, tp);
    FwdArgs a;
    memset(&a, 0, sizeof(a));
    a.batch = p->batch; a.L = p->seqlen;
    a.H = p->nheads; a.P = p->headdim; a.N = p->dstate; a.G = p->ngroups;
    a.split_len = plan_split_len(p);
    a.nsplit = ns;
    a.dtype = p->dtype;
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.init = init;
    a.cu = cu; a.ndocs = p->ndocs;
    a.y = y; a.fin = fin;
    a.ws = (WsHeader*)workspace;
    a.ws_tau = (float*)((char*)workspace + wl.tau_off);
    a.ws_state = (float*)((char*)workspace + wl.state_off);
    a.wait_iters = fi ? fi->wait_iters : kDefaultWaitIters;
    a.stall_loads = fi ? fi->stall_loads : 0;
    cudaStream_t st = (cudaStream_t)stream;

    fastdiv_consts((uint32_t)p->nheads, &a.divH_m, &a.divH_l);
    fastdiv_consts((uint32_t)ns, &a.divS_m, &a.divS_l);
    fastdiv_consts((uint32_t)(p->nheads / p->ngroups), &a.divHG_m, &a.divHG_l);
    const bool tc = use_tc(p);
    const bool doc_init = tc && cu && init;   // packed documents with initial states
    if (fi && !tc) return SSD_ERR_UNSUPPORTED;   // only the tensor-core kernel has device waits
    a.Q = tc ? p->chunk : simt_chunk(p);
    if (a.Q == 0) return SSD_ERR_UNSUPPORTED;
    auto timed = [&](cudaError_t (*fn)(const FwdArgs&, cudaStream_t), const FwdArgs& aa) {
        const bool rec = tm && tm->n < kMaxTimedLaunches;
        if (rec) cudaEventRecord(tm->ev[2 * tm->n], st);
        const cudaError_t e = fn(aa, st);
        if (rec) cudaEventRecord(tm->ev[2 * tm->n++ + 1], st);
        return e;
    };
    auto launch = [&](const FwdArgs& aa) { return timed(tc ? launch_tc : launch_simt, aa); };
    // the launches after the first start as programmatic dependents of the one before
    // (not when each launch is timed: the events between them serialise the launches)
    const int pdl = (tc && !tm) ? 1 : 0;
    if (tc && tp.T > 0) {
        // leftover-unit plan: aggregates of the pieces, their composition, then the
        // whole units and the pieces in one launch
        const int64_t units = p->batch * p->nheads;
        a.nsplit = tp.m;
        a.split_len = tp.split_len;
        a.tail_units = tp.T;
        a.tail_first = units - tp.T;
        fastdiv_consts((uint32_t)tp.m, &a.divS_m, &a.divS_l);
        a.mode = kModeAggregate;
        a.grid_units = (int64_t)tp.T * tp.m;
        if (launch(a) != cudaSuccess) return SSD_ERR_CUDA;
        a.pdl = pdl;
        if (doc_init && timed(launch_doc_init_agg, a) != cudaSuccess) return SSD_ERR_CUDA;
        FwdArgs sa = a;   // the scan runs over T "rows" of m splits
        sa.batch = 1;
        sa.H = tp.T;
        if (timed(launch_split_scan, sa) != cudaSuccess) return SSD_ERR_CUDA;
        a.mode = kModeFull;
        a.grid_units = a.tail_first + (int64_t)tp.T * tp.m;
        if (launch(a) != cudaSuccess) return SSD_ERR_CUDA;
        return SSD_OK;
    }
    if (ns > 1) {
        // split plan: the splits' aggregates, their composition, then the full pass.
        // Splits of several chunks take the tensor-core aggregate kernel (one
        // contraction per split and pair of heads); splits of one to three chunks
        // the full kernel's aggregate mode, whose persistent grid carries its
        // pipeline across such short units.
        a.mode = kModeAggregate;
        const bool agg_tc = tc && a.split_len >= (int64_t)kAggMinChunks * p->chunk;
        if ((agg_tc ? timed(launch_agg_tc, a) : launch(a)) != cudaSuccess) return SSD_ERR_CUDA;
        // (not after the persistent aggregate grid of short splits: the scan's blocks,
        // launched as soon as that grid starts, measured slower there)
        a.pdl = agg_tc ? pdl : 0;
        if (doc_init && timed(launch_doc_init_agg, a) != cudaSuccess) return SSD_ERR_CUDA;
        if (timed(launch_split_scan, a) != cudaSuccess) return SSD_ERR_CUDA;
    }
    a.mode = kModeFull;
    if (launch(a) != cudaSuccess) return SSD_ERR_CUDA;
    return SSD_OK;
}

}  // namespace

extern "C" {

int ssd_fwd(const ssd_params_t* p, const void* x, const float* dt, const float* A, const void* B,
            const void* C, const float* D, const float* init, const int32_t* cu, void* y,
            float* fin, void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_impl(p, x, dt, A, B, C, D, init, cu, y, fin, workspace, workspace_bytes, stream, nullptr);
}

int ssd_fwd_timed(const ssd_params_t* p, const void* x, const float* dt, const float* A, const void* B,
                  const void* C, const float* D, const float* init, const int32_t* cu, void* y,
                  float* fin, void* workspace, size_t workspace_bytes, void* stream,
                  float* ms_per_launch, int max_launches, int* nlaunches) {
    if (!ms_per_launch || max_launches < 1 || !nlaunches) return SSD_ERR_INVALID_ARG;
    LaunchTimer tm;
    int made = 0;
    for (; made < 2 * kMaxTimedLaunches; ++made)
        if (cudaEventCreate(&tm.ev[made]) != cudaSuccess) break;
    int rc = made == 2 * kMaxTimedLaunches ? SSD_OK : SSD_ERR_CUDA;
    if (rc == SSD_OK) rc = fwd_impl(p, x, dt, A, B, C, D, init, cu, y, fin, workspace, workspace_bytes, stream, &tm);
    *nlaunches = 0;
    if (rc == SSD_OK && tm.n > 0 && cudaEventSynchronize(tm.ev[2 * tm.n - 1]) != cudaSuccess) rc = SSD_ERR_CUDA;
    if (rc == SSD_OK) {
        for (int k = 0; k < tm.n && k < max_launches; ++k)
            if (cudaEventElapsedTime(&ms_per_launch[k], tm.ev[2 * k], tm.ev[2 * k + 1]) != cudaSuccess) rc = SSD_ERR_CUDA;
        *nlaunches = tm.n;
    }
    for (int k = 0; k < made; ++k) cudaEventDestroy(tm.ev[k]);
    return rc;
}

int ssd_fwd_fault_inject(const ssd_params_t* p, const void* x, const float* dt, const float* A, const void* B,
                         const void* C, const float* D, const float* init, const int32_t* cu, void* y,
                         float* fin, void* workspace, size_t workspace_bytes, uint32_t max_wait_rounds,
                         void* stream) {
    if (max_wait_rounds < kMinInjectWaitRounds) return SSD_ERR_INVALID_ARG;
    const FaultInject fi{max_wait_rounds, 1};
    return fwd_impl(p, x, dt, A, B, C, D, init, cu, y, fin, workspace, workspace_bytes, stream, nullptr, &fi);
}

int ssd_fwd_static_scratch(const ssd_params_t* p, const void* x, const float* dt, const float* A,
                           const void* B, const void* C, const float* D, const float* init,
                           const int32_t* cu, void* y, float* fin, void* stream) {
    int rc = check_params(p);
    if (rc != SSD_OK) return rc;
    const size_t need = ssd_fwd_workspace_size(p);
    if (need > kStaticScratchBytes) return SSD_ERR_WORKSPACE;   // problem too large for the static scratch
    void* ws = nullptr;
    if ((rc = static_scratch_ptr(&ws)) != SSD_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    // the array keeps the previous call's contents: the status word must start at zero
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess) return SSD_ERR_CUDA;
    rc = ssd_fwd(p, x, dt, A, B, C, D, init, cu, y, fin, ws, kStaticScratchBytes, stream);
    if (rc != SSD_OK) return rc;
    // synchronous: wait for the work and report what the device recorded
    return ssd_check_status(ws, stream);
}

size_t ssd_bwd_workspace_size(const ssd_params_t* p) {
    BwdLayout l;
    return bwd_layout(p, false, &l) ? l.total : 0;
}

size_t ssd_bwd_workspace_size_doc_states(const ssd_params_t* p) {
    BwdLayout l;
    return p && p->ndocs > 0 && bwd_layout(p, true, &l) ? l.total : 0;
}

int ssd_bwd(const ssd_params_t* p, const void* x, const float* dt, const float* A, const void* B,
            const void* C, const float* D, const float* init, const int32_t* cu, const void* dy,
            const float* dfin, void* dx, float* ddt, float* dA, void* dB, void* dC, float* dD,
            float* dinit, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_params(p);
    if (rc != SSD_OK) return rc;
    if ((cu == nullptr) != (p->ndocs == 0)) return SSD_ERR_INVALID_ARG;
    // packed documents with initial states, final-state gradients or initial-state
    // gradients: the CUDA-core kernel (its own, larger workspace layout)
    const bool doc_states = cu && (init || dfin || dinit);
    if (cu && !aligned(cu, 4)) return SSD_ERR_INVALID_ARG;
    if (bwd_chunk(p->headdim, p->dstate, kSmemLimit) == 0) return SSD_ERR_UNSUPPORTED;
    if (p->batch * p->nheads >= ((int64_t)1 << 31)) return SSD_ERR_UNSUPPORTED;
    if (!x || !dt || !A || !B || !C || !dy || !dx || !ddt || !dA || !dB || !dC) return SSD_ERR_INVALID_ARG;
    const void* in[] = {x, dt, A, B, C, D, init, dy, dfin};
    const void* out[] = {dx, ddt, dA, dB, dC, dD, dinit};
    for (const void* q : in)
        if (q && !aligned(q, 16)) return SSD_ERR_INVALID_ARG;
    for (const void* q : out) {
        if (q && !aligned(q, 16)) return SSD_ERR_INVALID_ARG;
        for (const void* r : in)
            if (q && q == r) return SSD_ERR_INVALID_ARG;   // outputs never alias inputs
    }
    BwdLayout l;
    if (!bwd_layout(p, doc_states, &l)) return SSD_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < l.total || !aligned(workspace, 256)) return SSD_ERR_WORKSPACE;
    BwdArgs a;
    memset(&a, 0, sizeof(a));
    a.batch = p->batch; a.L = p->seqlen;
    a.H = p->nheads; a.P = p->headdim; a.N = p->dstate; a.G = p->ngroups;
    a.Qb = l.Qb;
    a.dtype = p->dtype;
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.init = init; a.dy = dy; a.dfin = dfin;
    a.cu = cu; a.ndocs = p->ndocs;
    a.dx = dx; a.ddt = ddt; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = D ? dD : nullptr; a.dinit = dinit;
    char* ws = static_cast<char*>(workspace);
    a.ws_ckpt = (float*)(ws + l.ckpt);
    a.ws_dB = (float*)(ws + l.dB);
    a.ws_dC = (float*)(ws + l.dC);
    a.ws_dA = (float*)(ws + l.dA);
    a.ws_dD = (float*)(ws + l.dD);
    a.ws = (WsHeader*)ws;
    a.wait_iters = kDefaultWaitIters;
    a.shares_bf16 = l.tc ? 1 : 0;
    a.nsplit = l.shares;   // (the reduction sums this many dA / dD shares per (row, head))
    a.split_len = l.split_len;
    a.ws_sin = (const float*)(ws + l.sin);
    a.ws_lam = (const float*)(ws + l.lam);
    a.doc_units = l.doc_units ? 1 : 0;
    // a fresh status word for this call's bounded device waits
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess) return SSD_ERR_CUDA;
    if (l.nsplit > 1) {
        // the state entering each split (the forward pass's split aggregates and
        // their composition), then the adjoint leaving each split (the reverse
        // aggregates V_s = sum 2^{P_i} dy_i C_i^T and their composition from dfin)
        FwdArgs f;
        memset(&f, 0, sizeof(f));
        f.batch = p->batch; f.L = p->seqlen;
        f.H = p->nheads; f.P = p->headdim; f.N = p->dstate; f.G = p->ngroups;
        f.Q = kBwdTcChunk;
        f.dtype = p->dtype;
        f.x = x; f.dt = dt; f.A = A; f.B = B; f.C = C; f.D = D; f.init = init;
        f.cu = cu; f.ndocs = p->ndocs;
        f.mode = kModeAggregate;
        f.split_len = l.split_len;
        f.nsplit = l.nsplit;
        f.ws = (WsHeader*)ws;
        f.wait_iters = kDefaultWaitIters;
        f.ws_tau = (float*)(ws + l.tau_f);
        f.ws_state = (float*)(ws + l.sin);
        if (launch_agg_tc(f, st) != cudaSuccess || launch_split_scan(f, st) != cudaSuccess) return SSD_ERR_CUDA;
        FwdArgs r = f;
        r.x = dy; r.B = C; r.init = nullptr;
        r.ws_tau = (float*)(ws + l.tau_r);
        r.ws_state = (float*)(ws + l.lam);
        if (launch_agg_rev_tc(r, st) != cudaSuccess || launch_split_rscan(r, dfin, st) != cudaSuccess)
            return SSD_ERR_CUDA;
    }
    if ((l.tc ? launch_bwd_tc(a, st) : launch_bwd(a, st)) != cudaSuccess)
        return SSD_ERR_CUDA;
    return SSD_OK;
}

int ssd_gate_norm(int64_t rows, int32_t width, int32_t group_size, int32_t dtype, const void* y,
                  const void* z, const float* weight, float eps, void* out, void* stream) {
    if (rows < 1 || width < 1 || group_size < 1 || width % group_size != 0) return SSD_ERR_INVALID_ARG;
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || eps > 3.0e38f) return SSD_ERR_INVALID_ARG;   // rejects NaN and inf
    const int vec = dtype == SSD_BF16 ? 8 : 4;                          // elements per 16-byte vector
    if (group_size % vec != 0 || group_size > 8192) return SSD_ERR_UNSUPPORTED;
    if (rows * (width / group_size) >= ((int64_t)1 << 31)) return SSD_ERR_UNSUPPORTED;
    if (!y || !z || !weight || !out) return SSD_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(z, 16) || !aligned(out, 16) || !aligned(weight, 16)) return SSD_ERR_INVALID_ARG;
    GateNormArgs a;
    a.rows = rows; a.width = width; a.group_size = group_size; a.dtype = dtype; a.eps = eps;
    a.y = y; a.z = z; a.weight = weight; a.out = out;
    if (launch_gate_norm(a, (cudaStream_t)stream) != cudaSuccess) return SSD_ERR_CUDA;
    return SSD_OK;
}

int ssd_step(int64_t batch, int32_t nheads, int32_t headdim, int32_t dstate, int32_t ngroups, int32_t dtype,
             const float* state_in, float* state_out, const void* x, const float* dt, const float* A,
             const void* B, const void* C, const float* D, void* y, void* stream) {
    if (batch < 1 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1 || nheads % ngroups != 0)
        return SSD_ERR_INVALID_ARG;
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (dstate % 4 != 0 || dstate > kStepMaxN || headdim > kStepMaxP) return SSD_ERR_UNSUPPORTED;
    if (batch * nheads >= ((int64_t)1 << 31)) return SSD_ERR_UNSUPPORTED;   // one CTA per (row, head)
    if (!state_in || !state_out || !x || !dt || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    const size_t esz = dtype == SSD_BF16 ? 2 : 4;
    if (!aligned(state_in, 16) || !aligned(state_out, 16) || !aligned(dt, 4) || !aligned(A, 4) ||
        (D && !aligned(D, 4)) || !aligned(x, esz) || !aligned(B, esz) || !aligned(C, esz) || !aligned(y, esz))
        return SSD_ERR_INVALID_ARG;
    // the state is updated in place or written to a disjoint buffer
    const size_t sbytes = (size_t)batch * nheads * headdim * dstate * sizeof(float);
    const uintptr_t si = (uintptr_t)state_in, so = (uintptr_t)state_out;
    if (si != so && si < so + sbytes && so < si + sbytes) return SSD_ERR_INVALID_ARG;
    if (y == x || y == B || y == C || y == (const void*)state_in || y == (void*)state_out)
        return SSD_ERR_INVALID_ARG;
    StepArgs a;
    a.batch = batch; a.H = nheads; a.P = headdim; a.N = dstate; a.G = ngroups; a.dtype = dtype;
    a.state_in = state_in; a.state_out = state_out;
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.y = y;
    if (launch_step(a, (cudaStream_t)stream) != cudaSuccess) return SSD_ERR_CUDA;
    return SSD_OK;
}

int ssd_segsum_dump(const float* l2, int64_t nrows, int32_t chunk, float* seg, float* L, float* pexp,
                    float* sfx, void* stream) {
    if (!l2 || nrows < 0 || (chunk != 64 && chunk != 128)) return SSD_ERR_INVALID_ARG;
    if (nrows == 0) return SSD_OK;
    if (launch_segsum_dump(l2, nrows, chunk, seg, L, pexp, sfx, (cudaStream_t)stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    return SSD_OK;
}

}  // extern "C"
