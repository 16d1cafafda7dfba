// Host-side declarations shared by the libssd CUDA sources.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssd {

struct WsHeader;

enum { kModeFull = 0, kModeAggregate = 1 };

// Polls a device-side wait of the tensor-core kernels makes before it gives up
// (each poll is an mbarrier try_wait, which may suspend the thread for a while;
// every wait also gives up after 2 s).
constexpr uint32_t kDefaultWaitIters = 1u << 26;

// Everything one launch of a chunk kernel needs (passed by value).
struct FwdArgs {
    int64_t batch, L;
    int H, P, N, G;
    int Q;                 // chunk the kernel uses
    int64_t split_len;     // tokens per split (== L rounded up when one split)
    int nsplit;
    int dtype;             // ssd_dtype_t
    int mode;              // kModeFull or kModeAggregate
    const void* x;
    const float* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const float* init;
    const int32_t* cu;
    int ndocs;
    void* y;
    float* fin;
    float* ws_tau;         // [batch * H * nsplit] natural-log split decays
    float* ws_state;       // [batch * H * nsplit * P * N] split aggregates (slot s); after the
                           // scan, slot s - 1 holds the state entering split s
    WsHeader* ws;
    // n / H, n / nsplit and n / (H / G) for 0 <= n < 2^31 as (mulhi(m, n) + n) >> l
    uint32_t divH_m, divH_l, divS_m, divS_l, divHG_m, divHG_l;
    // leftover-unit plan (tail_units > 0, one split otherwise): the (row, head) units
    // [0, tail_first) run whole, the last tail_units are cut into nsplit pieces of
    // split_len tokens; grid_units = CTAs of this launch (0: batch * H * nsplit)
    int tail_units;
    int64_t tail_first;
    int64_t grid_units;
    // bounded waits give up after this many polls (kDefaultWaitIters) or 2 s
    uint32_t wait_iters;
    // fault injection (test aid, 0 otherwise): the TMA producer issues no loads,
    // so every wait that depends on them runs out
    int stall_loads;
    // launched as a programmatic dependent of the call's previous launch (tensor-core
    // full pass, split scan, document-start aggregates)
    int pdl;
};

// One decode step (ssd_step): everything the launch needs.
struct StepArgs {
    int64_t batch;
    int H, P, N, G;
    int dtype;             // ssd_dtype_t of x, B, C and y
    const float* state_in;
    float* state_out;      // == state_in for an in-place step
    const void* x;
    const float* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    void* y;
};

// Backward pass (ssd_bwd): everything its two launches need.
struct BwdArgs {
    int64_t batch, L;
    int H, P, N, G;
    int Qb;                // backward chunk (tokens)
    int dtype;             // ssd_dtype_t of x, B, C, dy, dx, dB, dC
    const void* x;
    const float* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const float* init;
    const void* dy;
    const float* dfin;
    const int32_t* cu;     // packed documents (batch 1), or NULL
    int ndocs;
    void* dx;
    float* ddt;
    float* dA;
    void* dB;
    void* dC;
    float* dD;
    float* dinit;
    float* ws_ckpt;        // [batch * H * nchunks * P * N] state entering each chunk
    float* ws_dB;          // [batch * L * H * N] per-head shares of dB (fp32, or bf16: shares_bf16)
    float* ws_dC;          // [batch * L * H * N] per-head shares of dC
    int shares_bf16;       // the shares are bf16 (the tensor-core backward)
    float* ws_dA;          // [batch * H]
    float* ws_dD;          // [batch * H]
    WsHeader* ws;          // status word (the tensor-core kernel's bounded waits)
    // sequence splits of the tensor-core backward (nsplit 1: whole rows); units are
    // (b * H + h) * nsplit + s, and ws_dA / ws_dD hold one share per unit (the
    // CUDA-core kernel with packed documents: nsplit = ndocs, units h * ndocs + d)
    int nsplit;
    int64_t split_len;     // tokens per split, a multiple of 128
    const float* ws_sin;   // [batch * H * nsplit * P * N] slot s - 1: the state entering split s
    const float* ws_lam;   // [batch * H * nsplit * P * N] slot s + 1: the adjoint of the state leaving split s
    uint32_t wait_iters;   // poll cap of each bounded wait (0: the default)
    // packed documents with their own states on the tensor cores: units h * ndocs + d
    // (nsplit = ndocs), each document in chunks from its first token; ws_ckpt holds
    // L / 128 + ndocs chunks per head
    int doc_units;
};

// Gated RMS normalisation (ssd_gate_norm): everything its launch needs.
struct GateNormArgs {
    int64_t rows;
    int width, group_size;
    int dtype;             // ssd_dtype_t of y, z and out
    float eps;
    const void* y;
    const void* z;
    const float* weight;
    void* out;
};

// Constants of division by an invariant divisor d >= 1 through one high
// multiply and a shift (Granlund and Montgomery, "Division by Invariant
// Integers using Multiplication", 1994): l = ceil(log2 d),
// m = floor(2^32 (2^l - d) / d) + 1; then n / d = (mulhi(m, n) + n) >> l,
// exact for 0 <= n < 2^31 (the sum cannot wrap).
inline void fastdiv_consts(uint32_t d, uint32_t* m, uint32_t* l) {
    uint32_t k = 0;
    while ((1ull << k) < d) ++k;
    *l = k;
    *m = (uint32_t)((((1ull << k) - d) << 32) / d + 1);
}

constexpr int kMaxDevices = 256;   // device ordinals the per-device caches cover

// SM count of the current device (cached per device); 0 when no device is visible.
int device_sms();

size_t simt_smem_bytes(int Q, int P, int N);
cudaError_t launch_simt(const FwdArgs& a, cudaStream_t st);
cudaError_t launch_split_scan(const FwdArgs& a, cudaStream_t st);
// 4-D TMA map over a (batch, L, heads_or_groups, inner) bf16 tensor; box = one
// 64-element x 128-row tile of one head (group), 128-byte swizzle.
bool encode_4d(CUtensorMap* tm, const void* base, int64_t inner, int64_t mid, int64_t L, int64_t batch);
size_t tc_smem_bytes();
bool tc_supported(int P, int N, int Q, int dtype);
cudaError_t launch_tc(const FwdArgs& a, cudaStream_t st);
// adds the initial states of packed documents that start inside a split to the
// split aggregates (after the aggregate pass, before their composition)
cudaError_t launch_doc_init_agg(const FwdArgs& a, cudaStream_t st);
int agg_heads_per_cta(int H, int G);
cudaError_t launch_agg_tc(const FwdArgs& a, cudaStream_t st);
cudaError_t launch_agg_rev_tc(const FwdArgs& a, cudaStream_t st);
cudaError_t launch_split_rscan(const FwdArgs& a, const float* dfin, cudaStream_t st);
cudaError_t launch_gate_norm(const GateNormArgs& a, cudaStream_t st);
size_t bwd_smem_bytes(int Qb, int P, int N);
int bwd_chunk(int P, int N, size_t smem_limit);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t st);
// sums the per-head dB, dC shares over each group and the per-row dA, dD shares
cudaError_t launch_bwd_reduce(const BwdArgs& a, cudaStream_t st);
// the backward on the tensor cores: bf16, P = 64, N = 128, chunks of 128 tokens
bool bwd_tc_supported(int P, int N, int dtype);
constexpr int kBwdTcChunk = 128;
cudaError_t launch_bwd_tc(const BwdArgs& a, cudaStream_t st);
size_t step_smem_bytes(int P, int N);
cudaError_t launch_step(const StepArgs& a, cudaStream_t st);
cudaError_t launch_segsum_dump(const float* l2, int64_t nrows, int chunk, float* seg, float* L, float* pexp,
                               float* sfx, cudaStream_t st);

}  // namespace ssd
