/*
 * libssd: Mamba-2 structured-state-space-duality (SSD) chunked-scan forward
 * pass for NVIDIA GB300 (sm_103a).  C ABI: plain pointers and sizes only.
 *
 * The operation ("State Space Duality and Mamba-2", sections "The
 * Mathematical Bridge" and "The SSD Block Decomposition Algorithm"; the
 * discretisation is the selective-scan one of "NVIDIA Accelerates Mamba-2
 * Forward Kernel with CUDA Tile", where the decay and input matrices depend
 * on the step size dt):  per batch row b and head h, with group
 * g = h / (H / G),
 *
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t B_t^T        (P x N state)
 *     y_t = h_t C_t + D_h * x_t
 *
 * computed chunk by chunk: the intra-chunk block ((C B^T) o L) X with the
 * 1-semiseparable decay mask L_ij = exp(sum_{k=j+1..i} dt_k A_h), chunk
 * states B^T (decay o X), inter-chunk state passing and the off-diagonal
 * output C * state.  A sequence may also be cut into splits of split_len
 * tokens that run in parallel and are joined by composing their states
 * ("GPU Hierarchy Meets Structured Matrices", abstract: the split-sequence
 * algorithm; "Parallel Scan and Hardware-Aware SSM Kernels", "The scan": the
 * affine-step composition).  Packed documents (cu_seqlens) restart the state
 * at every document start (same page, "When it breaks"): document d starts
 * from initial_states[d] (or zero), which its first token decays like any
 * carried state.
 *
 * Layouts (all row-major, contiguous, device memory, 16-byte aligned bases):
 *   x, y            (batch, seqlen, nheads, headdim)      dtype
 *   dt              (batch, seqlen, nheads)               fp32, >= 0 (post-softplus)
 *   A, D            (nheads)                              fp32 (A <= 0; D optional)
 *   B, C            (batch, seqlen, ngroups, dstate)      dtype
 *   initial_states  (nstates, nheads, headdim, dstate)    fp32, optional (zeros)
 *   final_states    (nstates, nheads, headdim, dstate)    fp32, optional
 *   cu_seqlens      (ndocs + 1) int32, cu[0] = 0 < cu[1] < ... < cu[ndocs] = seqlen
 *                   (no empty document), optional.  The offsets are in device
 *                   memory, so the host cannot check them; the last launch of
 *                   ssd_fwd() / ssd_bwd() does, and records SSD_ERR_DEVICE_CHECK
 *                   (where 40) in the workspace status word when they break
 *                   this rule.  The kernels keep every index in bounds either
 *                   way; the outputs are then undefined.
 *   nstates = ndocs when cu_seqlens is given (then batch must be 1), else batch.
 *
 * Ownership: the caller owns every buffer; the library keeps no pointer past
 * a call and allocates no device memory.  Calls are asynchronous on the given
 * stream (a cudaStream_t passed as void*; NULL = legacy default stream).
 *
 * Errors: argument errors return a status before anything is launched and
 * nothing is written.  A failed launch returns SSD_ERR_CUDA.  Errors found on
 * the device (a bounded wait that ran out) are recorded in a status word at
 * the start of the workspace and are read by ssd_check_status().
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or layout */
    SSD_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. chunk 256) */
    SSD_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    SSD_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    SSD_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out */
    SSD_ERR_DEVICE_CHECK = 6   /* a device-side consistency check failed (cu_seqlens) */
} ssd_status_t;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype_t;

typedef struct {
    int64_t batch;      /* batch rows (1 when cu_seqlens is given)                  */
    int64_t seqlen;     /* tokens per row (total packed length with cu_seqlens)      */
    int32_t nheads;     /* H                                                         */
    int32_t headdim;    /* P                                                         */
    int32_t dstate;     /* N                                                         */
    int32_t ngroups;    /* G, H % G == 0; head h reads B, C of group h / (H / G)     */
    int32_t chunk;      /* Q: 64 or 128                                              */
    int32_t split_len;  /* tokens per split: a multiple of chunk; 0 = automatic;
                           >= seqlen = one split.  Never changes the result beyond
                           rounding.                                                 */
    int32_t ndocs;      /* documents when cu_seqlens is given, else 0                */
    int32_t dtype;      /* ssd_dtype_t of x, B, C and y                              */
} ssd_params_t;

/* Bytes of device workspace ssd_fwd() needs for these parameters (>= 256:
 * the first 256 bytes hold the device status word).  0 on invalid params. */
SSD_API size_t ssd_fwd_workspace_size(const ssd_params_t* p);

/* Zero the workspace's status word (async on `stream`).  Call once after
 * allocating a workspace; the status word then stays zero until a device
 * error is recorded, and ssd_check_status() clears it again. */
SSD_API int ssd_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* The SSD forward pass: y (and optionally final_states) from x, dt, A, B, C
 * and the optional D, initial_states and cu_seqlens, as defined above.
 * `workspace` is device scratch of at least ssd_fwd_workspace_size(p) bytes,
 * initialised once by ssd_workspace_init(); calls that share a workspace must
 * be ordered on one stream.  y must not alias any input.  final_states may
 * alias initial_states.  Bitwise deterministic for fixed inputs and params. */
SSD_API int ssd_fwd(const ssd_params_t* p,
            const void* x, const float* dt, const float* A,
            const void* B, const void* C, const float* D,
            const float* initial_states, const int32_t* cu_seqlens,
            void* y, float* final_states,
            void* workspace, size_t workspace_bytes, void* stream);

/* ssd_fwd() for measurement: the same call, with a CUDA event recorded on
 * `stream` before and after each of its kernel launches.  Synchronises on the
 * last event, writes the first min(launches, max_launches) launch durations in
 * milliseconds to ms_per_launch (in launch order: for split plans the
 * aggregate pass, the composition, then the full pass) and the launch count
 * to *nlaunches.  Creates and destroys its events on every call: meant for
 * benchmarks, not for the hot path.  Errors as ssd_fwd(); SSD_ERR_INVALID_ARG
 * when ms_per_launch or nlaunches is NULL or max_launches < 1. */
SSD_API int ssd_fwd_timed(const ssd_params_t* p,
            const void* x, const float* dt, const float* A,
            const void* B, const void* C, const float* D,
            const float* initial_states, const int32_t* cu_seqlens,
            void* y, float* final_states,
            void* workspace, size_t workspace_bytes, void* stream,
            float* ms_per_launch, int max_launches, int* nlaunches);

/* ssd_fwd() for callers that cannot allocate device memory (for example a
 * plugin inside a host application that owns every device allocation, or a
 * C caller that only holds the input and output pointers it was given).
 * The paper has no counterpart of this entry point.
 *
 * Same operation, arguments and layouts as ssd_fwd(), without a workspace:
 * the workspace is a library-owned device array of 8 MiB that every GPU
 * loading the library reserves until process exit.  Problems whose
 * ssd_fwd_workspace_size() exceeds 8 MiB are rejected with
 * SSD_ERR_WORKSPACE before anything is launched; single-split problems need
 * less than 4.01 MiB: the 256-byte status header, the pieces' log-decays
 * (4 bytes each, rounded up to 256 bytes) and their states (at most 4 MiB),
 * for the pieces the leftover-unit plan cuts the last wave's units into.  The
 * caller still passes all inputs and outputs.
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress) and keeps it for the life of the
 * process; make no call after resetting the device (cudaDeviceReset), which
 * invalidates the kept address.  Every call uses the same array: calls whose GPU work
 * overlaps (other streams or other host threads) race on it.  The call
 * clears the status word, enqueues the work on `stream`, then synchronises
 * the stream and returns the device status (SSD_OK or the first device
 * error).  It calls no allocating routine. */
SSD_API int ssd_fwd_static_scratch(const ssd_params_t* p,
            const void* x, const float* dt, const float* A,
            const void* B, const void* C, const float* D,
            const float* initial_states, const int32_t* cu_seqlens,
            void* y, float* final_states, void* stream);

/* Bytes of device workspace ssd_bwd() needs for these parameters; 0 when the
 * parameters are invalid or the backward pass does not support them. */
SSD_API size_t ssd_bwd_workspace_size(const ssd_params_t* p);

/* Bytes of device workspace ssd_bwd() needs for packed documents (ndocs > 0)
 * when the call passes initial_states, dfinal_states or dinitial_states: that
 * call runs one unit per (head, document), in chunks from each document's first
 * token (on the tensor cores for their shape, 128 tokens; else on CUDA cores,
 * at most 32), so its chunk-state layout holds up to ndocs more chunks per head
 * than whole rows need.
 * 0 when the parameters are invalid, ndocs is 0 or the backward pass does not
 * support them. */
SSD_API size_t ssd_bwd_workspace_size_doc_states(const ssd_params_t* p);

/* Backward pass of ssd_fwd(): the gradients of the scalar
 *     <dy, y> + <dfinal_states, final_states>
 * with respect to every input, where y and final_states are ssd_fwd()'s outputs
 * for the same inputs.  The states are recomputed from the inputs, as "Parallel
 * Scan and Hardware-Aware SSM Kernels" ("Why the kernel matters more than the
 * algorithm") describes: only the state entering each backward chunk is kept, in
 * the workspace.  bf16 with headdim 64 and dstate 128 (the Mamba-2 head
 * shape) runs on the tensor cores: chunks of 128 tokens, every contraction a
 * bf16 x bf16 -> fp32 MMA (the decay-masked Q x Q products, the adjoint and
 * the incoming state are rounded to bf16 as MMA operands; sums, scans and
 * the adjoint recurrence stay fp32).  When rows x heads leave SMs idle it
 * cuts each sequence into splits that run in parallel ("GPU Hierarchy Meets
 * Structured Matrices": the split-sequence algorithm, here for the adjoint
 * too): the forward pass's split aggregates and their composition give the
 * state entering each split, and reverse aggregates (sum of 2^{P_i} dy_i C_i^T
 * over a split, P_i the log-decays from the split's start through i) composed
 * from dfinal_states give the adjoint leaving it.  split_len in p sets the
 * split (0: automatic; rounded up to a multiple of 128, at least 512).  Every other shape, and fp32, runs on
 * CUDA cores in fp32 (bf16 inputs widened, bf16 gradients rounded once at the
 * end).
 *
 * Inputs: x, dt, A, B, C, D (optional), initial_states (optional: zeros) exactly
 * as for ssd_fwd(); dy (batch, seqlen, nheads, headdim) dtype;
 * dfinal_states (batch, nheads, headdim, dstate) fp32 or NULL (zeros); with
 * cu_seqlens, initial_states, dfinal_states and dinitial_states are per
 * document, (ndocs, nheads, headdim, dstate).
 * Outputs (written, not accumulated into):
 *   dx               (batch, seqlen, nheads, headdim)   dtype
 *   ddt              (batch, seqlen, nheads)            fp32
 *   dA               (nheads)                           fp32
 *   dB, dC           (batch, seqlen, ngroups, dstate)   dtype (summed over each group's heads)
 *   dD               (nheads) fp32, or NULL; written only when D is given
 *   dinitial_states  (batch, nheads, headdim, dstate)   fp32, or NULL
 * All pointers are device memory with 16-byte aligned bases; no output may equal
 * an input.  Packed documents (cu_seqlens with ndocs, batch 1; strictly
 * increasing, from 0 to seqlen) are independent sequences: no state and no
 * gradient crosses a document boundary.  Without per-document states the
 * tensor-core path for its shape runs whole rows (a -inf log-decay at each
 * document start); with initial_states, dfinal_states or dinitial_states every
 * path runs one unit per (head, document), walking the document's own chunks
 * from its first token: each document
 * starts from its initial state (its first token's decay applied to it), its
 * final state receives dfinal_states[d], and dinitial_states[d] is the
 * gradient of initial_states[d].  headdim * dstate > 8192 and shapes whose
 * tiles do not fit in shared memory return SSD_ERR_UNSUPPORTED.
 * `chunk` and `split_len` in p are validated; they change only the rounding.
 * `workspace`: at least ssd_bwd_workspace_size(p) bytes, or
 * ssd_bwd_workspace_size_doc_states(p) for packed documents with any of the
 * three states, 256-byte aligned (else SSD_ERR_WORKSPACE).  Asynchronous on `stream`; a status-word reset
 * and two launches (six with splits: the two aggregate passes and their
 * compositions first).  The tensor-core path's device waits are bounded: one that
 * runs out records SSD_ERR_TIMEOUT (where codes 31-39, or 21-26 from the
 * split aggregates) in the status word at
 * the start of `workspace`, read by ssd_check_status(); the CUDA-core path has
 * no device waits.  Bitwise deterministic (fixed summation orders). */
SSD_API int ssd_bwd(const ssd_params_t* p,
            const void* x, const float* dt, const float* A,
            const void* B, const void* C, const float* D,
            const float* initial_states, const int32_t* cu_seqlens,
            const void* dy, const float* dfinal_states,
            void* dx, float* ddt, float* dA, void* dB, void* dC, float* dD,
            float* dinitial_states,
            void* workspace, size_t workspace_bytes, void* stream);

/* Gated RMS normalisation of the scan's output in one pass ("NVIDIA Accelerates
 * Mamba-2 Forward Kernel with CUDA Tile", operator fusion: the scan is followed
 * by gating and normalisation, fused so the gated values never leave the chip).
 * For each row r and each group of group_size consecutive channels:
 *
 *     g[r,k]   = y[r,k] * silu(z[r,k]),   silu(v) = v / (1 + exp(-v))
 *     out[r,k] = g[r,k] / sqrt(mean_{k' in group} g[r,k']^2 + eps) * weight[k]
 *
 * (the Mamba-2 block's output gate and its grouped RMS norm, gate applied before
 * the norm).  Layouts: y, z, out (rows, width) dtype, row-major, contiguous,
 * 16-byte aligned; weight (width) fp32, 16-byte aligned.  rows = batch * seqlen and width =
 * nheads * headdim for ssd_fwd's y.  width must be a multiple of group_size;
 * group_size a multiple of 8 (bf16) or 4 (fp32) and at most 8192 (else
 * SSD_ERR_UNSUPPORTED); eps >= 0 and finite.  out may be y itself (in place).
 * One launch on `stream`, no workspace; bitwise deterministic. */
SSD_API int ssd_gate_norm(int64_t rows, int32_t width, int32_t group_size, int32_t dtype,
             const void* y, const void* z, const float* weight, float eps, void* out, void* stream);

/* One autoregressive (decode) step: a single new token per batch row from a
 * resident state.  "State Space Duality and Mamba-2", section "Performance and
 * Serving Economics": generation keeps a fixed-size recurrent state and costs
 * constant time and memory per token.  The step is the recurrence above taken
 * once per (b, h), g = h / (H / G):
 *
 *     state'[b,h] = exp(dt[b,h] A_h) state[b,h] + dt[b,h] x[b,h] B[b,g]^T
 *     y[b,h]      = state'[b,h] C[b,g] + D_h x[b,h]
 *
 * so a prefill by ssd_fwd() (final_states) followed by steps gives the same
 * outputs, up to rounding, as one ssd_fwd() over the whole sequence.
 *
 * Layouts (row-major, contiguous, device memory): the forward's layouts with
 * one token per row (seqlen = 1):
 *   state_in, state_out (batch, nheads, headdim, dstate)  fp32, 16-byte aligned
 *   x, y                (batch, nheads, headdim)          dtype
 *   dt                  (batch, nheads)                   fp32, >= 0
 *   A, D                (nheads)                          fp32 (D optional)
 *   B, C                (batch, ngroups, dstate)          dtype
 * state_out may equal state_in (an in-place update) or be a disjoint buffer;
 * any other overlap is an argument error, as is y equal to an input.
 * dtype is an ssd_dtype_t.  dstate must be a multiple of 4 and at most 512,
 * headdim at most 2048 (else SSD_ERR_UNSUPPORTED).
 *
 * No workspace and no device-side waits: the call enqueues one kernel on
 * `stream` and returns (SSD_OK, an argument error before any launch, or
 * SSD_ERR_CUDA for a failed launch).  It can be captured in a CUDA graph.
 * Bitwise deterministic. */
SSD_API int ssd_step(int64_t batch, int32_t nheads, int32_t headdim, int32_t dstate, int32_t ngroups,
             int32_t dtype, const float* state_in, float* state_out,
             const void* x, const float* dt, const float* A, const void* B, const void* C,
             const float* D, void* y, void* stream);

/* Synchronise `stream`, read the device status word of `workspace`, clear it,
 * and return it (SSD_OK when no device error was recorded). */
SSD_API int ssd_check_status(void* workspace, void* stream);

/* ssd_check_status(), also returning in *where (if not NULL) which device wait
 * recorded the error: 0 with SSD_OK, else a code of the tensor-core full-pass
 * kernel (1 stage free, 2 stage loaded, 3 mask ready, 4 output buffer free,
 * 5 state summary buffer free, 6 scaled-X tile ready, 7 chunk values free,
 * 8 state summary done, 9 C B^T done, 10 chunk values ready, 11 off-diagonal
 * output done, 12 drain of copies or MMAs in flight, 13 diagonal output done,
 * 14 C init_d^T done, 15 state terms of a chunk with document starts ready)
 * or of the split-aggregate kernel (21 stage free, 22 stage loaded, 23 scaled
 * tile ready, 24 split contraction done, 25 drain of copies in flight, 26 the
 * other scaling group's decay product ready); with SSD_ERR_DEVICE_CHECK, 40:
 * the packed-document offsets are not 0 = cu[0] < ... < cu[ndocs] = seqlen. */
SSD_API int ssd_check_status_where(void* workspace, void* stream, uint32_t* where);

/* Test aid for the device-side failure path: ssd_fwd() with an injected stall.
 * The tensor-core kernel's TMA producer issues no loads, and every bounded
 * wait gives up after max_wait_rounds polls of its barrier (ordinary calls
 * allow 2^26 polls, and every wait gives up after 2 s).  The waits that depend on the loads run out;
 * the first records SSD_ERR_TIMEOUT and its code in the status word, and
 * every CTA stops waiting, lets its copies and MMAs finish, frees its tensor
 * memory and exits.  y and final_states are undefined afterwards;
 * ssd_check_status_where() reports the error and clears it, and the
 * workspace serves ordinary calls again.  Arguments as ssd_fwd(); returns
 * SSD_ERR_INVALID_ARG when max_wait_rounds < 4096 (the drain waits share the
 * cap) and SSD_ERR_UNSUPPORTED for problems the tensor-core kernel does not
 * run (the SIMT kernel has no device waits).  Not for production use. */
SSD_API int ssd_fwd_fault_inject(const ssd_params_t* p,
            const void* x, const float* dt, const float* A,
            const void* B, const void* C, const float* D,
            const float* initial_states, const int32_t* cu_seqlens,
            void* y, float* final_states,
            void* workspace, size_t workspace_bytes, uint32_t max_wait_rounds, void* stream);

/* Human-readable name of a status code (static storage). */
SSD_API const char* ssd_status_string(int status);

/* Which kernel family ssd_fwd() uses for these params:
 * 0 = SIMT fp32 kernel, 1 = tcgen05 tensor-core kernel; -1 on invalid params.
 * *launches (if not NULL) receives the number of kernel launches per call. */
SSD_API int ssd_fwd_plan(const ssd_params_t* p, int has_initial_states, int has_final_states,
                 int* launches, int* nsplits);

/* The hierarchy-aware segsum device routines on their own (test aid).  Both
 * forms of csrc/segsum.cuh run here with the inputs the forward kernels give
 * them: the log-domain form, whose seg the SIMT kernel exponentiates, and the
 * linear-domain form, whose factors the tensor-core kernel multiplies in.
 * log2decay: (nrows, chunk) fp32 log2-domain log-decays (<= 0, may be -inf),
 * chunk 64 or 128.  Per row (each output may be NULL):
 *   seg_out  (chunk x chunk) seg[i][j] = sum_{k=j+1..i} log2decay[k] for j <= i,
 *            as the log-domain routine forms it (no prefix subtraction),
 *            -inf above the diagonal;
 *   L_out    (chunk x chunk) the decay mask prod_{k=j+1..i} a_k of the
 *            linear-domain routine, with a_k = ex2.approx(log2decay[k]) (the
 *            tensor-core kernel's factors): products grown from the diagonal
 *            on the 32 x 32 diagonal blocks, the rank-one product of the row
 *            factor and the column factor on the blocks left of them, 0 above
 *            the diagonal;
 *   pexp_out (chunk) the row prefixes prod_{k=0..i} a_k (decay of the state
 *            entering the chunk, at row i);
 *   sfx_out  (chunk) the column suffixes prod_{k=j+1..chunk-1} a_k (decay of
 *            token j's contribution to the state leaving the chunk).
 * Device pointers; async on `stream`.  Returns SSD_ERR_INVALID_ARG for a NULL
 * input or an unsupported chunk, SSD_ERR_CUDA for a failed launch.
 * Source: "GPU Hierarchy Meets Structured Matrices" (abstract): the 1-SS mask
 * as 1-SS diagonal blocks plus rank-one off-diagonal blocks. */
SSD_API int ssd_segsum_dump(const float* log2decay, int64_t nrows, int32_t chunk,
                    float* seg_out, float* L_out, float* pexp_out, float* sfx_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SSD_H_ */
