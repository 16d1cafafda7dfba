// Shared definitions of the libssd CUDA sources (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/ssd.h"

namespace ssd {

// Workspace layout: [0, 256) status header, then the split buffers.
struct WsHeader {
    uint32_t status;       // first device error recorded (0 = none)
    uint32_t where;        // kernel-specific code of the failing wait
    uint32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr float kLog2e = 1.4426950408889634f;

// Record a device-side error once (first writer wins).
__device__ __forceinline__ void record_error(WsHeader* ws, uint32_t code, uint32_t where) {
    if (ws && atomicCAS(&ws->status, 0u, code) == 0u) ws->where = where;
}

// where code of a failed packed-document offset check
constexpr uint32_t kWhereCuSeqlens = 40;

// Packed-document offsets must run 0 = cu[0] < cu[1] < ... < cu[ndocs] = L (no
// empty document).  The host cannot read them (device memory), so the last
// launch of a call checks them: threads t = 0 .. stride - 1 of one CTA each
// take every stride-th pair and record SSD_ERR_DEVICE_CHECK (where 40) on a
// violation.  Every kernel that reads cu_seqlens keeps its indexes in bounds
// whatever the offsets hold; the results are undefined when this check fails.
__device__ __forceinline__ void check_cu_seqlens(const int32_t* cu, int ndocs, int64_t L, WsHeader* ws, int t,
                                                 int stride) {
    bool bad = t == 0 && (__ldg(cu) != 0 || (int64_t)__ldg(cu + ndocs) != L);
    for (int k = t; k < ndocs; k += stride)
        if (__ldg(cu + k) >= __ldg(cu + k + 1)) bad = true;
    if (bad) record_error(ws, SSD_ERR_DEVICE_CHECK, kWhereCuSeqlens);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p) { return *p; }
    static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// Split plan shared by host and device: splits of `split_len` tokens over
// each batch row; unit u = ((b * H) + h) * nsplit + s.
struct SplitPlan {
    int64_t split_len;
    int32_t nsplit;
};

// Offsets (in bytes) of the split buffers inside the workspace.
struct WsLayout {
    size_t tau_off;     // float   [batch * H * nsplit]
    size_t state_off;   // float   [batch * H * nsplit * P * N]  aggregates, then incoming states (slot s - 1: split s)
    size_t total;
};

// Programmatic dependent launch.  A forward call's launches after its first are
// programmatic dependents of the one before: they may start on SMs the earlier
// kernel leaves free, and wait for its completion (and the visibility of its
// writes) only where they read its output.  Every kernel of the call triggers its
// dependent at its start; a dependent waits before its first read of earlier
// output, and also before it exits, so that its completion implies the
// completion of every earlier launch.  Without the launch attribute both are
// no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch kern<<<grid, block, smem, st>>>(args...), as a programmatic dependent of
// the previous launch on st when dep is set.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                                 bool dep, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = dep ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int64_t batch, int H, int P, int N, int nsplit) {
    WsLayout l;
    l.tau_off = sizeof(WsHeader);
    if (nsplit <= 1) {
        l.state_off = l.tau_off;
        l.total = sizeof(WsHeader);
        return l;
    }
    size_t units = (size_t)batch * H * nsplit;
    l.state_off = align_up(l.tau_off + units * sizeof(float), 256);
    l.total = align_up(l.state_off + units * (size_t)P * N * sizeof(float), 256);
    return l;
}

}  // namespace ssd
