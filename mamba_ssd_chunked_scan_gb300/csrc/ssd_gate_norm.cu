// Gated RMS normalisation of the scan's output, in one pass:
//   ssd_gate_norm_kernel   out = g / sqrt(mean_group(g^2) + eps) * w,
//                          g = y * silu(z) = y * z / (1 + exp(-z))
//
// "NVIDIA Accelerates Mamba-2 Forward Kernel with CUDA Tile", operator fusion:
// in the Mamba-2 forward pass the scan is followed by gating and normalisation,
// and fusing them keeps the gated values on chip instead of writing them out
// and reading them back.  The gate is the output gate of the Mamba-2 block
// (silu of the gate branch z) and the normalisation is a root-mean-square norm
// over groups of `group_size` consecutive channels with a per-channel weight.
//
// One CTA takes one (row, group) with just enough threads that each holds
// kNormVecs 16-byte vectors of y and z: every load is issued before any value
// is used (one HBM round trip per CTA), the gated values stay in registers
// while the sum of squares is reduced (warp shuffles, then the warps'
// partials in a fixed order), and each output vector is written once.
#include "ssd_common.cuh"
#include "ssd_kernels.h"

namespace ssd {
namespace {

constexpr int kNormVecs = 2;   // 16-byte vectors of y (and of z) per thread
// group_size <= 8192: at most 1024 bf16 or 2048 fp32 vectors, so at most
// 512 (bf16) or 1024 (fp32) threads
template <typename T>
constexpr int kNormMaxThreads = sizeof(T) == 2 ? 512 : 1024;
// CTAs per SM the bf16 kernel is compiled for: registers for 4 CTAs of 512
// threads keep enough rows' loads in flight (2 vectors per thread and more
// threads measured 84.6 us against 99.3 us for 4 vectors per thread at the
// 2.7B-like layer's output; the loads' latency, not issue, is the bound)
template <typename T>
constexpr int kNormMinBlocks = sizeof(T) == 2 ? 4 : 1;

// y silu(z) = y z / (1 + e^{-z}), with e^{-z} = 2^{-z log2 e} and the reciprocal
// taken by the special-function unit (ex2.approx, rcp.approx: relative errors of a
// few units in the last place, far inside the fp32 and bf16 tolerances).  The
// gate is issue-bound with an IEEE exp and divide per element.  Large negative z
// gives 1 / inf = 0 (the limit), large positive z gives 1.
__device__ __forceinline__ float silu_gate(float y, float z) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-z * 1.4426950408889634f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
    return y * z * r;
}

template <typename T>
struct Vec;   // 16 bytes of T
template <>
struct Vec<float> {
    static constexpr int n = 4;
    static __device__ __forceinline__ void load(const float* p, float* v) {
        const float4 q = *reinterpret_cast<const float4*>(p);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
    static __device__ __forceinline__ void store(float* p, const float* v) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int n = 8;
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* v) {
        const uint4 q = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* v) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            w[k] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <typename T>
__global__ void __launch_bounds__(kNormMaxThreads<T>, kNormMinBlocks<T>) ssd_gate_norm_kernel(GateNormArgs a) {
    __shared__ float part[kNormMaxThreads<T> / 32];
    constexpr int V = Vec<T>::n;
    const int gs = a.group_size, nvec = gs / V;
    const int ngroup = a.width / gs;
    const int64_t row = blockIdx.x / ngroup;
    const int grp = (int)(blockIdx.x - row * ngroup);
    const size_t base = (size_t)row * a.width + (size_t)grp * gs;
    const T* y = static_cast<const T*>(a.y) + base;
    const T* z = static_cast<const T*>(a.z) + base;
    const int nt = blockDim.x;
    uint4 yr[kNormVecs], zr[kNormVecs];
#pragma unroll
    for (int r = 0; r < kNormVecs; ++r) {
        const int k = threadIdx.x + r * nt;
        if (k < nvec) {
            yr[r] = __ldcs(reinterpret_cast<const uint4*>(y + k * V));
            zr[r] = __ldcs(reinterpret_cast<const uint4*>(z + k * V));
        }
    }
    float gv[kNormVecs][V];
    float ss = 0.f;
#pragma unroll
    for (int r = 0; r < kNormVecs; ++r) {
        const int k = threadIdx.x + r * nt;
        if (k < nvec) {
            float yv[V], zv[V];
            Vec<T>::load(reinterpret_cast<const T*>(&yr[r]), yv);
            Vec<T>::load(reinterpret_cast<const T*>(&zr[r]), zv);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                gv[r][e] = silu_gate(yv[e], zv[e]);
                ss = fmaf(gv[r][e], gv[r][e], ss);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < nt / 32; ++w) tot += part[w];
    const float rstd = rsqrtf(tot / (float)gs + a.eps);
    const float* wt = a.weight + (size_t)grp * gs;
    T* out = static_cast<T*>(a.out) + base;
#pragma unroll
    for (int r = 0; r < kNormVecs; ++r) {
        const int k = threadIdx.x + r * nt;
        if (k < nvec) {
            float wv[V];
#pragma unroll
            for (int e = 0; e < V; e += 4) {
                const float4 w4 = __ldg(reinterpret_cast<const float4*>(wt + k * V + e));
                wv[e] = w4.x; wv[e + 1] = w4.y; wv[e + 2] = w4.z; wv[e + 3] = w4.w;
            }
            float ov[V];
#pragma unroll
            for (int e = 0; e < V; ++e) ov[e] = gv[r][e] * rstd * wv[e];
            Vec<T>::store(out + k * V, ov);
        }
    }
}

}  // namespace

cudaError_t launch_gate_norm(const GateNormArgs& a, cudaStream_t st) {
    const int V = a.dtype == SSD_BF16 ? 8 : 4;
    const int nvec = a.group_size / V;
    // threads: enough warps that each thread holds at most kNormVecs vectors
    int threads = (nvec + kNormVecs - 1) / kNormVecs;
    threads = (threads + 31) / 32 * 32;
    if (threads > (a.dtype == SSD_BF16 ? kNormMaxThreads<__nv_bfloat16> : kNormMaxThreads<float>))
        return cudaErrorInvalidValue;
    const int64_t ctas = a.rows * (a.width / a.group_size);
    if (a.dtype == SSD_BF16)
        ssd_gate_norm_kernel<__nv_bfloat16><<<(unsigned)ctas, threads, 0, st>>>(a);
    else
        ssd_gate_norm_kernel<float><<<(unsigned)ctas, threads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ssd
