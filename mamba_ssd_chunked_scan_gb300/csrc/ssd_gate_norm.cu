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
// One CTA takes one (row, group): it reads y and z once as 16-byte vectors,
// keeps g in shared memory while the sum of squares is reduced (warp shuffles,
// then the warps' partials in a fixed order), and writes out once.
#include "ssd_common.cuh"
#include "ssd_kernels.h"

namespace ssd {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormVecs = 4;   // 16-byte vectors per thread loaded before any is used

__device__ __forceinline__ float silu_gate(float y, float z) { return y * (z / (1.f + expf(-z))); }

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
__global__ void __launch_bounds__(kNormThreads) ssd_gate_norm_kernel(GateNormArgs a) {
    extern __shared__ __align__(16) float g[];   // [group_size] gated values
    __shared__ float part[kNormThreads / 32];
    constexpr int V = Vec<T>::n;
    const int gs = a.group_size, nvec = gs / V;
    const int ngroup = a.width / gs;
    const int64_t row = blockIdx.x / ngroup;
    const int grp = (int)(blockIdx.x - row * ngroup);
    const size_t base = (size_t)row * a.width + (size_t)grp * gs;
    const T* y = static_cast<const T*>(a.y) + base;
    const T* z = static_cast<const T*>(a.z) + base;
    float ss = 0.f;
    auto gate = [&](int k, const uint4& yr, const uint4& zr) {
        float yv[V], zv[V];
        Vec<T>::load(reinterpret_cast<const T*>(&yr), yv);
        Vec<T>::load(reinterpret_cast<const T*>(&zr), zv);
#pragma unroll
        for (int e = 0; e < V; ++e) {
            const float gv = silu_gate(yv[e], zv[e]);
            g[k * V + e] = gv;
            ss = fmaf(gv, gv, ss);
        }
    };
    if (nvec <= kNormVecs * kNormThreads) {
        // all of this thread's vectors in flight at once: one HBM round trip
        uint4 yr[kNormVecs], zr[kNormVecs];
#pragma unroll
        for (int r = 0; r < kNormVecs; ++r) {
            const int k = threadIdx.x + r * kNormThreads;
            if (k < nvec) {
                yr[r] = *reinterpret_cast<const uint4*>(y + k * V);
                zr[r] = *reinterpret_cast<const uint4*>(z + k * V);
            }
        }
#pragma unroll
        for (int r = 0; r < kNormVecs; ++r) {
            const int k = threadIdx.x + r * kNormThreads;
            if (k < nvec) gate(k, yr[r], zr[r]);
        }
    } else {
        for (int k = threadIdx.x; k < nvec; k += kNormThreads)
            gate(k, *reinterpret_cast<const uint4*>(y + k * V), *reinterpret_cast<const uint4*>(z + k * V));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += part[w];
    const float rstd = rsqrtf(tot / (float)gs + a.eps);
    const float* wt = a.weight + (size_t)grp * gs;
    T* out = static_cast<T*>(a.out) + base;
    for (int k = threadIdx.x; k < nvec; k += kNormThreads) {
        float ov[V];
#pragma unroll
        for (int e = 0; e < V; ++e) ov[e] = g[k * V + e] * rstd * wt[k * V + e];
        Vec<T>::store(out + k * V, ov);
    }
}

}  // namespace

cudaError_t launch_gate_norm(const GateNormArgs& a, cudaStream_t st) {
    const size_t smem = (size_t)a.group_size * sizeof(float);
    const int64_t ctas = a.rows * (a.width / a.group_size);
    if (a.dtype == SSD_BF16)
        ssd_gate_norm_kernel<__nv_bfloat16><<<(unsigned)ctas, kNormThreads, smem, st>>>(a);
    else
        ssd_gate_norm_kernel<float><<<(unsigned)ctas, kNormThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ssd
