// Single-token (decode) step of the SSD recurrence:
//   ssd_step_kernel     one token per (batch row, head) from a resident state
//
// "State Space Duality and Mamba-2", section "Performance and Serving
// Economics": during autoregressive generation the model keeps a fixed-size
// recurrent state and spends constant time and memory per generated token.
// One step is the selective-SSM recurrence of section "The Mathematical
// Bridge" (scalar-identity transition) taken once, per (b, h), g = h / (H / G):
//
//     a        = exp(dt A_h)
//     S'[p][n] = a S[p][n] + (dt x_p) B_n
//     y_p      = sum_n S'[p][n] C_n + D_h x_p
//
// The step reads and writes the P x N fp32 state once and touches little
// else, so it is bound by HBM bandwidth on the state: one CTA per (b, h)
// streams the state rows as float4 vectors (each row owned by a segment of
// SEG lanes, VPL vectors per lane), 16 / VPL rows in flight per segment (64
// state registers per thread: all 64 rows of a Mamba-2 head in one pass, so
// that small batches, whose CTAs are all resident at once, keep enough bytes
// in flight), and reduces y_p within the segment by shuffles.
#include "ssd_common.cuh"
#include "ssd_kernels.h"

namespace ssd {
namespace {

constexpr int kStepThreads = 128;

template <typename T, int SEG, int VPL>
__global__ void __launch_bounds__(kStepThreads) ssd_step_kernel(StepArgs a) {
    constexpr int kStepRows = 16 / VPL;   // rows each segment has in flight
    extern __shared__ float sm[];
    const int P = a.P, N = a.N, N4 = a.N >> 2;
    float* sB = sm;            // [N]  B_n
    float* sC = sB + N;        // [N]  C_n
    float* sx = sC + N;        // [P]  x_p
    float* sy = sx + P;        // [P]  sum_n S'[p][n] C_n
    const int tid = threadIdx.x;
    const int64_t bh = blockIdx.x;
    const int h = (int)(bh % a.H);
    const int64_t b = bh / a.H;
    const int g = h / (a.H / a.G);
    const T* xg = static_cast<const T*>(a.x) + bh * P;
    const T* Bg = static_cast<const T*>(a.B) + (b * a.G + g) * N;
    const T* Cg = static_cast<const T*>(a.C) + (b * a.G + g) * N;
    for (int n = tid; n < N; n += kStepThreads) {
        sB[n] = Elem<T>::load(Bg + n);
        sC[n] = Elem<T>::load(Cg + n);
    }
    for (int p = tid; p < P; p += kStepThreads) sx[p] = Elem<T>::load(xg + p);
    const float dtv = a.dt[bh];
    const float decay = expf(dtv * a.A[h]);
    __syncthreads();

    constexpr int kSegs = kStepThreads / SEG;   // rows a CTA pass covers
    const int li = tid % SEG;                   // lane within the row's segment
    const int rs = tid / SEG;                   // segment
    float4 bv[VPL], cv[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
        const int n4 = li + k * SEG;
        bv[k] = (n4 < N4) ? reinterpret_cast<const float4*>(sB)[n4] : make_float4(0.f, 0.f, 0.f, 0.f);
        cv[k] = (n4 < N4) ? reinterpret_cast<const float4*>(sC)[n4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float4* Sin = reinterpret_cast<const float4*>(a.state_in + bh * P * N);
    float4* Sout = reinterpret_cast<float4*>(a.state_out + bh * P * N);
    for (int p0 = 0; p0 < P; p0 += kSegs * kStepRows) {
        float4 s[kStepRows][VPL];
#pragma unroll
        for (int r = 0; r < kStepRows; ++r) {
            const int p = p0 + r * kSegs + rs;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int n4 = li + k * SEG;
                s[r][k] = (p < P && n4 < N4) ? __ldcs(Sin + (size_t)p * N4 + n4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int r = 0; r < kStepRows; ++r) {
            const int p = p0 + r * kSegs + rs;
            const float xd = (p < P) ? dtv * sx[p] : 0.f;
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int n4 = li + k * SEG;
                float4 v = s[r][k];
                v.x = fmaf(decay, v.x, xd * bv[k].x);
                v.y = fmaf(decay, v.y, xd * bv[k].y);
                v.z = fmaf(decay, v.z, xd * bv[k].z);
                v.w = fmaf(decay, v.w, xd * bv[k].w);
                acc = fmaf(v.x, cv[k].x, acc);
                acc = fmaf(v.y, cv[k].y, acc);
                acc = fmaf(v.z, cv[k].z, acc);
                acc = fmaf(v.w, cv[k].w, acc);
                if (p < P && n4 < N4) __stcs(Sout + (size_t)p * N4 + n4, v);
            }
#pragma unroll
            for (int o = SEG / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (li == 0 && p < P) sy[p] = acc;
        }
    }
    __syncthreads();
    const float Dh = a.D ? a.D[h] : 0.f;
    T* yg = static_cast<T*>(a.y) + bh * P;
    for (int p = tid; p < P; p += kStepThreads) Elem<T>::store(yg + p, fmaf(Dh, sx[p], sy[p]));
}

template <typename T, int SEG, int VPL>
cudaError_t launch_one(const StepArgs& a, size_t smem, cudaStream_t st) {
    ssd_step_kernel<T, SEG, VPL><<<(unsigned)(a.batch * a.H), kStepThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const StepArgs& a, size_t smem, cudaStream_t st) {
    const int N4 = a.N / 4;
    if (N4 > 64) return launch_one<T, 32, 4>(a, smem, st);
    if (N4 > 32) return launch_one<T, 32, 2>(a, smem, st);
    if (N4 > 16) return launch_one<T, 32, 1>(a, smem, st);
    if (N4 > 8) return launch_one<T, 16, 1>(a, smem, st);
    if (N4 > 4) return launch_one<T, 8, 1>(a, smem, st);
    return launch_one<T, 4, 1>(a, smem, st);
}

}  // namespace

size_t step_smem_bytes(int P, int N) { return (2 * (size_t)N + 2 * (size_t)P) * sizeof(float); }

cudaError_t launch_step(const StepArgs& a, cudaStream_t st) {
    const size_t smem = step_smem_bytes(a.P, a.N);
    return a.dtype == SSD_BF16 ? launch_typed<__nv_bfloat16>(a, smem, st) : launch_typed<float>(a, smem, st);
}

}  // namespace ssd
