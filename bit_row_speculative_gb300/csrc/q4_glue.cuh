// Inter-layer glue of the chained verify pass: y_j (fp32 [M, N_prev]) becomes
// x_{j+1} (bf16 [M, K]).
//
//   kind 1 (RMSNORM):        v_k = y[m, k]                       k < K <= N_prev
//   kind 2 (SWIGLU_RMSNORM): v_k = silu(y[m, k]) * y[m, K + k]   N_prev == 2K
//   x[m, k] = bf16_RNE( v_k / sqrt( (1/K) sum_j v_j^2 + eps ) ),  silu(a) = a / (1 + exp(-a))
//
// The pages' own between-layer operators (attention, Gated DeltaNet, gated
// norms) are not on the matmul path; this fixed, bounded stand-in keeps the
// values of a long chain of linears in range.  One CTA per row: the sum of
// squares is a fixed-order reduction in double (per-thread strided partials,
// then a tree over lanes and warps), so each row's result depends on that row
// alone, and the single rounding to bf16 is taken from a double value.
// Programmatic dependent launch: the kernel lets the next matmul start its
// weight stream at once and reads y only after the preceding kernel finished.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace q4 {
namespace glue {

constexpr int kThreads = 1024;

// v_k in double: exact for kind 1; for kind 2 only expf is single precision,
// so the one rounding to bf16 below almost always matches an all-double
// evaluation of the same definition.
__device__ __forceinline__ double glue_value(const float* yr, int64_t K, int64_t k, int kind) {
    const float a = yr[k];
    if (kind == 2) return (double)a / (1.0 + (double)expf(-a)) * (double)yr[K + k];
    return (double)a;
}

__global__ void __launch_bounds__(kThreads) glue_kernel(const float* __restrict__ y, int64_t n_prev, int64_t K,
                                                        int kind, double eps, uint16_t* __restrict__ x) {
    __shared__ double part[kThreads / 32];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");     // y comes from the preceding kernel
    const int m = blockIdx.x;
    const float* yr = y + (int64_t)m * n_prev;
    double ss = 0.0;
    for (int64_t k = threadIdx.x; k < K; k += kThreads) {
        const double v = glue_value(yr, K, k, kind);
        ss = fma(v, v, ss);
    }
    // fixed tree: lanes, then warps in order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        double t = part[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
        if (threadIdx.x == 0) part[0] = t;
    }
    __syncthreads();
    const double inv = 1.0 / sqrt(part[0] / (double)K + eps);
    uint16_t* xr = x + (int64_t)m * K;
    for (int64_t k = threadIdx.x; k < K; k += kThreads) {
        const __nv_bfloat16 h = __double2bfloat16(glue_value(yr, K, k, kind) * inv);   // round to nearest even
        xr[k] = *reinterpret_cast<const uint16_t*>(&h);
    }
}

}  // namespace glue
}  // namespace q4
