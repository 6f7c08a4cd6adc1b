// Inter-layer glue of the chained verify pass: y_j (fp32 [M, N_prev]) becomes
// x_{j+1} (bf16 [M, K]).
//
//   kind 1 (RMSNORM):        v_k = y[m, k]                       k < K <= N_prev
//   kind 2 (SWIGLU_RMSNORM): v_k = silu(y[m, k]) * y[m, K + k]   N_prev == 2K
//   x[m, k] = bf16_RNE( v_k / sqrt( (1/K) sum_j v_j^2 + eps ) ),  silu(a) = a / (1 + exp(-a))
//
// The pages' own between-layer operators (attention, Gated DeltaNet, gated
// norms) are not on the matmul path; this fixed, bounded stand-in keeps the
// values of a long chain of linears in range.  One CTA per row.
//
// Arithmetic: the definition is evaluated as if in double, at single-precision
// cost.  The sum of squares is kept as an unevaluated pair of floats (each
// square split exactly by an fma, the pairs added with error-free two-sums),
// which carries about 48 significant bits; its per-thread pairs are combined
// in a fixed tree, and the scale 1/sqrt(ss/K + eps) is formed in double.  Each
// output is first computed in float; only when that value lies within a few
// float ulps of a bf16 rounding boundary -- where float error could decide
// the rounding -- is the element recomputed entirely in double (exp included)
// and rounded from there.  Each row's result depends on that row alone.
// Programmatic dependent launch: the kernel lets the next kernel start at once
// and reads y only after the preceding kernel finished.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace q4 {
namespace glue {

constexpr int kThreads = 1024;
// An output computed in float is trusted unless its low 16 bits (the bits
// bf16 rounding drops) are within this many float ulps of the halfway point.
constexpr int kTieMargin = 16;

__device__ __forceinline__ float value_f(const float* yr, int64_t K, int64_t k, int kind) {
    const float a = yr[k];
    if (kind == 2) return a / (1.0f + expf(-a)) * yr[K + k];
    return a;
}

__device__ __forceinline__ double value_d(const float* yr, int64_t K, int64_t k, int kind) {
    const double a = (double)yr[k];
    if (kind == 2) return a / (1.0 + exp(-a)) * (double)yr[K + k];
    return a;
}

// (hi, lo) += (p, e) with an error-free two-sum of the high parts.
__device__ __forceinline__ void ff_add(float& hi, float& lo, float p, float e) {
    const float t = __fadd_rn(hi, p);
    const float z = __fsub_rn(t, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(t, z)), __fsub_rn(p, z));
    hi = t;
    lo = __fadd_rn(lo, __fadd_rn(err, e));
}

__global__ void __launch_bounds__(kThreads) glue_kernel(const float* __restrict__ y, int64_t n_prev, int64_t K,
                                                        int kind, double eps, uint16_t* __restrict__ x) {
    __shared__ float part_hi[kThreads / 32], part_lo[kThreads / 32];
    __shared__ double inv_s;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");     // y comes from the preceding kernel
    const int m = blockIdx.x;
    const float* yr = y + (int64_t)m * n_prev;
    float hi = 0.0f, lo = 0.0f;
    for (int64_t k = threadIdx.x; k < K; k += kThreads) {
        const float v = value_f(yr, K, k, kind);
        const float p = __fmul_rn(v, v);
        ff_add(hi, lo, p, __fmaf_rn(v, v, -p));
    }
    // fixed tree: lanes, then warps in order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(0xFFFFFFFFu, hi, o), ol = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
        ff_add(hi, lo, oh, ol);
    }
    if ((threadIdx.x & 31) == 0) {
        part_hi[threadIdx.x >> 5] = hi;
        part_lo[threadIdx.x >> 5] = lo;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        float th = part_hi[threadIdx.x], tl = part_lo[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float oh = __shfl_xor_sync(0xFFFFFFFFu, th, o), ol = __shfl_xor_sync(0xFFFFFFFFu, tl, o);
            ff_add(th, tl, oh, ol);
        }
        if (threadIdx.x == 0) inv_s = 1.0 / sqrt(((double)th + (double)tl) / (double)K + eps);
    }
    __syncthreads();
    const double inv = inv_s;
    const float inv_f = (float)inv;
    uint16_t* xr = x + (int64_t)m * K;
    for (int64_t k = threadIdx.x; k < K; k += kThreads) {
        const float t = __fmul_rn(value_f(yr, K, k, kind), inv_f);
        const int low = (int)(__float_as_uint(t) & 0xFFFFu);
        __nv_bfloat16 h;
        if (abs(low - 0x8000) <= kTieMargin)
            h = __double2bfloat16(value_d(yr, K, k, kind) * inv);    // near a tie: decide in double
        else
            h = __float2bfloat16_rn(t);
        xr[k] = *reinterpret_cast<const uint16_t*>(&h);
    }
}

}  // namespace glue
}  // namespace q4
