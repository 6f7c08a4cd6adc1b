// Generic Q4 verify-matmul kernel: any K that is a positive multiple of 64.
//
// y[m,n] = sum_k x[m,k] * (s[n,k/64] * q[n,k] + b[n,k/64])
//
// Each weight is dequantized once in fp32 (w = fma(s, q, b): the product s*q
// is exact, one rounding for the add) and then multiplied into every verify
// row with fp32 FMAs.  Error: at most about (K/32 + 6) * 2^-24 * sum|x*w| per
// output, far inside the 2e-3 relative tolerance, and w == 0 gives exactly 0.
//
// Row invariance (row m independent of M): every row m has its own
// accumulators, its own fixed sequence of FMAs over k and a fixed butterfly
// reduction, whatever the template row count MT or the number of live rows.
//
// Work split: a CTA of 8 warps owns 16 consecutive output rows n, 2 per warp;
// lane l of a warp reads 16-byte nibble chunks l, l+32, ... of each row (32
// consecutive inputs per chunk), so a warp reads 512 contiguous bytes per row
// per step.  x is staged in shared memory in chunks of KC inputs.
#pragma once

#include <cstdint>

namespace q4 {
namespace generic {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;
constexpr int kKc = 2048;   // inputs of x per shared-memory chunk

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int MT>
__global__ void __launch_bounds__(kWarps * 32)
matmul_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ W, int M, int64_t N,
              int64_t K, float* __restrict__ y) {
    extern __shared__ uint4 xs_raw[];                 // [MT][kKc] bf16
    uint16_t* xs = reinterpret_cast<uint16_t*>(xs_raw);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t G = K / 64;
    const int64_t row_bytes = K / 2;
    const uint16_t* scales = reinterpret_cast<const uint16_t*>(W + N * row_bytes);
    const uint16_t* biases = scales + N * G;
    const int64_t n_base = (int64_t)blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;

    float acc[kRowsPerWarp][MT];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.0f;

    for (int64_t kc0 = 0; kc0 < K; kc0 += kKc) {
        const int kcl = (int)((K - kc0) < kKc ? (K - kc0) : kKc);   // multiple of 64
        __syncthreads();
        // stage x[:, kc0 : kc0 + kcl] (rows >= M read as zero), 16 bytes per thread-step
        const int units_per_row = kcl / 8;
        for (int u = threadIdx.x; u < MT * units_per_row; u += blockDim.x) {
            const int m = u / units_per_row;
            const int j = u - m * units_per_row;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (m < M) v = *reinterpret_cast<const uint4*>(x + (int64_t)m * K + kc0 + 8 * j);
            *reinterpret_cast<uint4*>(xs + m * kKc + 8 * j) = v;
        }
        __syncthreads();

        for (int c = lane; c < kcl / 32; c += 32) {
            const int64_t k = kc0 + 32 * c;
            const int64_t g = k >> 6;
            uint4 nv[kRowsPerWarp];
            float sv[kRowsPerWarp], bv[kRowsPerWarp];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int64_t n = n_base + r;
                if (n < N) {
                    nv[r] = ldg_stream(W + n * row_bytes + k / 2);
                    sv[r] = bf16_bits_to_f32(scales[n * G + g]);
                    bv[r] = bf16_bits_to_f32(biases[n * G + g]);
                } else {
                    nv[r] = make_uint4(0, 0, 0, 0);
                    sv[r] = 0.0f;
                    bv[r] = 0.0f;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float wt[kRowsPerWarp][8];
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r) {
                    const uint32_t word = j == 0 ? nv[r].x : j == 1 ? nv[r].y : j == 2 ? nv[r].z : nv[r].w;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        // exact small integer -> float via the 2^23 bias trick
                        const float q = __fsub_rn(__uint_as_float(0x4B000000u | ((word >> (4 * i)) & 0xFu)),
                                                  8388608.0f);
                        wt[r][i] = __fmaf_rn(sv[r], q, bv[r]);
                    }
                }
                const int kl = 32 * c + 8 * j;      // offset inside the staged chunk
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(xs + m * kKc + kl);
                    const float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                                         bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
                    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[r][m] = __fmaf_rn(xf[i], wt[r][i], acc[r][m]);
                }
            }
        }
    }

    // fixed butterfly reduction across the warp
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float v = acc[r][m];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
            acc[r][m] = v;
        }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int64_t n = n_base + r;
            if (n < N)
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m < M) y[(int64_t)m * N + n] = acc[r][m];
        }
    }
}

inline size_t smem_bytes(int MT) { return (size_t)MT * kKc * sizeof(uint16_t); }

}  // namespace generic
}  // namespace q4
