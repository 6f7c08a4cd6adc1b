// x preparation for the tensor-core kernel: once per call, the M <= 16 rows of
// x are written per group of 64 inputs as one 2112-byte record:
//   bytes    0..2047  the 16 x 64 bf16 block (rows >= M zero) in the tensor
//                     core's K-major core-matrix layout, with the inputs of each
//                     8-block in the order the dequantized weights use
//                     (k0 k4 k1 k5 k2 k6 k3 k7);
//   bytes 2048..2111  X[m] = sum of the group's 64 inputs of row m (fp32), in a
//                     fixed order (8 sequential adds per 8-block, then the 8
//                     block sums in increasing k).
// Core matrix (kc, mg) of the block (8 inputs x 8 rows) sits at kc*256 + mg*128,
// row r of it at +16*r.
#pragma once

#include <cstdint>

namespace q4 {
namespace prep {

constexpr int kRecordBytes = 2112;
constexpr int kThreads = 128;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// One CTA per group of 64 inputs; thread t handles row m = t / 8, 8-block kc = t % 8.
__global__ void __launch_bounds__(kThreads) prep_x_kernel(const uint16_t* __restrict__ x, int M, int64_t K,
                                                          uint8_t* __restrict__ xt) {
    __shared__ float part[16][8];
    pdl_launch_dependents();
    // x may come from the kernel before this one, and an earlier call on the
    // stream may still read the scratch: wait for the preceding grid first
    pdl_wait();
    const int g = blockIdx.x;
    const int t = threadIdx.x;
    const int m = t >> 3, kc = t & 7;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (m < M) v = *reinterpret_cast<const uint4*>(x + (int64_t)m * K + (int64_t)g * 64 + kc * 8);
    // fixed-order partial sum of the 8 inputs (natural order)
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        s = __fadd_rn(s, __uint_as_float(w[i] << 16));
        s = __fadd_rn(s, __uint_as_float(w[i] & 0xFFFF0000u));
    }
    part[m][kc] = s;
    uint4 o;
    o.x = prmt(v.x, v.z, 0x5410u);     // (k0, k4)
    o.y = prmt(v.x, v.z, 0x7632u);     // (k1, k5)
    o.z = prmt(v.y, v.w, 0x5410u);     // (k2, k6)
    o.w = prmt(v.y, v.w, 0x7632u);     // (k3, k7)
    __syncthreads();
    uint8_t* rec = xt + (int64_t)g * kRecordBytes;
    *reinterpret_cast<uint4*>(rec + kc * 256 + (m >> 3) * 128 + (m & 7) * 16) = o;
    if (t < 16) {
        float X = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) X = __fadd_rn(X, part[t][j]);
        reinterpret_cast<float*>(rec + 2048)[t] = X;
    }
}

}  // namespace prep
}  // namespace q4

namespace q4 {
namespace prep {

// x preparation for the register-operand (mma.sync m16n8k16) kernel: per group
// of 64 inputs one 2112-byte record:
//   bytes    0..2047  the B fragments of the group's 4 k-steps for n8 tiles 0
//                     (rows 0-7) and 1 (rows 8-15): word ((kk*2 + t)*32 + lane)*2 + h
//                     of lane (gid, tig) holds rows m = 8t + gid, inputs
//                     16*tig + kk + 8h and 16*tig + kk + 8h + 4 -- the inputs
//                     the dequantized weight pairs of that lane pair with --
//                     scaled by 2^kFragScale (by 2^(kFragScale-4) for odd kk,
//                     whose weight pairs carry 2^-129 instead of 2^-133);
//   bytes 2048..2111  X[m] = sum of the group's 64 inputs of row m, unscaled,
//                     in a fixed order (8 sequential adds per 8-block, then
//                     the 8 block sums in increasing k).
// Rows >= M are zero.  The scale is a fixed power of two, so every value is
// exact (|x| < 2^27) and no row's record depends on another row.
constexpr int kFragScale = 100;

__global__ void __launch_bounds__(256) prep_x_frag_kernel(const uint16_t* __restrict__ x, int M, int64_t K,
                                                          uint8_t* __restrict__ xt) {
    __shared__ float xs[16][64];
    __shared__ float part[16][8];
    pdl_launch_dependents();
    pdl_wait();       // x may come from the preceding kernel; an earlier call may still read the scratch
    const int g = blockIdx.x;
    const int t = threadIdx.x;
    // 16 rows x 64 inputs: thread t loads 4 inputs of row t / 16
    {
        const int m = t >> 4, k4 = (t & 15) * 4;
        uint2 v = make_uint2(0, 0);
        if (m < M) v = *reinterpret_cast<const uint2*>(x + (int64_t)m * K + (int64_t)g * 64 + k4);
        xs[m][k4 + 0] = __uint_as_float(v.x << 16);
        xs[m][k4 + 1] = __uint_as_float(v.x & 0xFFFF0000u);
        xs[m][k4 + 2] = __uint_as_float(v.y << 16);
        xs[m][k4 + 3] = __uint_as_float(v.y & 0xFFFF0000u);
    }
    __syncthreads();
    uint8_t* rec = xt + (int64_t)g * kRecordBytes;
    // 512 fragment words, 2 per thread
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int wi = t * 2 + i;                    // word index
        const int h = wi & 1, lane = (wi >> 1) & 31, tt = (wi >> 6) & 1, kk = wi >> 7;
        const int gid = lane >> 2, tig = lane & 3;
        const int m = 8 * tt + gid;
        const int k_lo = 16 * tig + kk + 8 * h;
        const int sc = kFragScale - ((kk & 1) ? 4 : 0);
        const float lo = ldexpf(xs[m][k_lo], sc), hi = ldexpf(xs[m][k_lo + 4], sc);
        const uint32_t lo_b = __float_as_uint(lo) >> 16, hi_b = __float_as_uint(hi) >> 16;   // exact: 8-bit significands
        reinterpret_cast<uint32_t*>(rec)[wi] = lo_b | (hi_b << 16);
    }
    // fixed-order group sums
    if (t < 128) {
        const int m = t >> 3, kc = t & 7;
        float s = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) s = __fadd_rn(s, xs[m][kc * 8 + e]);
        part[m][kc] = s;
    }
    __syncthreads();
    if (t < 16) {
        float X = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) X = __fadd_rn(X, part[t][j]);
        reinterpret_cast<float*>(rec + 2048)[t] = X;
    }
}

}  // namespace prep
}  // namespace q4
