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
