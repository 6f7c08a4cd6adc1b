// Inter-layer glue of the chained verify pass: y_j (fp32 [M, N_prev]) becomes
// x_{j+1} (bf16 [M, K]).
//
//   kind 1 (RMSNORM):        v_k = y[m, k]                       k < K <= N_prev
//   kind 2 (SWIGLU_RMSNORM): v_k = silu(y[m, k]) * y[m, K + k]   N_prev == 2K
//   x[m, k] = bf16_RNE( v_k / sqrt( (1/K) sum_j v_j^2 + eps ) ),  silu(a) = a / (1 + exp(-a))
//
// The pages' own between-layer operators (attention, Gated DeltaNet, gated
// norms) are not on the matmul path; this fixed, bounded stand-in keeps the
// values of a long chain of linears in range.
//
// Work split: S CTAs per row (at most 8), each writing the outputs of a
// contiguous slice of the row made of whole groups of 64 inputs, so a step's
// glue runs on up to 8*M SMs instead of M.  S and the slices depend on K and
// the kind only.  RMSNORM rows of at most 6144 inputs: S = 8 (fewer if K has
// fewer groups), and every CTA forms the whole row's sum of squares itself
// (thread t: 8-input blocks t, t + 288, t + 576), so no CTA waits for another.
// Otherwise S = slices(K), the S CTAs of a row form a cluster and each sums its
// own slice (the order below).
//
// Two outputs.  x mode writes x_next as bf16 [M, K].  Record mode (inside a
// chained pass, when the next matmul runs the tensor-memory kernel) writes the
// next matmul's x records instead -- the same bf16 values, permuted and scaled
// into the record layout, and the group sums X added in the order of the
// matmul's own record build -- so that matmul builds none and x_next is never
// stored.
//
// Arithmetic: the definition is evaluated as if in double, on the
// single-precision pipes.  The sum of squares is kept as an unevaluated pair of
// floats (each square split exactly by an fma, the pairs added with error-free
// two-sums), which carries about 48 significant bits.  Each thread takes 8-input
// blocks (t, t + 288, ... of the row, or of its slice in a cluster) and adds their
// squares in increasing k; the threads' sums go through a fixed tree over lanes
// and warps; in a cluster each CTA pushes its slice's sum into every CTA's
// shared memory (distributed shared memory) before one cluster barrier, and
// every CTA adds the slices' sums in rank order.  The scale
// 1/sqrt(ss/K + eps) is formed as a float pair (one Newton step from the float
// value; relative error below 3e-14).  y is read once per CTA: a thread's first
// blocks stay in registers for the outputs (all of a slice up to 4608 inputs,
// or of a row up to 6144).
//   RMSNORM: v is an exact float, so v * scale is formed as a normalised float
//   pair and rounded to bf16 from it (the dropped 16 bits of the high part, and
//   at an exact float midpoint the sign of the low part): the rounding of the
//   exact product, except within about 2^-48 of a bf16 midpoint.
//   SWIGLU: silu(a) * b is formed in fp32 (within 9 float ulps); the output is
//   rounded from its fp32 product with the scale unless that lies within 10
//   float ulps of a bf16 midpoint, where v is recomputed in float pairs from the
//   inputs kept in registers (e^-a by
//   range reduction with ln 2 split into three floats and a Taylor series, then
//   a pair division; about 1e-14) and rounded from the pair.  Its sum of squares
//   is over the fp32 values, so its scale is within about 5e-7 of an all-double
//   one (typically 1e-8).
// No double arithmetic.  Each row's result depends on that row and
// K alone.
// Programmatic dependent launch: the kernel lets the next kernel start at once
// and reads y only after the preceding kernel finished.  The cluster barrier is
// a hardware barrier among CTAs that are always co-scheduled.
#pragma once

#include <cstdint>
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "q4_pair.cuh"
#include "q4_tm.cuh"

namespace q4 {
namespace glue {

using namespace q4::pair;

constexpr int kThreads = 288;                 // 9 warps: a SWIGLU slice of 2176 inputs is one 8-input block per thread
constexpr int kMaxSlices = 8;                 // portable cluster size
constexpr int64_t kSliceMin = 1024;           // inputs per slice below which fewer slices are used
// An output computed in float is trusted unless its low 16 bits (the bits
// bf16 rounding drops) are within this many float ulps of the halfway point.
constexpr int kTieMarginSwiglu = 10;          // SWIGLU: the fp32 output is within 9 float ulps of exact
constexpr int kKeep = 2;                      // 8-input blocks per thread held in registers (slices <= 4608 inputs)

// RMSNORM rows of at most kRowMax inputs: every CTA of the row forms the row's sum
// of squares itself, kRowKeep 8-input blocks per thread (no cluster).
constexpr int kRowKeep = 3;
constexpr int64_t kRowMax = 6144;
static_assert(kRowMax <= (int64_t)kRowKeep * kThreads * 8, "a row of kRowMax inputs fits the threads' registers");

__host__ __device__ inline bool one_cta_rows(int kind, int64_t K) { return kind == 1 && K <= kRowMax; }

inline int slices(int64_t K) {
    int64_t s = (K + kSliceMin - 1) / kSliceMin;
    return (int)(s < 1 ? 1 : (s > kMaxSlices ? kMaxSlices : s));
}

// v_k as a float pair: y itself (RMSNORM, exact) or silu(a) * b = a * b / (1 + e^-a)
// (SWIGLU, relative error about 1e-14).  a > 60: e^-a does not change 1 + e^-a in
// 48 bits; a < -88: e^-a overflows a float and the value (below 1e-36 * |b|) is 0.
__device__ __forceinline__ fpair value_pair(float a, float b, int kind) {
    if (kind != 2) return {a, 0.0f};
    if (a < -88.0f) return {0.0f, 0.0f};
    const fpair d = a > 60.0f ? fpair{1.0f, 0.0f} : pair_add(exp_pair(-a), fpair{1.0f, 0.0f});
    return pair_mul_f(f_div_pair(a, d), b);
}

// bf16 bits of the pair hi + lo (|lo| <= half an ulp of hi) rounded to nearest
// even: by the high part's dropped 16 bits, and at an exact float midpoint by
// the sign of the low part.
__device__ __forceinline__ uint16_t round_pair_bf16(float hi, float lo) {
    const uint32_t b = __float_as_uint(hi);
    const uint32_t low = b & 0xFFFFu;
    const uint32_t h = b >> 16;
    bool up;
    if (low != 0x8000u) {
        up = low > 0x8000u;                           // |lo| cannot move the value across the midpoint
    } else if (lo != 0.0f) {
        up = (lo > 0.0f) == (hi > 0.0f);              // beyond the midpoint in magnitude
    } else {
        up = (h & 1u) != 0u;                          // an exact tie: to even
    }
    return (uint16_t)(h + (up ? 1u : 0u));
}


// One output x[m, k] as bf16 bits.  RMSNORM (v exact): v * scale as a
// normalised float pair, rounded from the pair.  SWIGLU: v * scale rounded in
// float, unless that lies within kTieMarginSwiglu float ulps of a bf16 rounding
// midpoint (the fp32 value is within 9 ulps of exact), where it is recomputed
// as a float pair from the inputs a and b and rounded from the pair.
__device__ __forceinline__ uint16_t output_bits(float v, float a, float b, int kind, float inv_f, float inv_lo) {
    if (kind != 2) {                                              // RMSNORM: the exact pair, no branch
        const float p = __fmul_rn(v, inv_f);
        const fpair w = fast_two_sum(p, __fadd_rn(__fmaf_rn(v, inv_f, -p), __fmul_rn(v, inv_lo)));
        return round_pair_bf16(w.hi, w.lo);
    }
    const float t = __fmul_rn(v, inv_f);
    const int low = (int)(__float_as_uint(t) & 0xFFFFu);
    if (abs(low - 0x8000) <= kTieMarginSwiglu) {
        const fpair w = pair_mul(value_pair(a, b, kind), fpair{inv_f, inv_lo});
        return round_pair_bf16(w.hi, w.lo);
    }
    const __nv_bfloat16 h = __float2bfloat16_rn(t);
    return *reinterpret_cast<const uint16_t*>(&h);
}

// (hi, lo) += (p, e) with an error-free two-sum of the high parts.
__device__ __forceinline__ void ff_add(float& hi, float& lo, float p, float e) {
    const float t = __fadd_rn(hi, p);
    const float z = __fsub_rn(t, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(t, z)), __fsub_rn(p, z));
    hi = t;
    lo = __fadd_rn(lo, __fadd_rn(err, e));
}

// grid (S, M), cluster (S, 1, 1): CTA (s, m) owns inputs [s*L, min(K, (s+1)*L)) of row m.
// The inputs of the 8 values v_k, k = kb .. kb+7 (kb a multiple of 8): a = y[k]
// and, for SWIGLU, b = y[K + k]; all loads issued together.
__device__ __forceinline__ void inputs8(const float* yr, int64_t K, int64_t kb, int kind, bool vec, float (&a)[8],
                                        float (&b)[8]) {
    if (vec) {
        const float4 a0 = __ldcg(reinterpret_cast<const float4*>(yr + kb));
        const float4 a1 = __ldcg(reinterpret_cast<const float4*>(yr + kb + 4));
        a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
        if (kind == 2) {
            const float4 b0 = __ldcg(reinterpret_cast<const float4*>(yr + K + kb));
            const float4 b1 = __ldcg(reinterpret_cast<const float4*>(yr + K + kb + 4));
            b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            a[e] = __ldcg(yr + kb + e);
            if (kind == 2) b[e] = __ldcg(yr + K + kb + e);
        }
    }
    if (kind != 2) {
#pragma unroll
        for (int e = 0; e < 8; ++e) b[e] = 0.0f;
    }
}

// v_k in fp32 (exact for RMSNORM).
__device__ __forceinline__ float value_f(float a, float b, int kind) {
    return kind == 2 ? a / (1.0f + expf(-a)) * b : a;
}

// The scale 1/sqrt(ss/K + eps) of a row from its sum of squares th + tl, as a
// float pair: one Newton step from the correctly rounded float reciprocal square
// root (relative error below 3e-14, checked on the CPU against 40-digit
// arithmetic).  eps_hi + eps_lo: eps as a float pair.
__device__ __forceinline__ fpair row_scale(float th, float tl, int64_t K, float eps_hi, float eps_lo) {
    fpair t = pair_div_f(fast_two_sum(th, tl), (float)K);
    t = pair_add(t, fpair{eps_hi, eps_lo});
    const float r0 = __fdiv_rn(1.0f, __fsqrt_rn(t.hi));
    const float q = __fmul_rn(r0, r0);
    const fpair tr = pair_mul(t, fpair{q, __fmaf_rn(r0, r0, -q)});   // t * r0^2, close to 1
    const fpair e = pair_add(fpair{1.0f, 0.0f}, fpair{-tr.hi, -tr.lo});
    return fast_two_sum(r0, __fmul_rn(__fmul_rn(0.5f, r0), __fadd_rn(e.hi, e.lo)));
}

// x: bf16 [M, K] (x mode) or nullptr; rec: the next matmul's records [K/64][rec_bytes(rec_w)] (record mode) or nullptr.
// grid (S, M); a cluster of the S CTAs of a row unless one_cta_rows(kind, K).
__global__ void __launch_bounds__(kThreads) glue_kernel(const float* __restrict__ y, int64_t n_prev, int64_t K,
                                                        int kind, float eps_hi, float eps_lo, uint16_t* __restrict__ x,
                                                        uint8_t* __restrict__ rec, int rec_w) {
    namespace cg = cooperative_groups;
    __shared__ float part_hi[kThreads / 32], part_lo[kThreads / 32];
    __shared__ float slice_sum[2];
    __shared__ float2 sums[kMaxSlices];             // cluster rows: every slice's sum, in rank order
    __shared__ float inv_s[2];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");     // y comes from the preceding kernel
    const int S = (int)gridDim.x;
    const int s = (int)blockIdx.x;
    const int m = (int)blockIdx.y;
    const int64_t L = (K / 64 + S - 1) / S * 64;     // whole groups
    const int64_t k0 = (int64_t)s * L;
    const int64_t k1 = (k0 + L < K) ? k0 + L : K;
    const float* yr = y + (int64_t)m * n_prev;
    const bool vec = (n_prev & 3) == 0;              // rows 16-byte aligned

    // The block of inputs kb .. kb+7 (of this CTA's slice when active): its 8 outputs
    // to x, or into the next matmul's records (uniform over the CTA: whole warps call it).
    const int rb = q4::tm::rec_bytes(rec_w), rb0 = q4::tm::rec_b(rec_w);
    // v: the 8 values (value_f of a and bv).
    auto emit = [&](int64_t kb, bool active, const float (&v)[8], const float (&a)[8], const float (&bv)[8],
                    float inv_f, float inv_lo) {
        uint32_t h[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (active) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                h[e] = output_bits(v[e], a[e], bv[e], kind, inv_f, inv_lo);
        }
        if (rec == nullptr) {
            if (active) {
                uint4 o;
                o.x = h[0] | (h[1] << 16);
                o.y = h[2] | (h[3] << 16);
                o.z = h[4] | (h[5] << 16);
                o.w = h[6] | (h[7] << 16);
                *reinterpret_cast<uint4*>(x + (int64_t)m * K + kb) = o;
            }
            return;
        }
        // record mode: the group sum X, the 8 values in increasing k, then the 8 blocks of the
        // group (8 consecutive lanes, all active or none: slices are whole groups) by a fixed xor tree
        float sx = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) sx = __fadd_rn(sx, __uint_as_float(h[e] << 16));
        sx = __fadd_rn(sx, __shfl_xor_sync(0xFFFFFFFFu, sx, 1));
        sx = __fadd_rn(sx, __shfl_xor_sync(0xFFFFFFFFu, sx, 2));
        sx = __fadd_rn(sx, __shfl_xor_sync(0xFFFFFFFFu, sx, 4));
        if (active) {
            const int64_t g = kb / 64;
            const int kc = (int)((kb / 8) & 7);
            uint8_t* r = rec + g * rb;
            uint4 o;                                  // pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7), scaled
            o.x = q4::tm::bf16x2_mul(h[0] | (h[4] << 16), q4::tm::kXScaleEven);
            o.y = q4::tm::bf16x2_mul(h[1] | (h[5] << 16), q4::tm::kXScaleOdd);
            o.z = q4::tm::bf16x2_mul(h[2] | (h[6] << 16), q4::tm::kXScaleEven);
            o.w = q4::tm::bf16x2_mul(h[3] | (h[7] << 16), q4::tm::kXScaleOdd);
            *reinterpret_cast<uint4*>(r + rb0 + (m >> 3) * 1024 + kc * 128 + (m & 7) * 16) = o;
            if (kc == 0) reinterpret_cast<float*>(r)[m] = sx;
        }
    };
    // The CTA's sum of the threads' (hi, lo): a fixed tree over the lanes, then the
    // warps in order (thread 0); every thread returns with __syncthreads behind it.
    auto cta_sum = [&](float hi, float lo) {
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
        if (threadIdx.x == 0) {
            float th = part_hi[0], tl = part_lo[0];
            for (int w = 1; w < kThreads / 32; ++w) ff_add(th, tl, part_hi[w], part_lo[w]);
            slice_sum[0] = th;
            slice_sum[1] = tl;
        }
        __syncthreads();
    };

    if (one_cta_rows(kind, K)) {
        // RMSNORM of at most kRowMax inputs: every CTA of the row sums the whole row
        // itself (thread t: blocks t, t + 288, t + 576 in increasing k, all in
        // registers), so no CTA waits for another; it then writes the outputs of its
        // slice's blocks among them.
        const int64_t nb = K / 8;
        float a[kRowKeep][8], zero[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) zero[e] = 0.0f;
#pragma unroll
        for (int j = 0; j < kRowKeep; ++j) {
            const int64_t b = threadIdx.x + (int64_t)j * kThreads;
            if (b < nb) inputs8(yr, K, 8 * b, kind, vec, a[j], zero);
        }
        float hi = 0.0f, lo = 0.0f;
#pragma unroll
        for (int j = 0; j < kRowKeep; ++j) {
            if ((int64_t)threadIdx.x + (int64_t)j * kThreads < nb) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float v = a[j][e];
                    const float p = __fmul_rn(v, v);
                    ff_add(hi, lo, p, __fmaf_rn(v, v, -p));
                }
            }
        }
        cta_sum(hi, lo);
        const fpair inv = row_scale(slice_sum[0], slice_sum[1], K, eps_hi, eps_lo);
#pragma unroll
        for (int j = 0; j < kRowKeep; ++j) {
            const int64_t b = threadIdx.x + (int64_t)j * kThreads;
            emit(8 * b, b < nb && 8 * b >= k0 && 8 * b < k1, a[j], a[j], zero, inv.hi, inv.lo);
        }
        return;
    }

    cg::cluster_group cluster = cg::this_cluster();
    const int64_t nblk = (k1 > k0 ? k1 - k0 : 0) / 8; // 8-input blocks of this slice; thread t takes t, t + 288, ...

    // 1. the slice's sum of squares: each thread's blocks in increasing k; the first kKeep
    //    blocks stay in registers for step 2 (all their loads in flight together)
    float keep_a[kKeep][8], keep_b[kKeep][8], keep_v[kKeep][8];
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int u = 0; u < kKeep; ++u) {
        const int64_t b = threadIdx.x + (int64_t)u * kThreads;
        if (b < nblk) inputs8(yr, K, k0 + 8 * b, kind, vec, keep_a[u], keep_b[u]);
    }
#pragma unroll
    for (int u = 0; u < kKeep; ++u) {
        if ((int64_t)threadIdx.x + (int64_t)u * kThreads < nblk) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float v = value_f(keep_a[u][e], keep_b[u][e], kind);
                keep_v[u][e] = v;                     // for the outputs
                const float p = __fmul_rn(v, v);
                ff_add(hi, lo, p, __fmaf_rn(v, v, -p));
            }
        }
    }
    for (int64_t b = threadIdx.x + (int64_t)kKeep * kThreads; b < nblk; b += kThreads) {
        float a[8], bb[8];
        inputs8(yr, K, k0 + 8 * b, kind, vec, a, bb);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float v = value_f(a[e], bb[e], kind);
            const float p = __fmul_rn(v, v);
            ff_add(hi, lo, p, __fmaf_rn(v, v, -p));
        }
    }
    // the slice's sum (the same tree as cta_sum), pushed by thread 0 into slot s of
    // every CTA's sums, so that after the cluster barrier each CTA reads its own
    // shared memory only (and may leave without waiting for the others)
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
    if (threadIdx.x == 0) {
        float th = part_hi[0], tl = part_lo[0];
        for (int w = 1; w < kThreads / 32; ++w) ff_add(th, tl, part_hi[w], part_lo[w]);
        for (int r = 0; r < S; ++r) cluster.map_shared_rank(sums, r)[s] = make_float2(th, tl);
    }
    cluster.sync();                                   // every CTA's sums hold every slice's sum
    if (threadIdx.x < 32) {
        // the slices' sums (lane r: slice r), added in rank order
        const int r = (int)threadIdx.x;
        const float2 o = r < S ? sums[r] : make_float2(0.0f, 0.0f);
        float th = 0.0f, tl = 0.0f;
        for (int j = 0; j < S; ++j)
            ff_add(th, tl, __shfl_sync(0xFFFFFFFFu, o.x, j), __shfl_sync(0xFFFFFFFFu, o.y, j));
        if (r == 0) {
            const fpair inv = row_scale(th, tl, K, eps_hi, eps_lo);
            inv_s[0] = inv.hi;
            inv_s[1] = inv.lo;
        }
    }
    __syncthreads();
    const float inv_f = inv_s[0];
    const float inv_lo = inv_s[1];

    // 2. the outputs, block by block
#pragma unroll
    for (int u = 0; u < kKeep; ++u)
        if ((int64_t)u * kThreads < nblk)
            emit(k0 + 8 * ((int64_t)u * kThreads + threadIdx.x), (int64_t)u * kThreads + threadIdx.x < nblk, keep_v[u],
                 keep_a[u], keep_b[u], inv_f, inv_lo);
    for (int64_t b0 = (int64_t)kKeep * kThreads; b0 < nblk; b0 += kThreads) {
        float a[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        float bv[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        if (b0 + threadIdx.x < nblk) inputs8(yr, K, k0 + 8 * (b0 + threadIdx.x), kind, vec, a, bv);
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = value_f(a[e], bv[e], kind);
        emit(k0 + 8 * (b0 + threadIdx.x), b0 + threadIdx.x < nblk, v, a, bv, inv_f, inv_lo);
    }
}

}  // namespace glue
}  // namespace q4
