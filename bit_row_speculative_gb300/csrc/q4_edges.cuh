// Edge scores of the draft selector ("Splash engine" analysis, section "The
// draft is a small model with an unusual selector"): for each row r (one draft
// position of one lane), each of its 16 predecessor tokens i and each of its 16
// candidate tokens j,
//
//   context[d]     = pred_cb[pred_ids[r][i]][d] * hidden[r][d]
//   score[r][i][j] = sum over d < R of context[d] * succ_cb[cand_ids[r][j]][d]
//
// a trilinear form over a rank-R embedding of the previous token, a rank-R
// projection of the position's hidden state and a rank-R embedding of the
// candidate (R = 256 on the pages; the codebooks are bf16, vocabulary x R).
//
// One CTA per row, 256 threads, one score per thread.  The 32 codebook rows a
// row needs (16 predecessor, 16 candidate rows of 2R bytes each) are gathered
// with 16-byte loads, each warp reading whole rows, all of a thread's loads in
// flight together (the hidden values even before the ids arrive), into shared
// memory as fp32:
// context rows (the predecessor row times hidden, rounded once) and candidate
// rows.  Thread (i, j) then forms its dot product over d with four fp32
// accumulators (d mod 4), fused multiply-adds in increasing d, combined as
// (a0 + a1) + (a2 + a3): a fixed order, so a row's scores depend on that row's
// inputs alone.  Rows are padded to R + 4 floats so that the 16-byte shared
// loads of the dot loop are conflict-free.
//
// An id outside 0..V-1 is not read: the row of the codebook it names counts as
// zeros and the kernel sets a bit in the library's device error word, which the
// next status query reports.
// Programmatic dependent launch: ids and hidden come from the preceding kernel.
#pragma once

#include <cstdint>

namespace q4 {
namespace edges {

constexpr int kPairs = 16;                    // predecessors and candidates per row
constexpr int kThreads = kPairs * kPairs;     // one score per thread
constexpr int kMaxRank = 256;
constexpr int kMaxEdgeRows = 1 << 20;
constexpr int kStride = kMaxRank + 4;         // floats per shared row
constexpr unsigned int kErrBadIndex = 0x40000000u;
constexpr int kIter = 2 * kPairs * (kMaxRank / 8) / kThreads;   // gathered 16-byte chunks per thread, at most

__device__ __forceinline__ void widen8(const uint4& w, float (&v)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        v[2 * e] = __uint_as_float(u[e] << 16);              // lower address: element 2e
        v[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
    }
}

// grid: rows; hidden [rows][R] fp32; ids [rows][16]; score [rows][16][16].
__global__ void __launch_bounds__(kThreads) edges_kernel(const uint16_t* __restrict__ pred_cb,
                                                         const uint16_t* __restrict__ succ_cb, int64_t V, int R,
                                                         const float* __restrict__ hidden,
                                                         const int32_t* __restrict__ pred_ids,
                                                         const int32_t* __restrict__ cand_ids,
                                                         float* __restrict__ score, unsigned int* error_word) {
    __shared__ __align__(16) float ctx[kPairs][kStride];    // context rows
    __shared__ __align__(16) float suc[kPairs][kStride];    // candidate rows
    __shared__ int64_t row_of[2 * kPairs];                  // codebook row, -1 when out of range
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");     // ids and hidden come from the preceding kernel
    const int r = (int)blockIdx.x;
    const int tid = threadIdx.x;
    // chunk q = tid + it * 256 is chunk c of gathered row k (rows 0..15: predecessors, 16..31: candidates)
    const int cpr = R / 8;
    const int total = 2 * kPairs * cpr;
    const float4* h4 = reinterpret_cast<const float4*>(hidden + (int64_t)r * R);
    int32_t id = 0;
    if (tid < 2 * kPairs)
        id = tid < kPairs ? pred_ids[(int64_t)r * kPairs + tid] : cand_ids[(int64_t)r * kPairs + (tid - kPairs)];
    // the hidden values of this thread's context chunks do not depend on the ids: in flight meanwhile
    float4 h0[kIter], h1[kIter];
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const int q = tid + it * kThreads;
        const int k = q / cpr, c = q - k * cpr;
        h0[it] = h1[it] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (q < total && k < kPairs) {
            h0[it] = __ldg(h4 + 2 * c);
            h1[it] = __ldg(h4 + 2 * c + 1);
        }
    }
    if (tid < 2 * kPairs) {
        const bool ok = id >= 0 && (int64_t)id < V;
        if (!ok) atomicOr(error_word, kErrBadIndex);
        row_of[tid] = ok ? (int64_t)id : -1;
    }
    __syncthreads();

    // gather: every row load of the thread issued before any is used
    uint4 w[kIter];
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const int q = tid + it * kThreads;
        const int k = q / cpr, c = q - k * cpr;
        w[it] = make_uint4(0u, 0u, 0u, 0u);
        if (q < total) {
            const int64_t row = row_of[k];
            if (row >= 0) w[it] = __ldg(reinterpret_cast<const uint4*>((k < kPairs ? pred_cb : succ_cb) + row * R) + c);
        }
    }
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const int q = tid + it * kThreads;
        const int k = q / cpr, c = q - k * cpr;
        if (q < total) {
            float v[8];
            widen8(w[it], v);
            if (k < kPairs) {
                float4* dst = reinterpret_cast<float4*>(&ctx[k][8 * c]);
                dst[0] = make_float4(__fmul_rn(v[0], h0[it].x), __fmul_rn(v[1], h0[it].y), __fmul_rn(v[2], h0[it].z),
                                     __fmul_rn(v[3], h0[it].w));
                dst[1] = make_float4(__fmul_rn(v[4], h1[it].x), __fmul_rn(v[5], h1[it].y), __fmul_rn(v[6], h1[it].z),
                                     __fmul_rn(v[7], h1[it].w));
            } else {
                float4* dst = reinterpret_cast<float4*>(&suc[k - kPairs][8 * c]);
                dst[0] = make_float4(v[0], v[1], v[2], v[3]);
                dst[1] = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
    }
    __syncthreads();

    const int i = tid >> 4, j = tid & 15;
    const float4* a = reinterpret_cast<const float4*>(&ctx[i][0]);
    const float4* b = reinterpret_cast<const float4*>(&suc[j][0]);
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    for (int d4 = 0; d4 < R / 4; ++d4) {
        const float4 x = a[d4], y = b[d4];
        a0 = __fmaf_rn(x.x, y.x, a0);
        a1 = __fmaf_rn(x.y, y.y, a1);
        a2 = __fmaf_rn(x.z, y.z, a2);
        a3 = __fmaf_rn(x.w, y.w, a3);
    }
    score[(int64_t)r * kThreads + tid] = __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3));
}

}  // namespace edges
}  // namespace q4
