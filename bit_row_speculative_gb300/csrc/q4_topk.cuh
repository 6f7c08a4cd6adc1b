// Sampling epilogue of the LM head: per row of logits, the top_k (<= 32)
// entries by logit and their probabilities -- "temperature over its first
// top_k entries, truncated by top_p, renormalized" ("Splash engine" analysis,
// section "Exact, up to top-32").
//
// Order: logit descending, equal logits by lower index first, so the selected
// set and its order are unique.  Logits are compared through a monotone 32-bit
// key (sign-magnitude flipped; -0 counted as +0); NaN logits are outside the
// contract.
//
// Phase 1 (topk_slice_kernel, grid (S, M)): CTA (s, m) stages slice s of row m
// (at most kMaxSlice logits) in shared memory, finds its 32nd largest key by an
// exact 8-bit radix select (4 rounds of histograms, MSB first), and writes its
// top min(32, slice length) entries -- every key above that threshold, then
// the lowest-index keys equal to it -- as 64-bit candidates (key << 32 | ~index,
// so a larger candidate ranks first) in index order.  The global top 32 of a row
// is contained in the union of its slices' top 32.
// Phase 2 (topk_merge_kernel, grid M): sorts a row's S*32 candidates (bitonic,
// descending) and one thread forms the probabilities in double in rank order:
// p_j = exp((l_j - l_0)/T) / sum_i exp((l_i - l_0)/T) over the top_k, keeps the
// shortest prefix whose cumulative probability reaches top_p (all if
// top_p >= 1), renormalizes it, and stores fp32 probabilities and int32
// indices (-1 past top_k, probability 0 past the kept prefix).
// Both kernels use programmatic dependent launch and read the logits only
// after the preceding kernel finished.
#pragma once

#include <cstdint>

namespace q4 {
namespace topk {

constexpr int kWidth = 32;                 // candidates per slice and output entries per row
constexpr int kMaxSlice = 16384;           // logits per slice (64 KB of keys in shared memory)
constexpr int kMaxSlices = 64;             // slices per row (N <= kMaxSlice * kMaxSlices)
constexpr int kSliceThreads = 512;
constexpr int kMergeThreads = 256;
constexpr int kSliceWarps = kSliceThreads / 32;

__device__ __forceinline__ uint32_t monotone_key(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

inline size_t slice_smem_bytes() {
    return (size_t)kMaxSlice * 4 + (size_t)kSliceWarps * 256 * 4 + 256 * 4 + 2 * kSliceThreads * 4 + 64;
}

// cand: [M][S][32] 64-bit candidates (0 = empty).
__global__ void __launch_bounds__(kSliceThreads) topk_slice_kernel(const float* __restrict__ logits, int64_t N,
                                                                   int64_t L, uint64_t* __restrict__ cand) {
    extern __shared__ uint32_t sm[];
    uint32_t* keys = sm;                                     // [kMaxSlice]
    uint32_t* whist = keys + kMaxSlice;                      // [warps][256]
    uint32_t* hist = whist + kSliceWarps * 256;              // [256]
    uint32_t* cnt_gt = hist + 256;                           // [threads]
    uint32_t* cnt_eq = cnt_gt + kSliceThreads;               // [threads]
    __shared__ uint32_t sel_prefix, sel_need;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");      // the logits come from the preceding kernel
    const int s = (int)blockIdx.x, m = (int)blockIdx.y;
    const int S = (int)gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t base = (int64_t)s * L;
    const int len = (int)((base + L <= N) ? L : (N - base));
    const float* row = logits + (int64_t)m * N + base;
    for (int i = tid; i < len; i += kSliceThreads) keys[i] = monotone_key(row[i]);
    const int k = len < kWidth ? len : kWidth;

    // radix select of the k-th largest key, most significant digit first
    uint32_t prefix = 0, mask = 0, need = (uint32_t)k;
    for (int d = 3; d >= 0; --d) {
        uint32_t* wh = whist + warp * 256;
        for (int b = lane; b < 256; b += 32) wh[b] = 0;
        __syncthreads();                                     // keys staged, histograms cleared
        const int sh = 8 * d;
        for (int i = tid; i < len; i += kSliceThreads) {
            const uint32_t key = keys[i];
            if ((key & mask) == prefix) atomicAdd(&wh[(key >> sh) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t h = 0;
            for (int w = 0; w < kSliceWarps; ++w) h += whist[w * 256 + tid];
            hist[tid] = h;
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t cum = 0, nd = need;
            int b = 255;
            for (; b > 0; --b) {
                if (cum + hist[b] >= nd) break;
                cum += hist[b];
            }
            sel_prefix = prefix | ((uint32_t)b << sh);
            sel_need = nd - cum;                             // how many keys equal to the prefix so far are needed
        }
        __syncthreads();
        prefix = sel_prefix;
        need = sel_need;
        mask |= 255u << sh;
    }
    // prefix is now the k-th largest key; keys above it all enter, then the
    // `need` lowest-index keys equal to it.  Each thread takes a contiguous chunk.
    const int chunk = (len + kSliceThreads - 1) / kSliceThreads;
    const int i0 = tid * chunk, i1 = (i0 + chunk < len) ? i0 + chunk : len;
    uint32_t ngt = 0, neq = 0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t key = keys[i];
        ngt += key > prefix;
        neq += key == prefix;
    }
    cnt_gt[tid] = ngt;
    cnt_eq[tid] = neq;
    __syncthreads();
    if (tid == 0) {                                          // exclusive scans in thread order
        uint32_t a = 0, b = 0;
        for (int t = 0; t < kSliceThreads; ++t) {
            const uint32_t x = cnt_gt[t], y = cnt_eq[t];
            cnt_gt[t] = a;
            cnt_eq[t] = b;
            a += x;
            b += y;
        }
    }
    __syncthreads();
    uint64_t* out = cand + ((int64_t)m * S + s) * kWidth;
    const uint32_t n_gt = (uint32_t)k - need;                // keys strictly above the threshold
    uint32_t pg = cnt_gt[tid], pe = cnt_eq[tid];
    for (int i = i0; i < i1; ++i) {
        const uint32_t key = keys[i];
        const uint64_t c = ((uint64_t)key << 32) | (uint64_t)(~(uint32_t)(base + i));
        if (key > prefix) {
            out[pg++] = c;
        } else if (key == prefix) {
            if (pe < need) out[n_gt + pe] = c;
            ++pe;
        }
    }
    for (int j = k + tid; j < kWidth; j += kSliceThreads) out[j] = 0ull;
}

// idx, probs: [M][32].
__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(const uint64_t* __restrict__ cand, int S, int top_k,
                                                                   float temperature, float top_p,
                                                                   int32_t* __restrict__ idx,
                                                                   float* __restrict__ probs) {
    __shared__ uint64_t c[kMaxSlices * kWidth];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");      // candidates come from the slice kernel
    const int m = (int)blockIdx.x;
    const int n = S * kWidth;
    int P = 1;
    while (P < n) P <<= 1;                                   // padded to a power of two with empty (0) entries
    for (int i = threadIdx.x; i < P; i += kMergeThreads) c[i] = i < n ? cand[(int64_t)m * n + i] : 0ull;
    __syncthreads();
    // bitonic sort, descending
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < P; i += kMergeThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const uint64_t a = c[i], b = c[j];
                    if (desc ? (a < b) : (a > b)) {
                        c[i] = b;
                        c[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    if (threadIdx.x == 0) {
        double e[kWidth];
        const double l0 = (double)key_value((uint32_t)(c[0] >> 32));
        const double t = (double)temperature;
        double total = 0.0;
        for (int j = 0; j < top_k; ++j) {
            e[j] = exp(((double)key_value((uint32_t)(c[j] >> 32)) - l0) / t);
            total += e[j];
        }
        for (int j = 0; j < top_k; ++j) e[j] = e[j] / total;
        int keep = top_k;
        if (top_p < 1.0f) {
            double cum = 0.0;
            for (int j = 0; j < top_k; ++j) {
                cum += e[j];
                if (cum >= (double)top_p) {
                    keep = j + 1;
                    break;
                }
            }
        }
        double kept = 0.0;
        for (int j = 0; j < keep; ++j) kept += e[j];
        for (int j = 0; j < kWidth; ++j) {
            idx[m * kWidth + j] = j < top_k ? (int32_t)(~(uint32_t)(c[j] & 0xFFFFFFFFull)) : -1;
            probs[m * kWidth + j] = j < keep ? (float)(e[j] / kept) : 0.0f;
        }
    }
}

}  // namespace topk
}  // namespace q4
