// Sampling epilogue of the LM head: per row of logits, the top_k (<= 32)
// entries by logit and their probabilities -- "temperature over its first
// top_k entries, truncated by top_p, renormalized" ("Splash engine" analysis,
// section "Exact, up to top-32").
//
// Order: logit descending, equal logits by lower index first, so the selected
// set and its order are unique.  Each logit becomes a 64-bit candidate
// (monotone 32-bit key of the float << 32 | ~index): a larger candidate ranks
// first, and no two candidates are equal.  -0 counts as +0; NaN logits are
// outside the contract.
//
// One kernel, grid (S, M), S = ceil(N / 8192) slices per row:
//  1. CTA (s, m) reads slice s of row m, 32 logits per thread (thread t owns
//     runs of 4 consecutive logits starting at 4t, 4t + 1024, ...), and each
//     thread keeps the largest of its candidates.
//  2. A lower bound for the slice's 32nd candidate: the 32nd largest of the 256
//     per-thread maxima (warp sorts, then merges).  Those 32 maxima are distinct
//     candidates at or above the bound, so the slice's top 32 are all at or
//     above it; and only the 32 threads whose maximum reaches the bound can hold
//     such candidates, so at most 32 * 32 = 1024 pass -- the candidate buffer
//     never overflows, whatever the data.  The slice is read a second time
//     (from L1) to collect them.
//  3. The passing candidates are sorted in chunks of 32 by the warps (bitonic
//     networks on shuffles), the chunks' top 32 merged, and the slice's top 32
//     written to scratch.
//  4. The last CTA of the row to finish (an acq_rel ticket) merges the S sorted
//     lists, each warp a share of them and then a tree over the warps (the top 32 of the union of two sorted lists is the elementwise
//     maximum of one list and the other reversed, merged bitonically), and one
//     warp forms the probabilities in float pairs (about 48 bits, rounding like
//     double ones; an exponential below e^-60 in double):
//     p_j = exp((l_j - l_0)/T) / sum_i exp((l_i - l_0)/T) over the top_k, the
//     shortest prefix whose cumulative probability reaches top_p kept (all if
//     top_p >= 1), renormalized; fp32 probabilities and int32 indices out
//     (-1 past top_k, probability 0 past the kept prefix).
// The kernel uses programmatic dependent launch and reads the logits only after
// the preceding kernel finished.  No thread waits on another CTA.
#pragma once

#include <cstdint>

#include "q4_pair.cuh"

namespace q4 {
namespace topk {

constexpr int kWidth = 32;                    // candidates per slice and output entries per row
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 32;                      // logits per thread
constexpr int kRuns = kPer / 4;               // runs of 4 consecutive logits per thread
constexpr int kSlice = kThreads * kPer;       // logits per CTA
constexpr int kMaxSlices = 128;               // N <= kSlice * kMaxSlices
constexpr int kCap = 32 * kPer;               // most candidates that can reach the bound
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t monotone_key(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t candidate(uint32_t key, int64_t index) {
    return ((uint64_t)key << 32) | (uint64_t)(~(uint32_t)index);
}

__device__ __forceinline__ uint64_t umax(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t umin(uint64_t a, uint64_t b) { return a < b ? a : b; }

// One value per lane; returns the warp's values sorted descending by lane.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint64_t o = __shfl_xor_sync(kFull, v, stride);
            const bool lower = (lane & stride) == 0;
            const bool desc = (lane & size) == 0;   // the block's direction; size 32 is all descending
            v = (lower == desc) ? umax(v, o) : umin(v, o);
        }
    }
    return v;
}

// A bitonic sequence across the warp, sorted descending.
__device__ __forceinline__ uint64_t warp_merge_desc(uint64_t v, int lane) {
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const uint64_t o = __shfl_xor_sync(kFull, v, stride);
        v = (lane & stride) == 0 ? umax(v, o) : umin(v, o);
    }
    return v;
}

// Logits i .. i+3 of a slice (those past len are not read).
__device__ __forceinline__ void load_run(const float* row, int i, int len, bool vec, float (&v)[4]) {
    if (vec) {
        if (i < len) {
            const float4 q = *reinterpret_cast<const float4*>(row + i);
            v[0] = q.x;
            v[1] = q.y;
            v[2] = q.z;
            v[3] = q.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (i + e < len) v[e] = row[i + e];
    }
}

// lists[w] (w < kWarps), each sorted descending: the top 32 of their union, by
// a tree of merges (kWarps/2, then kWarps/4, ... warps at a time).  Called by
// every thread of the CTA; every thread gets lists[0][lane] of the result.
__device__ __forceinline__ uint64_t tree_merge(uint64_t (&lists)[kWarps][32], int warp, int lane) {
#pragma unroll
    for (int half = kWarps / 2; half >= 1; half >>= 1) {
        uint64_t v = 0;
        if (warp < half) v = warp_merge_desc(umax(lists[warp][lane], lists[warp + half][31 - lane]), lane);
        __syncthreads();                                      // every list of this level has been read
        if (warp < half) lists[warp][lane] = v;
        __syncthreads();
    }
    return lists[0][lane];
}

// cand: [M][S][32] scratch; tickets: [M] counters, zero between launches.
// idx, probs: [M][32].
// discard != 0 (logits in the library's own scratch): once the slice is read,
// its whole 128-byte L2 lines are invalidated without being written back.
__global__ void __launch_bounds__(kThreads, 4) topk_kernel(const float* __restrict__ logits, int64_t N, int64_t L,
                                                        int top_k, float temperature, float top_p,
                                                        uint64_t* __restrict__ cand, int* __restrict__ tickets,
                                                        int32_t* __restrict__ idx, float* __restrict__ probs,
                                                        int discard) {
    __shared__ uint64_t buf[kCap];
    __shared__ uint64_t lists[kWarps][32];
    __shared__ int count, is_last;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");      // the logits come from the preceding kernel
    const int s = (int)blockIdx.x, m = (int)blockIdx.y;
    const int S = (int)gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t base = (int64_t)s * L;
    const int len = (int)((base + L <= N) ? L : (N - base));
    const float* row = logits + (int64_t)m * N + base;
    if (tid == 0) count = 0;

    // 1. each thread's largest candidate (its bucket: 8 runs of 4 consecutive logits)
    const bool vec = ((N | L) & 3) == 0;                       // rows and slices 16-byte aligned
    uint64_t mx = 0;
#pragma unroll
    for (int c = 0; c < kRuns; ++c) {
        const int i = 4 * (c * kThreads + tid);
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        load_run(row, i, len, vec, v);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (i + e < len) mx = umax(mx, candidate(monotone_key(v[e]), base + i + e));
    }

    // 2. the bound: 32nd largest of the per-thread maxima (0 if fewer than 32 threads hold logits)
    mx = warp_sort_desc(mx, lane);
    lists[warp][lane] = mx;
    __syncthreads();
    if (warp == 0) {
        uint64_t a = lists[0][lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) a = warp_merge_desc(umax(a, lists[w][31 - lane]), lane);
        if (lane == 31) lists[0][31] = a;
    }
    __syncthreads();
    const uint64_t lb = lists[0][31];
    // the slice again (the CTA's own recent reads: from L1), candidates at or above the bound
#pragma unroll
    for (int c = 0; c < kRuns; ++c) {
        const int i = 4 * (c * kThreads + tid);
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        load_run(row, i, len, vec, v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (i + e < len) {
                const uint64_t cv = candidate(monotone_key(v[e]), base + i + e);
                if (cv >= lb) buf[atomicAdd(&count, 1)] = cv;
            }
        }
    }
    __syncthreads();                                           // every logit of the slice has been read
    if (discard) {
        const uintptr_t b0 = (reinterpret_cast<uintptr_t>(row) + 127) & ~uintptr_t(127);
        const uintptr_t b1 = reinterpret_cast<uintptr_t>(row + len) & ~uintptr_t(127);
        for (uintptr_t a = b0 + (uintptr_t)tid * 128; a < b1; a += (uintptr_t)kThreads * 128)
            asm volatile("discard.global.L2 [%0], 128;" ::"l"(a) : "memory");
    }

    // 3. the slice's top 32: warp w sorts chunks w, w + 8, ... of 32 candidates and
    //    keeps the top 32 of them; the warps' lists are then merged by warp 0
    const int n = count;
    const int nch = (n + 31) / 32;
    uint64_t a = 0;                                            // an empty list is all zeros
    for (int ch = warp; ch < nch; ch += kWarps) {
        const int i = ch * 32 + lane;
        const uint64_t b = warp_sort_desc(i < n ? buf[i] : 0ull, lane);
        a = warp_merge_desc(umax(a, __shfl_sync(kFull, b, 31 - lane)), lane);
    }
    if (nch > 1) {                                             // uniform: n is read by every thread
        lists[warp][lane] = a;
        __syncthreads();
        if (warp == 0) {
            const int nw = nch < kWarps ? nch : kWarps;
            for (int w = 1; w < nw; ++w) a = warp_merge_desc(umax(a, lists[w][31 - lane]), lane);
        }
    }

    // 4. publish the slice's top 32 (warp 0); the row's last CTA merges.  The warp
    //    barrier orders the lanes' stores before lane 0's release of the ticket.
    uint64_t* row_cand = cand + (int64_t)m * S * kWidth;
    if (warp == 0) {
        __stcg(row_cand + (int64_t)s * kWidth + lane, a);
        __syncwarp();
        if (lane == 0) {
            int old;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(tickets + m) : "memory");
            const int lst = old == S - 1;
            if (lst) asm volatile("st.relaxed.gpu.global.s32 [%0], 0;" ::"l"(tickets + m) : "memory");
            is_last = lst;
        }
    }
    __syncthreads();                                           // lane 0's acquire, then the barrier, orders the
    if (!is_last) return;                                      // other CTAs' lists before the reads below

    // warp w merges lists w, w + 8, ..., loading four at a time
    a = 0;
    for (int l0 = warp; l0 < S; l0 += 4 * kWarps) {
        uint64_t r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int l = l0 + u * kWarps;
            r[u] = l < S ? __ldcg(row_cand + (int64_t)l * kWidth + (31 - lane)) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) a = warp_merge_desc(umax(a, r[u]), lane);
    }
    lists[warp][lane] = a;
    __syncthreads();
    a = tree_merge(lists, warp, lane);
    if (warp != 0) return;

    // lane j holds the rank-j candidate.  Probabilities in float pairs (about
    // 48 significant bits, so they round like double-precision ones):
    // exponentials lane-parallel, the sum as a butterfly and the cumulative sums
    // as a scan (a fixed order; it differs from a left-to-right sum by roundings
    // of about 1e-14 only)
    using namespace q4::pair;
    const float f0 = key_value((uint32_t)(__shfl_sync(kFull, a, 0) >> 32));
    const float fj = key_value((uint32_t)(a >> 32));
    fpair e = {0.0f, 0.0f};
    if (lane < top_k) {
        const fpair x = pair_div_f(two_sum(fj, -f0), temperature);   // (l_j - l_0) / T, <= 0
        if (x.hi >= -60.0f) {
            // exp(x.hi + x.lo) = exp(x.hi) * (1 + x.lo + x.lo^2 / 2), |x.lo| < 4e-6
            const float c = __fmaf_rn(__fmul_rn(0.5f, x.lo), x.lo, x.lo);
            e = pair_mul(exp_pair(x.hi), fast_two_sum(1.0f, c));
        } else {
            // below e^-60 (rare: a logit gap of 60 temperatures): the exponential in double
            const double ed = exp((double)x.hi + (double)x.lo);
            e = fpair{(float)ed, (float)(ed - (double)(float)ed)};
        }
    }
    fpair total = e;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const fpair t = {__shfl_xor_sync(kFull, total.hi, o), __shfl_xor_sync(kFull, total.lo, o)};
        total = pair_add(total, t);
    }
    const fpair pj = pair_div(e, total);
    fpair cum = pj;                                            // inclusive scan over ranks
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const fpair t = {__shfl_up_sync(kFull, cum.hi, o), __shfl_up_sync(kFull, cum.lo, o)};
        if (lane >= o) cum = pair_add(cum, t);
    }
    int keep = top_k;
    if (top_p < 1.0f) {
        const bool reached = cum.hi > top_p || (cum.hi == top_p && cum.lo >= 0.0f);
        const unsigned reach = __ballot_sync(kFull, lane < top_k && reached);
        if (reach) keep = __ffs(reach);                        // the entry that reaches top_p is kept
    }
    const fpair kept = {__shfl_sync(kFull, cum.hi, keep - 1), __shfl_sync(kFull, cum.lo, keep - 1)};
    const fpair out = pair_div(pj, kept);
    idx[m * kWidth + lane] = lane < top_k ? (int32_t)(~(uint32_t)(a & 0xFFFFFFFFull)) : -1;
    probs[m * kWidth + lane] = lane < keep ? out.hi : 0.0f;     // the pair's high part: its value rounded to float
}

}  // namespace topk
}  // namespace q4
