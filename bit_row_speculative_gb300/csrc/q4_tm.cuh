// Q4 verify-matmul kernel for sm_103a (K a multiple of 512).
//
// y[m,n] = sum_g ( s[n,g] * P[m,n,g] + r[n,g] * X[m,g] )
//   P[m,n,g] = sum_{k in g} (q[n,k] - c[n,g]) * x[m,k]      (tensor core, exact products)
//   X[m,g]   = sum_{k in g} x[m,k]
//   c[n,g]   = clamp(rint(-b/s), 0, 15),  r[n,g] = b + c*s
// which is w = s*q + b = s*(q - c) + r regrouped: q - c is an exact small
// integer, |r| <= s/2 whenever -b/s lies in [0,15], so s*P and r*X never cancel
// catastrophically, and an all-zero weight row (q == c, b == -c*s) gives
// exactly zero.
//
// Dequantization leaves the nibbles in place: the bf16 pair (v & 0x000F000F)
// is exactly q * 2^-133 (subnormal) and (v & 0x00F000F0) exactly q * 2^-129
// (subnormal, or the lowest binade for q >= 8); subtracting c in the same form
// (bf16x2, exact) gives (q - c) times a power of two.  One word of 8 nibbles
// costs one shift, four AND and four bf16x2 subtractions.  The x operand
// carries the inverse powers (x * 2^100 for even inputs, x * 2^96 for odd
// ones), so every tensor-core product is (q - c) * x * 2^-33 exactly and the
// fold applies s * 2^33.  (|x| must stay below 2^28 for x * 2^100 to be finite.)
//
// Two kernels per call, chained by programmatic dependent launch:
//   xrec_kernel  writes each group's x record to global scratch: the fp32
//                group sums X[0..W-1], then the rows of x for the group's 64
//                inputs as tensor-core core matrices (8 rows x 8 inputs, 128 B
//                each), 8-row blocks one after another (2112 bytes at W = 16,
//                4224 at W = 32; W = 16 for M <= 16, 32 for M <= 32).  Inputs
//                of each 8-block are in the dequantized order k0 k4 k1 k5 k2
//                k6 k3 k7 and scaled as above; rows >= M are zero.  A kernel
//                for M <= 8 copies only the first 1088 bytes (X and rows 0-7).
//                Inside a chained pass the glue kernel writes the records
//                instead, and this kernel is not launched.
//   q4_tm_kernel one persistent CTA per SM, 16 warps; tiles of 128 rows, a
//                stage is two groups (128 inputs) of one tile.
//     warp 0       producer: per stage one 128-row x 64-byte nibble box (TMA,
//                  64-byte swizzle) into a ring of slots, and bulk copies of
//                  the two x records into the same slot.  The weight boxes of
//                  the first ring-full of stages are issued before the kernel
//                  waits for its predecessor (they need nothing from it);
//                  every record copy comes after that wait.
//     warps 1..3   MMA issuers, one per team: per stage of the team 8 MMAs
//                  M128 N=W K16 (A = the dequantized weights in the team's
//                  tensor memory, B = the x records in shared memory, D = the
//                  team's P) and a commit to the team's "done" barrier.  Each
//                  column of an N = 32 MMA carries the same bits as the same
//                  column of an N = 16 MMA (tested: rows at M = 17..32 equal
//                  the rows at M <= 16), so row invariance holds across widths.
//     warps 4..15  three consumer teams of 4 warps; stage i belongs to team
//                  i % 3.  Every team covers all 128 rows (one row per
//                  thread).  At W = 16 a team keeps two A buffers: in its
//                  iteration for stage i it dequantizes stage i into one
//                  buffer while the MMAs of its previous stage (i - 3) finish
//                  on the other, then folds that previous stage's P into its
//                  own fp32 sums with s, r and X, frees that stage's slot and
//                  hands stage i over.  At W = 32 (one A buffer, to fit tensor
//                  memory) it folds the previous stage first.  The three teams
//                  overlap with each other.  At the end of each tile segment
//                  the teams' sums are added in team order through shared
//                  memory.
// The ring has a multiple of 3 slots, so a slot always serves the same team,
// and every barrier is waited on by threads that pass through its phases in
// order (a parity wait never sees a phase two steps away).
// Work split: the T*G/2 (tile, group pair) units are cut into equal contiguous
// ranges, one per CTA (stream-K).  A tile whose units span several CTAs is
// finished by the last of them to arrive, which adds the partial sums in
// increasing CTA order.  The split depends only on N, K and the grid size, and
// nothing in the arithmetic of row m depends on the other rows, so every
// row's result is independent of M.
// No CTA waits for another except through the last-arriver counter, which
// never blocks.  Every barrier wait is bounded; a wait that runs out sets the
// error word and the CTA runs to its end without further waiting.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "q4_sm100.cuh"

namespace q4 {
namespace tm {

constexpr int kRowsTile = 128;              // rows per tile (tensor-memory lanes)
constexpr int kTeams = 3;                   // consumer teams (one warpgroup each)
constexpr int kIssuersPerTeam = 1;          // MMA issuing threads per team (they split the two groups)
constexpr int kIssuers = kIssuersPerTeam * kTeams;
constexpr int kConsumerWarp0 = 4;           // warps 4.. (warp % 4 = tensor-memory lane quarter)
constexpr int kThreads = (kConsumerWarp0 + 4 * kTeams) * 32;   // 512
constexpr int kConsumerThreads = kTeams * 128;
static_assert(kIssuers + 1 <= kConsumerWarp0, "control warps");

// Row width W: the x records and the MMAs cover W = 16 rows for M <= 16 and
// W = 32 rows for 16 < M <= 32.  Everything of the layout below depends on W.
template <int MT>
__host__ __device__ constexpr int width() { return MT > 16 ? 32 : 16; }
__host__ __device__ constexpr int rec_bytes(int W) { return 4 * W + (W / 8) * 1024; }   // X[W] fp32, then W/8 blocks of 8 rows
__host__ __device__ constexpr int rec_b(int W) { return 4 * W; }                        // offset of the core matrices
constexpr int kRecHalf = 1088;                        // W = 16: X and rows 0-7
constexpr int kNibStage = kRowsTile * 64;             // 8 KB: 128 rows x 64 B (two groups)
__host__ __device__ constexpr int stage_bytes(int W) { return ((kNibStage + 2 * rec_bytes(W) + 1023) / 1024) * 1024; }
__host__ __device__ constexpr int stages(int W) { return W == 16 ? 12 : 9; }            // a multiple of kTeams
// team sums of a segment: two buffers used alternately at W = 16, one at W = 32
__host__ __device__ constexpr int red_buffers(int W) { return W == 16 ? 2 : 1; }
__host__ __device__ constexpr int red_bytes(int W) { return red_buffers(W) * kTeams * W * kRowsTile * 4; }
constexpr int kBarrierBytes = 1024;
__host__ __device__ constexpr int smem_bytes_w(int W) {
    return stages(W) * stage_bytes(W) + red_bytes(W) + kBarrierBytes + 1024 /* alignment slack */;
}
static_assert(stages(16) % kTeams == 0 && stages(32) % kTeams == 0, "each ring slot must belong to one team");
static_assert(smem_bytes_w(16) <= 232448 && smem_bytes_w(32) <= 232448, "shared memory per CTA");

// tensor-memory columns per team: the dequantized A of a stage (two groups x
// 32), twice at W = 16 (double-buffered), once at W = 32; then P (two groups x W)
constexpr uint32_t kColsA = 64;
__host__ __device__ constexpr uint32_t a_buffers(int W) { return W == 16 ? 2 : 1; }
__host__ __device__ constexpr uint32_t col_p(int W) { return a_buffers(W) * kColsA; }
__host__ __device__ constexpr uint32_t cols_team(int W) { return col_p(W) + 2 * W; }
constexpr uint32_t kTmemCols = 512;
static_assert(kTeams * cols_team(16) <= kTmemCols && kTeams * cols_team(32) <= kTmemCols,
              "tensor memory over-subscribed");

constexpr long long kWaitLimit = 2000000000LL;     // cycles (about one second)
constexpr float kFoldScale = 8589934592.0f;        // 2^33: undoes 2^-133 (weights) * 2^100 (x)
constexpr uint32_t kXScaleEven = 0x71807180u;      // bf16 pair (2^100, 2^100)
constexpr uint32_t kXScaleOdd = 0x6F806F80u;       // bf16 pair (2^96, 2^96)

struct Params {
    const uint8_t* W;           // packed weights
    float* y;                   // [M, N]
    float* partials;            // scratch: [C][2][W][128]
    int* sems;                  // scratch: [C], zero between launches
    const uint8_t* xt;          // x records [G][rec_bytes(W)] (written by xrec_kernel)
    unsigned int* error_word;   // set on a timed-out wait
    int64_t N;
    int64_t K;
    int M;
    int G;                      // K / 64 (a multiple of 8)
    int GP;                     // G / 2 group pairs (stages per tile)
    int T;                      // tiles of 128 rows
    int U;                      // T * GP units
    int C;                      // CTAs (grid size)
#ifdef Q4_TRACE
    unsigned long long* trace;  // developer timing trace (compiled in only with Q4_TRACE)
#endif
};

#ifdef Q4_TRACE
#define Q4_TMTR(p, idx)                                                                   \
    do {                                                                                  \
        if ((p).trace && blockIdx.x == 0 && (idx) < 4096) (p).trace[(idx)] = clock64(); \
    } while (0)
// globaltimer (ns) of any CTA, for start/end skew across CTAs
#define Q4_TMGT(p, idx)                                                                  \
    do {                                                                                 \
        if ((p).trace && (idx) < 4096) {                                                 \
            unsigned long long gt_;                                                      \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(gt_));                      \
            (p).trace[(idx)] = gt_;                                                      \
        }                                                                                \
    } while (0)
#else
#define Q4_TMTR(p, idx) \
    do {                \
    } while (0)
#define Q4_TMGT(p, idx) \
    do {                \
    } while (0)
#endif

// Range of units owned by CTA c.
__device__ __forceinline__ int range_start(int U, int C, int c) { return (int)(((int64_t)U * c) / C); }

// CTA that owns unit u.
__device__ __forceinline__ int cta_of_unit(int U, int C, int u) {
    int c = (int)(((int64_t)u * C) / U);
    while (c + 1 < C && range_start(U, C, c + 1) <= u) ++c;
    while (c > 0 && range_start(U, C, c) > u) --c;
    return c;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t and32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, 0, 0xC0;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// acc0/acc1 = fma(a, b0/b1, acc0/acc1) in one packed instruction (each lane an
// IEEE fma, identical to two scalar fmas).
__device__ __forceinline__ void fma2(float& acc0, float& acc1, float a, float b0, float b1) {
    uint64_t d;
    const uint64_t A = ((uint64_t)__float_as_uint(a) << 32) | __float_as_uint(a);
    const uint64_t B = ((uint64_t)__float_as_uint(b1) << 32) | __float_as_uint(b0);
    const uint64_t C = ((uint64_t)__float_as_uint(acc1) << 32) | __float_as_uint(acc0);
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(A), "l"(B), "l"(C));
    acc0 = __uint_as_float((uint32_t)d);
    acc1 = __uint_as_float((uint32_t)(d >> 32));
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void record_timeout(const Params& p, unsigned int code, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(p.error_word, code);
}

// Bounded wait that also gives up at once when another role has already
// given up (the whole CTA then runs to its end without further waiting).
__device__ __forceinline__ bool wait_or_abort(const Params& p, uint64_t* bar, uint32_t parity, unsigned code,
                                              volatile int* abort_flag) {
    if (q4::sm100::mbar_try_wait(bar, parity)) return true;       // fast path: already complete
    if (*abort_flag) return false;
    if (q4::sm100::mbar_wait(bar, parity, kWaitLimit)) return true;
    record_timeout(p, code, abort_flag);
    return false;
}

// ------------------------------------------------------------------ x records
// One CTA per group of 64 inputs, 8 * W threads: thread t takes row m = t / 8
// and 8-block kc = t % 8 of the group.
template <int W>
__global__ void __launch_bounds__(8 * W) xrec_kernel(const uint16_t* __restrict__ x, int M, int64_t K,
                                                     uint8_t* __restrict__ xt) {
    pdl_launch_dependents();
    // x may come from the preceding kernel, and the preceding matmul may still
    // read the records of its own call: wait for it first
    pdl_wait();
    const int g = blockIdx.x;
    const int t = threadIdx.x;
    const int m = t >> 3, kc = t & 7;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (m < M) v = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)m * K + (int64_t)g * 64 + kc * 8));
    uint4 o;
    o.x = bf16x2_mul(prmt(v.x, v.z, 0x5410u), kXScaleEven);    // (k0, k4)
    o.y = bf16x2_mul(prmt(v.x, v.z, 0x7632u), kXScaleOdd);     // (k1, k5)
    o.z = bf16x2_mul(prmt(v.y, v.w, 0x5410u), kXScaleEven);    // (k2, k6)
    o.w = bf16x2_mul(prmt(v.y, v.w, 0x7632u), kXScaleOdd);     // (k3, k7)
    uint8_t* rec = xt + (int64_t)g * rec_bytes(W);
    *reinterpret_cast<uint4*>(rec + rec_b(W) + (m >> 3) * 1024 + kc * 128 + (m & 7) * 16) = o;
    // X: the 8 inputs in increasing k, then the 8 block sums of the row (in 8
    // consecutive lanes) by a fixed xor tree
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        s = __fadd_rn(s, __uint_as_float(w[i] << 16));
        s = __fadd_rn(s, __uint_as_float(w[i] & 0xFFFF0000u));
    }
    s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 1));
    s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 2));
    s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 4));
    if (kc == 0) reinterpret_cast<float*>(rec)[m] = s;
}

// Dequantize the 64 nibbles of one row and group (two 16-byte chunks) into 32
// bf16 pairs, (q - c) * 2^-133 for the even inputs and (q - c) * 2^-129 for the
// odd ones, word order (k0,k4) (k1,k5) (k2,k6) (k3,k7) per 8 inputs.
// cc0 = c * 0x00010001 (c * 2^-133 as a bf16 pair), cc1 = cc0 << 4.
__device__ __forceinline__ void dequant64(const uint4& n0, const uint4& n1, uint32_t cc0, uint32_t (&a)[32]) {
    const uint32_t cc1 = cc0 << 4;
    const uint32_t wv[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
        const uint32_t v = wv[wi], u = v >> 8;
        a[4 * wi + 0] = bf16x2_sub(and32(v, 0x000F000Fu), cc0);
        a[4 * wi + 1] = bf16x2_sub(and32(v, 0x00F000F0u), cc1);
        a[4 * wi + 2] = bf16x2_sub(and32(u, 0x000F000Fu), cc0);
        a[4 * wi + 3] = bf16x2_sub(and32(u, 0x00F000F0u), cc1);
    }
}

// Constants of one row and group from its bf16 scale and bias:
// c = clamp(rint(-b/s), 0, 15) (NaN -> 0), r = b + c*s, s * 2^33 and the bf16
// pair c * 2^-133.
__device__ __forceinline__ void group_constants(uint32_t s_bits, uint32_t b_bits, float& s_fold, float& r,
                                                uint32_t& cc0) {
    const float s = __uint_as_float(s_bits << 16);
    const float b = __uint_as_float(b_bits << 16);
    float cf = rintf(__fdividef(-b, s));
    cf = fminf(fmaxf(cf, 0.0f), 15.0f);
    r = __fmaf_rn(cf, s, b);
    s_fold = s * kFoldScale;
    const uint32_t ci = __float_as_uint(__fadd_rn(8388608.0f, cf)) & 0xFu;   // low bits of 2^23 + c
    cc0 = ci * 0x00010001u;
}

template <int MT>
__device__ __forceinline__ void fold_group(float (&acc)[MT], const uint32_t* P, const float* xs, float s, float r) {
    if (MT == 1) {
        acc[0] = __fmaf_rn(s, __uint_as_float(P[0]), __fmaf_rn(r, xs[0], acc[0]));
    } else {
#pragma unroll
        for (int m4 = 0; m4 < (MT + 3) / 4; ++m4) {
            float X[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (MT >= 4) {
                const float4 v = reinterpret_cast<const float4*>(xs)[m4];
                X[0] = v.x;
                X[1] = v.y;
                X[2] = v.z;
                X[3] = v.w;
            } else {
                X[0] = xs[0];
                X[1] = xs[1];
            }
#pragma unroll
            for (int i = 0; i < 4; i += 2) {
                const int m = 4 * m4 + i;
                if (m < MT) {
                    fma2(acc[m], acc[m + 1], r, X[i], X[i + 1]);
                    fma2(acc[m], acc[m + 1], s, __uint_as_float(P[m]), __uint_as_float(P[m + 1]));
                }
            }
        }
    }
}

// End of a tile segment: the teams' sums of rows [t*128, t*128+128) are added
// in team order; a whole tile is stored, a partial one published and finished
// by the last CTA to arrive (partials added in increasing CTA order).  Called
// by all consumer threads; thread (team, row) handles m = team + kTeams*j.
template <int MT>
__device__ void end_segment(const Params& p, float (&acc)[MT], float* red, int t, bool whole, int slot, int team,
                            int row, int c_id, int* bcast, bool live) {
    // red: this segment's buffer (at W = 16 the caller alternates two by segment)
    constexpr int W = width<MT>();
    constexpr int kJ = (MT + kTeams - 1) / kTeams;
#pragma unroll
    for (int m = 0; m < MT; ++m) red[(team * W + m) * kRowsTile + row] = acc[m];
    named_barrier(1, kConsumerThreads);
    const int64_t n = (int64_t)t * kRowsTile + row;
    float v[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
        const int m = team + kTeams * j;
        v[j] = 0.0f;
        if (m < MT) {
#pragma unroll
            for (int tm_ = 0; tm_ < kTeams; ++tm_) v[j] = __fadd_rn(v[j], red[(tm_ * W + m) * kRowsTile + row]);
        }
    }
    // one buffer: every thread has read it before any thread writes it for the next segment
    if (red_buffers(W) == 1) named_barrier(1, kConsumerThreads);
    if (whole) {
        if (live && n < p.N) {
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                const int m = team + kTeams * j;
                if (m < MT && m < p.M) p.y[(int64_t)m * p.N + n] = v[j];
            }
        }
    } else {
        float* dst = p.partials + (((int64_t)c_id * 2 + slot) * W) * kRowsTile + row;
        if (live) {
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                const int m = team + kTeams * j;
                if (m < MT) __stcg(dst + m * kRowsTile, v[j]);
            }
        }
        // the barrier orders every consumer thread's partial stores before
        // thread 0's release (acq_rel) increment of the tile counter; the last
        // contributor's acquire, followed by the next barrier, orders the other
        // CTAs' partials before every thread's reads below
        named_barrier(1, kConsumerThreads);
        const int tu = t * p.GP;
        const int c_first = cta_of_unit(p.U, p.C, tu);
        const int c_last = cta_of_unit(p.U, p.C, tu + p.GP - 1);
        if (team == 0 && row == 0) {
            int last = 0;
            if (live) {
                int* sem = p.sems + c_first;
                int old;
                asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(sem) : "memory");
                if (old == c_last - c_first) {
                    asm volatile("st.relaxed.gpu.global.s32 [%0], 0;" ::"l"(sem) : "memory");   // zero for the next launch
                    last = 1;
                }
            }
            *bcast = last;
        }
        named_barrier(1, kConsumerThreads);
        if (*bcast) {
#pragma unroll
            for (int j = 0; j < kJ; ++j) v[j] = 0.0f;
            for (int c = c_first; c <= c_last; ++c) {
                const int cs = range_start(p.U, p.C, c);
                const int cslot = (cs / p.GP == t) ? 0 : 1;   // the tile is c's first segment, or its last
                const float* src = p.partials + (((int64_t)c * 2 + cslot) * W) * kRowsTile + row;
#pragma unroll
                for (int j = 0; j < kJ; ++j) {
                    const int m = team + kTeams * j;
                    if (m < MT) v[j] = __fadd_rn(v[j], __ldcg(src + m * kRowsTile));
                }
            }
            if (n < p.N) {
#pragma unroll
                for (int j = 0; j < kJ; ++j) {
                    const int m = team + kTeams * j;
                    if (m < MT && m < p.M) p.y[(int64_t)m * p.N + n] = v[j];
                }
            }
        }
    }
    // At W = 16 red alternates between two buffers by segment, so a buffer is
    // rewritten only after every thread has passed the first barrier of the
    // segment between (and with it finished reading here); at W = 32 the
    // barrier after the reads above does that.  bcast is written only on the
    // partial path, between two barriers
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
q4_tm_kernel(const __grid_constant__ CUtensorMap map_nib, const Params p) {
    using namespace q4::sm100;
    constexpr int W = width<MT>();
    constexpr int kStages = stages(W);
    constexpr int kStageBytes = stage_bytes(W);
    constexpr int kRec = rec_bytes(W);
    constexpr int kRecB = rec_b(W);
    constexpr int kRedBytes = red_bytes(W);
    constexpr uint32_t kColP = col_p(W);
    constexpr uint32_t kColsTeam = cols_team(W);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* red = reinterpret_cast<float*>(smem + kStages * kStageBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kRedBytes);   // nibbles and records landed
    uint64_t* empty = full + kStages;                  // slot free: the owning team has folded it
    uint64_t* ready = empty + kStages;                 // [kTeams]: the team's A of a stage stored, its P free
    uint64_t* done = ready + kTeams;                   // [kTeams]: the team's MMAs of a stage complete
    uint64_t* fin = done + kTeams;                     // [kIssuers]
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(fin + kIssuers);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);
    int* bcast = const_cast<int*>(abort_flag) + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c_id = blockIdx.x;

    // the next kernel on the stream may start now
    pdl_launch_dependents();

    // This CTA's units (= stages) [u0, u1): unit u is group pair u % GP of tile u / GP.
    const int u0 = range_start(p.U, p.C, c_id);
    const int u1 = range_start(p.U, p.C, c_id + 1);
    const int nst = u1 - u0;
    const int t0 = u0 / p.GP, gp0 = u0 - t0 * p.GP;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 2);
            mbar_init(&empty[s], 4);
        }
        for (int i = 0; i < kTeams; ++i) {
            mbar_init(&ready[i], 4);
            mbar_init(&done[i], kIssuersPerTeam);
        }
        for (int i = 0; i < kIssuers; ++i) mbar_init(&fin[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) prefetch_tensormap(&map_nib);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_slot;
    if (threadIdx.x == 0) {
        Q4_TMTR(p, 4000);
        Q4_TMGT(p, 2400 + 8 * c_id);
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int tn = t0, gn = gp0;                     // tile and group pair of the next nibble load
            // one barrier per stage, two arrivals: the nibble box and the x records, each with its bytes
            auto issue_nibbles = [&](int slot) {
                mbar_arrive_expect_tx(&full[slot], (uint32_t)kNibStage);
                tma_load_2d_hint(smem + slot * kStageBytes, &map_nib, &full[slot], gn * 64, tn * kRowsTile, pol);
                if (++gn == p.GP) {
                    gn = 0;
                    ++tn;
                }
            };
            // the weight stream needs nothing from the preceding kernel
            const int pre = nst < kStages ? nst : kStages;
            for (int si = 0; si < pre; ++si) issue_nibbles(si);
            int issued = pre, rec_issued = 0;
            pdl_wait();                                // the x records of this call are complete
            Q4_TMTR(p, 4002);
            int gr = gp0;                              // group pair of the next record copy
            int slot = 0;
            uint32_t ph = 0;
            for (int si = 0; si < nst; ++si) {
                if (si >= kStages) {
                    if (!wait_or_abort(p, &empty[slot], ph ^ 1u, 1u, abort_flag)) break;
                    Q4_TMTR(p, si);
                    issue_nibbles(slot);
                    ++issued;
                }
                uint8_t* dst = smem + slot * kStageBytes + kNibStage;
                const uint8_t* src = p.xt + (int64_t)(2 * gr) * kRec;
                if (MT > 8) {
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(2 * kRec));
                    bulk_copy_g2s(dst, src, (uint32_t)(2 * kRec), &full[slot]);
                } else {
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(2 * kRecHalf));
                    bulk_copy_g2s(dst, src, (uint32_t)kRecHalf, &full[slot]);
                    bulk_copy_g2s(dst + kRec, src + kRec, (uint32_t)kRecHalf, &full[slot]);
                }
                ++rec_issued;
                if (++gr == p.GP) gr = 0;
                if (++slot == kStages) {
                    slot = 0;
                    ph ^= 1u;
                }
            }
            // every issued copy must have landed before the CTA may exit; a stage whose
            // records were never issued (a given-up wait) gets its second arrival without bytes
            for (int s2 = rec_issued; s2 < issued; ++s2) mbar_arrive(&full[s2 % kStages]);
            for (int s2 = (issued > kStages ? issued - kStages : 0); s2 < issued; ++s2)
                mbar_wait(&full[s2 % kStages], (s2 / kStages) & 1, kWaitLimit);
        }
    } else if (warp <= kIssuers) {
        // ------------------------------------------------------------ MMA issuers (warp-uniform loop)
        const int team = (warp - 1) / kIssuersPerTeam, gsel = (warp - 1) % kIssuersPerTeam;
        const uint32_t idesc = idesc_bf16_f32(128, W);
        // B: core matrices K-major, 128 B apart along K, rows 8-15 1024 B after rows 0-7
        const uint64_t bdesc0 = smem_desc_noswizzle(smem_u32(smem + kNibStage + kRecB), 128, 1024);
        const uint32_t tbase = tmem + (uint32_t)team * kColsTeam;
        for (int si = team; si < nst; si += kTeams) {
            const int slot = si % kStages;
            const int j = si / kTeams;
            if (!__all_sync(0xFFFFFFFFu, wait_or_abort(p, &full[slot], (uint32_t)((si / kStages) & 1), 2u, abort_flag)))
                break;
            if (!__all_sync(0xFFFFFFFFu, wait_or_abort(p, &ready[team], (uint32_t)(j & 1), 2u, abort_flag))) break;
            tc_fence_after();
            const uint64_t bd = bdesc0 + (uint64_t)((slot * kStageBytes) >> 4);
            const uint32_t aS = tbase + (a_buffers(W) == 2 ? (uint32_t)(j & 1) * kColsA : 0u);
            const uint32_t dS = tbase + kColP;
            if (lane == 0) {
                if (team == 0 && gsel == 0) Q4_TMTR(p, 2000 + 2 * si);
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    if (g % kIssuersPerTeam != gsel) continue;
                    const uint64_t bg = bd + (uint64_t)((g * kRec) >> 4);
                    // P of group g: W columns (N = W: the record's 8-row blocks, 1024 bytes apart)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_ts(dS + (uint32_t)W * g, aS + 32u * g + 8u * kk, bg + 16u * kk, idesc, kk > 0 ? 1u : 0u);
                }
                tc_commit(&done[team]);
                if (team == 0 && gsel == 0) Q4_TMTR(p, 2001 + 2 * si);
            }
            __syncwarp();
        }
        // no MMA of this warp may still run when tensor memory is freed
        if (lane == 0) {
            tc_commit(&fin[warp - 1]);
            mbar_wait(&fin[warp - 1], 0, kWaitLimit);
        }
        __syncwarp();
    } else if (warp >= kConsumerWarp0) {
        // ------------------------------------------------------------ consumer teams
        const int team = (warp - kConsumerWarp0) >> 2;
        const int q = warp & 3;                        // tensor-memory lane quarter of this warp
        const int row = q * 32 + lane;                 // row within the tile
        const uint32_t lane_field = (uint32_t)(q * 32) << 16;
        const uint32_t tbase = tmem + lane_field + (uint32_t)team * kColsTeam;
        const uint32_t dP = tbase + kColP;
        [[maybe_unused]] const int tr = (lane == 0 && q == 0 && team == 0) ? 1000 : 1 << 20;

        // scale and bias planes: this team's two groups of a stage are one 4-byte word per plane
        const uint8_t* splane = p.W + p.N * (p.K / 2);
        const uint8_t* bplane = splane + p.N * p.G * 2;
        // cursor of the next scale/bias load: the team's stages in order, each
        // kTeams units after the previous one (no divisions in the loop)
        int ld_si = team, ld_t = (u0 + team) / p.GP, ld_gp = (u0 + team) - ld_t * p.GP;
        auto load_next = [&](uint32_t& sv, uint32_t& bv) {
            const int64_t n = (int64_t)ld_t * kRowsTile + row;
            if (ld_si < nst && n < p.N) {
                const int64_t off = (n * p.G + 2 * ld_gp) * 2;
                sv = __ldg(reinterpret_cast<const uint32_t*>(splane + off));
                bv = __ldg(reinterpret_cast<const uint32_t*>(bplane + off));
            } else {
                sv = 0u;
                bv = 0u;
            }
            ld_si += kTeams;
            ld_gp += kTeams;
            while (ld_gp >= p.GP) {
                ld_gp -= p.GP;
                ++ld_t;
            }
        };
        // Scale/bias words are loaded two team stages before their constants are
        // formed, into two register pairs used alternately (the loop below is
        // unrolled by two), so no instruction reads a register whose load is
        // still in flight.
        uint32_t sA, bA, sB, bB;
        float s0, r0, s1, r1;                          // constants of the stage being dequantized
        uint32_t cc0, cc1;
        {
            uint32_t s_a, b_a;
            load_next(s_a, b_a);
            load_next(sA, bA);
            load_next(sB, bB);
            group_constants(s_a, b_a, s0, r0, cc0);
            group_constants(s_a >> 16, b_a >> 16, s1, r1, cc1);
        }
        // tile of the team's current stage, advanced the same way
        int st_t = (u0 + team) / p.GP, st_gp = (u0 + team) - st_t * p.GP;

        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
        bool live = true;

        // segments: tile t0 + k for k = 0 .. n_seg-1, each closed exactly once by every team
        const int n_seg = (u1 - 1) / p.GP - t0 + 1;
        int cur_seg = 0;
        auto close_segments_before = [&](int seg) {
            while (cur_seg < seg) {
                const int tt = t0 + cur_seg;
                const bool whole = u0 <= tt * p.GP && (tt + 1) * p.GP <= u1;
                if (team == 0 && row == 0 && cur_seg < 2) Q4_TMGT(p, 2403 + 8 * c_id + 2 * cur_seg);
                end_segment<MT>(p, acc, red + (red_buffers(W) == 2 ? (cur_seg & 1) : 0) * (kTeams * W * kRowsTile), tt, whole,
                                cur_seg == 0 ? 0 : 1, team, row, c_id, bcast, !*abort_flag);
                if (team == 0 && row == 0 && cur_seg < 2) {
                    Q4_TMGT(p, 2404 + 8 * c_id + 2 * cur_seg);
#ifdef Q4_TRACE
                    if (p.trace && !whole && *bcast) p.trace[2407 + 8 * c_id] |= 1ull << cur_seg;
#endif
                }
                ++cur_seg;
            }
        };

        // the stage handed over in the previous iteration, folded in this one
        int pend = -1, pend_seg = 0;
        float ps0 = 0.f, pr0 = 0.f, ps1 = 0.f, pr1 = 0.f;
        // hand the team's current stage to its issuer: its A is stored and P is free
        auto arrive_ready = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ready[team]);
        };
        // signal_ready (W = 16): the hand-over happens as soon as P has been loaded into
        // registers, so the next MMAs run while this stage's P is folded
        auto fold_pending = [&](bool signal_ready) {
            const int pslot = pend % kStages;
            live = __all_sync(0xFFFFFFFFu, live && wait_or_abort(p, &done[team], (uint32_t)((pend / kTeams) & 1), 4u,
                                                                 abort_flag));
            Q4_TMTR(p, tr + 8 * (pend / kTeams) + 7);
            close_segments_before(pend_seg);
            if (live) {
                tc_fence_after();
                const uint8_t* psb = smem + pslot * kStageBytes + kNibStage;
                const float* xs0 = reinterpret_cast<const float*>(psb);
                const float* xs1 = reinterpret_cast<const float*>(psb + kRec);
                if (MT <= 8) {
                    uint32_t P0[8], P1[8];
                    tmem_ld_32x32b_x8(dP, P0);
                    tmem_ld_32x32b_x8(dP + 16u, P1);
                    tmem_wait_ld();
                    if (signal_ready) arrive_ready();
                    fold_group<MT>(acc, P0, xs0, ps0, pr0);
                    fold_group<MT>(acc, P1, xs1, ps1, pr1);
                } else if (W == 32) {
                    // 32 columns per group, one group at a time (registers)
                    uint32_t P[32];
                    tmem_ld_32x32b_x32(dP, P);
                    tmem_wait_ld();
                    fold_group<MT>(acc, P, xs0, ps0, pr0);
                    tmem_ld_32x32b_x32(dP + 32u, P);
                    tmem_wait_ld();
                    fold_group<MT>(acc, P, xs1, ps1, pr1);
                } else {
                    uint32_t P0[16], P1[16];
                    tmem_ld_32x32b_x16(dP, P0);
                    tmem_ld_32x32b_x16(dP + 16u, P1);
                    tmem_wait_ld();
                    if (signal_ready) arrive_ready();
                    fold_group<MT>(acc, P0, xs0, ps0, pr0);
                    fold_group<MT>(acc, P1, xs1, ps1, pr1);
                }
            } else if (signal_ready) {
                arrive_ready();
            }
            // that stage's slot (nibbles, records) has been read, and so has P
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[pslot]);
        };

        // one team stage: sw/bw hold the words of the team's next stage on entry
        // and are reloaded with those of the stage after the one that follows
        auto team_stage = [&](int si, uint32_t& sw, uint32_t& bw) {
            const int slot = si % kStages;
            const int j = si / kTeams;
            Q4_TMTR(p, tr + 8 * j + 0);
            if (si == 0 && row == 0) Q4_TMGT(p, 2402 + 8 * c_id);
            live = __all_sync(0xFFFFFFFFu, live && wait_or_abort(p, &full[slot], (uint32_t)((si / kStages) & 1), 8u,
                                                                 abort_flag));
            Q4_TMTR(p, tr + 8 * j + 1);
            // one A buffer (W = 32): the previous stage's MMAs must have read it, so fold first
            if (a_buffers(W) == 1 && pend >= 0) fold_pending(false);
            // dequantize into this stage's A buffer (at W = 16 the other one may still feed the previous MMAs)
            if (live) {
                const uint8_t* nb = smem + slot * kStageBytes + row * 64;
                const int sx = (row >> 1) & 3;         // 64-byte swizzle: chunk index ^ bits 7-8 of the offset
                const uint32_t aA = tbase + (a_buffers(W) == 2 ? (uint32_t)(j & 1) * kColsA : 0u);
                uint32_t av0[32], av1[32];
                {
                    const uint4 na = *reinterpret_cast<const uint4*>(nb + ((0 ^ sx) << 4));
                    const uint4 nc = *reinterpret_cast<const uint4*>(nb + ((1 ^ sx) << 4));
                    dequant64(na, nc, cc0, av0);
                    tmem_st_32x32b_x32(aA, av0);
                }
                {
                    const uint4 na = *reinterpret_cast<const uint4*>(nb + ((2 ^ sx) << 4));
                    const uint4 nc = *reinterpret_cast<const uint4*>(nb + ((3 ^ sx) << 4));
                    dequant64(na, nc, cc1, av1);
                    tmem_st_32x32b_x32(aA + 32u, av1);
                }
                tmem_wait_st();
            }
            Q4_TMTR(p, tr + 8 * j + 2);
            // fold the previous stage (its MMAs ran meanwhile); then P is free again
            const bool early = a_buffers(W) == 2 && pend >= 0;   // W = 16: hand over inside the fold
            if (early) fold_pending(true);
            Q4_TMTR(p, tr + 8 * j + 3);
            if (!early) arrive_ready();
            Q4_TMTR(p, tr + 8 * j + 4);
            // this stage becomes the pending one; constants of the team's next stage
            pend = si;
            pend_seg = st_t - t0;
            st_gp += kTeams;
            while (st_gp >= p.GP) {
                st_gp -= p.GP;
                ++st_t;
            }
            ps0 = s0;
            pr0 = r0;
            ps1 = s1;
            pr1 = r1;
            group_constants(sw, bw, s0, r0, cc0);
            group_constants(sw >> 16, bw >> 16, s1, r1, cc1);
            Q4_TMTR(p, tr + 8 * j + 5);
            load_next(sw, bw);
            Q4_TMTR(p, tr + 8 * j + 6);
        };
        if (W == 32) {
            // one stage per iteration (fewer live registers at 32 rows); the prefetched
            // pairs rotate so that each stage again finds its words in sA, bA
            for (int si = team; si < nst; si += kTeams) {
                team_stage(si, sA, bA);
                const uint32_t ts = sA, tb = bA;
                sA = sB;
                bA = bB;
                sB = ts;
                bB = tb;
            }
        } else {
            for (int si = team; si < nst; si += 2 * kTeams) {
                team_stage(si, sA, bA);
                if (si + kTeams < nst) team_stage(si + kTeams, sB, bB);
            }
        }
        if (pend >= 0) fold_pending(false);
        close_segments_before(n_seg);
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        Q4_TMTR(p, 4001);
        Q4_TMGT(p, 2401 + 8 * c_id);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int MT>
inline int smem_bytes() { return smem_bytes_w(width<MT>()); }
inline size_t partial_floats(int C) { return (size_t)C * 2 * 32 * kRowsTile; }   // sized for W = 32
inline size_t sem_ints(int C) { return (size_t)C; }

}  // namespace tm
}  // namespace q4
