// Q4 verify-matmul kernel for sm_103a (K a multiple of 512): one launch per call,
// register-operand tensor-core MMAs (mma.sync m16n8k16, bf16 -> fp32).
//
// y[m,n] = sum_g ( s[n,g] * P[m,n,g] + r[n,g] * X[m,g] )
//   P[m,n,g] = sum_{k in g} (q[n,k] - c[n,g]) * x[m,k]     (tensor core, exact products)
//   X[m,g]   = sum_{k in g} x[m,k]
//   c[n,g]   = clamp(rint(-b/s), 0, 15),  r[n,g] = b + c*s
// which is w = s*q + b = s*(q - c) + r regrouped: q - c is an exact small
// integer, |r| <= s/2 when -b/s lies in [0,15], so s*P and r*X never cancel
// catastrophically, and an all-zero weight row gives exactly zero.
//
// Dequantization without shifts into the bf16 exponent: with the nibbles left
// in place, the bf16 pair (w & 0x000F000F) is exactly q * 2^-133 (subnormal)
// and (w & 0x00F000F0) exactly q * 2^-129 (subnormal, or the lowest binade
// for q >= 8); subtracting c in the same form (bf16x2, exact) gives (q - c)
// times a power of two.  The x operand carries the inverse powers (x * 2^100,
// x * 2^96 for the 2^-129 slots), so every product is (q - c) * x * 2^-33
// exactly, and the fold applies s * 2^33.  (|x| must stay below 2^28 for
// x * 2^100 to be finite.)  The weights go from shared memory through
// registers straight into the MMA: no tensor-memory traffic and no hand-off
// between warps inside a stage.
//
// One persistent CTA per SM, 16 warps, tiles of 480 rows; a stage is an
// aligned pair of groups (inputs 128k .. 128k+127) of one tile.
//   x records   each stage's two groups of x -- the M <= 16 rows for the
//               groups' 64 inputs as mma.sync B fragments, scaled as above, and
//               the group sums X -- are written into the stage's slot by the
//               consumer warps two stages ahead of their use, straight from x.
//   warp 0      producer: per stage four 120-row x 64-byte nibble boxes (TMA,
//               64-byte swizzle) into a 6-stage ring.  One barrier per stage:
//               the nibble bytes plus one arrival per consumer warp for the
//               records.
//   warps 1..15 consumers, 32 rows each (two m16 slabs): per stage they derive
//               the groups' constants (one row per lane, shared through shared
//               memory), dequantize into A fragments, run the m16n8k16 MMAs
//               against the B fragments of the records and fold P into fp32
//               sums held in registers.
// Work split: the T*G/2 (tile, stage) units are cut into equal contiguous
// ranges, one per CTA (stream-K).  A tile whose groups span several CTAs is
// finished by the last of them to arrive, adding the partial sums in
// increasing CTA order.  Nothing depends on M except how many n8 tiles run,
// and n8 tile 0 is computed identically for every M, so each row's result is
// independent of M and of the other rows.
// Programmatic dependent launch: the kernel lets the next kernel on the stream
// start at once; the weight stream needs nothing from the preceding kernel.
// Everything that touches x, y or the split-K scratch waits for the preceding
// kernel first (griddepcontrol.wait).
#pragma once

#include <cuda.h>
#include <cstdint>

#include "q4_sm100.cuh"

namespace q4 {
namespace rk {

constexpr int kThreads = 512;
constexpr int kCW = 15;                           // consumer warps
constexpr int kRowsW = 32;                        // rows per consumer warp
constexpr int kRowsTile = kCW * kRowsW;           // 480
constexpr int kBoxRows = 120;
constexpr int kBoxes = kRowsTile / kBoxRows;      // 4
constexpr int kStages = 6;
constexpr int kRec = 2112;                        // x record of one group: 2048 B of fragments + 16 fp32 sums
constexpr int kNibStage = kRowsTile * 64;         // 30720 B: 480 rows x 64 B (two groups)
constexpr int kStageBytes = ((kNibStage + 2 * kRec + 1023) / 1024) * 1024;
constexpr int kScratchBytes = kCW * kRowsW * 2 * 16;   // per-warp constants (s*2^33, r, cc, -)
constexpr int kBarrierBytes = 256;
constexpr int kSmemBytes = kStages * kStageBytes + kScratchBytes + kBarrierBytes + 1024 /* alignment */;
static_assert(kSmemBytes <= 232448, "shared memory per block exceeds the sm_103a limit");
constexpr long long kWaitLimit = 2000000000LL;   // cycles (about one second)
constexpr float kFoldScale = 8589934592.0f;      // 2^33: undoes 2^-133 (weights) * 2^100 (x)
constexpr uint32_t kXScaleEven = 0x71807180u;    // bf16 pair (2^100, 2^100)
constexpr uint32_t kXScaleOdd = 0x6F806F80u;     // bf16 pair (2^96, 2^96)

struct Params {
    const uint8_t* W;           // packed weights
    const uint16_t* x;          // bf16 [M, K]
    float* y;                   // [M, N]
    float* partials;            // scratch: [C][2][16][480]
    int* sems;                  // scratch: [C], zero between launches
    unsigned int* error_word;   // set on a timed-out wait
    int64_t N;
    int64_t K;
    int M;
    int G;                      // K / 64 (a multiple of 8)
    int T;                      // tiles of 480 rows
    int U;                      // T * G / 2 units (stages)
    int C;                      // CTAs (grid size)
#ifdef Q4_TRACE
    unsigned long long* trace;  // developer timing trace of CTA 0 (compiled in only with Q4_TRACE)
#endif
};

#ifdef Q4_TRACE
__device__ __forceinline__ unsigned long long q4_globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
#define Q4_GTR(p, idx)                                                  \
    do {                                                                \
        if ((p).trace && (idx) < 4096) (p).trace[(idx)] = q4_globaltimer(); \
    } while (0)
#define Q4_RTR(p, idx)                                                                                          \
    do {                                                                                                        \
        if ((p).trace && blockIdx.x == (unsigned)(p).trace[4095] && (idx) < 4095) (p).trace[(idx)] = clock64(); \
    } while (0)
#else
#define Q4_RTR(p, idx) \
    do {               \
    } while (0)
#define Q4_GTR(p, idx) \
    do {               \
    } while (0)
#endif

__device__ __forceinline__ int range_start(int U, int C, int c) { return (int)(((int64_t)U * c) / C); }

__device__ __forceinline__ int cta_of_unit(int U, int C, int u) {
    int c = (int)(((int64_t)u * C) / U);
    while (c + 1 < C && range_start(U, C, c + 1) <= u) ++c;
    while (c > 0 && range_start(U, C, c) > u) --c;
    return c;
}

__device__ __forceinline__ void record_timeout(const Params& p, unsigned int code, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(p.error_word, code);
}

__device__ __forceinline__ bool wait_or_abort(const Params& p, uint64_t* bar, uint32_t parity, unsigned code,
                                              volatile int* abort_flag) {
    if (q4::sm100::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (q4::sm100::mbar_wait(bar, parity, kWaitLimit)) return true;
    record_timeout(p, code, abort_flag);
    return false;
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

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 16 nibbles of one row (two words: inputs 16*tig .. 16*tig+15 of the group)
// into 8 bf16 pairs (q - c) * 2^-133 / 2^-129, pair kk = inputs (kk, kk+4) and
// pair 4+kk = inputs (8+kk, 12+kk), relative to 16*tig.
__device__ __forceinline__ void dequant16(uint32_t v0, uint32_t v1, uint32_t cc0, uint32_t (&A)[8]) {
    const uint32_t cc1 = cc0 << 4;
    const uint32_t u0 = v0 >> 8, u1 = v1 >> 8;
    A[0] = bf16x2_sub(and32(v0, 0x000F000Fu), cc0);
    A[1] = bf16x2_sub(and32(v0, 0x00F000F0u), cc1);
    A[2] = bf16x2_sub(and32(u0, 0x000F000Fu), cc0);
    A[3] = bf16x2_sub(and32(u0, 0x00F000F0u), cc1);
    A[4] = bf16x2_sub(and32(v1, 0x000F000Fu), cc0);
    A[5] = bf16x2_sub(and32(v1, 0x00F000F0u), cc1);
    A[6] = bf16x2_sub(and32(u1, 0x000F000Fu), cc0);
    A[7] = bf16x2_sub(and32(u1, 0x00F000F0u), cc1);
}

// Constants of one row and group from its bf16 scale and bias (low 16 bits of
// the arguments): s * 2^33, r = b + c*s and the bf16 pair c * 2^-133, with
// c = clamp(rint(-b/s), 0, 15) (NaN -> 0).
__device__ __forceinline__ float4 group_constants(uint32_t s_bits, uint32_t b_bits) {
    const float s = __uint_as_float(s_bits << 16);
    const float b = __uint_as_float(b_bits << 16);
    float cf = rintf(__fdividef(-b, s));
    cf = fminf(fmaxf(cf, 0.0f), 15.0f);
    const float r = __fmaf_rn(cf, s, b);
    // c as an integer: the low bits of 2^23 + c, copied into both halves
    const uint32_t cc = prmt(__float_as_uint(__fadd_rn(8388608.0f, cf)), 0u, 0x1010u) & 0x000F000Fu;
    return make_float4(s * kFoldScale, r, __uint_as_float(cc), 0.0f);
}

// One 8-input block (natural order, bf16) of row m of x into the four B
// fragment words it feeds -- pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7), the even
// k-steps scaled by 2^100 and the odd ones by 2^96 (exact) -- and the fp32 sum
// of the 8 unscaled inputs, added in increasing k.
__device__ __forceinline__ float x_block(const uint4& v, uint32_t (&o)[4]) {
    o[0] = bf16x2_mul(prmt(v.x, v.z, 0x5410u), kXScaleEven);    // (k0, k4)
    o[1] = bf16x2_mul(prmt(v.x, v.z, 0x7632u), kXScaleOdd);     // (k1, k5)
    o[2] = bf16x2_mul(prmt(v.y, v.w, 0x5410u), kXScaleEven);    // (k2, k6)
    o[3] = bf16x2_mul(prmt(v.y, v.w, 0x7632u), kXScaleOdd);     // (k3, k7)
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        s = __fadd_rn(s, __uint_as_float(w[i] << 16));
        s = __fadd_rn(s, __uint_as_float(w[i] & 0xFFFF0000u));
    }
    return s;
}

// Output element i (0..3) of n8 tile t for this lane: rows gid / gid+8 of the
// slab, columns 8t + 2tig / +1.
template <int NT>
__device__ void store_rows(const Params& p, const float (&acc)[2][NT][4], int t_tile, int wbase, int gid, int tig) {
#pragma unroll
    for (int sl = 0; sl < 2; ++sl)
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t n = (int64_t)t_tile * kRowsTile + wbase + 16 * sl + gid + 8 * (i >> 1);
                const int m = 8 * tt + 2 * tig + (i & 1);
                if (n < p.N && m < p.M) p.y[(int64_t)m * p.N + n] = acc[sl][tt][i];
            }
}

// Fixed-order finish of tile t, whose stages span CTAs [c_first, c_last]: the
// sum of their partials in increasing CTA order, stored as y.  Run by all
// consumer threads of the last CTA to arrive; each thread takes runs of 4 rows
// of one output column and keeps the loads of up to 4 CTAs in flight at once.
template <int NT>
__device__ __forceinline__ void finish_tile(const Params& p, int t, int ct, int c_first, int c_last) {
    constexpr int kRuns = kRowsTile / 4;                  // 120 runs of 4 rows per column
    for (int task = ct; task < 8 * NT * kRuns; task += kCW * 32) {
        const int m = task / kRuns, r4 = (task - m * kRuns) * 4;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = c_first; c0 <= c_last; c0 += 4) {
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = c0 + j;
                if (c <= c_last) {
                    const int cslot = (range_start(p.U, p.C, c) / (p.G >> 1) == t) ? 0 : 1;
                    v[j] = __ldcg(reinterpret_cast<const float4*>(p.partials + ((int64_t)c * 2 + cslot) * 16 * kRowsTile +
                                                                  m * kRowsTile + r4));
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c0 + j <= c_last) {
                    sum.x = __fadd_rn(sum.x, v[j].x);
                    sum.y = __fadd_rn(sum.y, v[j].y);
                    sum.z = __fadd_rn(sum.z, v[j].z);
                    sum.w = __fadd_rn(sum.w, v[j].w);
                }
        }
        if (m < p.M) {
            const int64_t n = (int64_t)t * kRowsTile + r4;
            float* yr = p.y + (int64_t)m * p.N;
            if (n + 0 < p.N) yr[n + 0] = sum.x;
            if (n + 1 < p.N) yr[n + 1] = sum.y;
            if (n + 2 < p.N) yr[n + 2] = sum.z;
            if (n + 3 < p.N) yr[n + 3] = sum.w;
        }
    }
}

// End of this CTA's segment of tile t (run by all consumer threads together):
// store the sums (whole tile), or publish them as a partial and let the last
// contributor add all partials of the tile in increasing CTA order.
template <int NT>
__device__ void end_segment(const Params& p, float (&acc)[2][NT][4], int t, bool whole, int slot, int wbase, int gid,
                            int tig, int ct, int c_id, int* bcast, bool live) {
    if (whole) {
        if (live) store_rows<NT>(p, acc, t, wbase, gid, tig);
    } else {
        float* part = p.partials + ((int64_t)c_id * 2 + slot) * 16 * kRowsTile;
        if (live) {
#pragma unroll
            for (int sl = 0; sl < 2; ++sl)
#pragma unroll
                for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = wbase + 16 * sl + gid + 8 * (i >> 1);
                        const int m = 8 * tt + 2 * tig + (i & 1);
                        __stcg(part + m * kRowsTile + row, acc[sl][tt][i]);
                    }
        }
        // every consumer's partial stores are ordered before the release of one
        // thread by the barrier; the last contributor's acquire publishes all
        // partials of the tile to its consumers after the second barrier
        Q4_RTR(p, threadIdx.x == 32 ? 3900 : 4094);
        named_barrier(1, kCW * 32);
        Q4_RTR(p, threadIdx.x == 32 ? 3901 : 4094);
        if (threadIdx.x == 32) {
            int last = 0;
            if (live) {
                const int Gh = p.G >> 1, tu = t * Gh;
                const int c_first = cta_of_unit(p.U, p.C, tu);
                const int c_last = cta_of_unit(p.U, p.C, tu + Gh - 1);
                int* sem = p.sems + c_first;
                int old;
                asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(sem) : "memory");
                if (old == c_last - c_first) {
                    asm volatile("st.relaxed.gpu.global.s32 [%0], 0;" ::"l"(sem) : "memory");   // zero for the next launch
                    last = 1;
                }
            }
            *bcast = last;
            Q4_RTR(p, 3902);
        }
        named_barrier(1, kCW * 32);
        Q4_RTR(p, threadIdx.x == 32 ? 3903 : 4094);
        if (*bcast) {
            const int Gh = p.G >> 1, tu = t * Gh;
            finish_tile<NT>(p, t, ct, cta_of_unit(p.U, p.C, tu), cta_of_unit(p.U, p.C, tu + Gh - 1));
        }
    }
#pragma unroll
    for (int sl = 0; sl < 2; ++sl)
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[sl][tt][i] = 0.0f;
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
q4_rk_kernel(const __grid_constant__ CUtensorMap map_nib, const Params p) {
    using namespace q4::sm100;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* scratch = smem + kStages * kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(scratch + kScratchBytes);   // nibbles landed, x records written
    uint64_t* empty = full + kStages;                                         // consumed by every consumer warp
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);
    int* bcast = const_cast<int*>(abort_flag) + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c_id = blockIdx.x;

    // the next kernel on the stream may start its own weight stream now
    pdl_launch_dependents();

    // This CTA's stages S0 .. S0+nst-1 (units are stages: stage S = groups 2k, 2k+1 of tile S / Gh).
    const int S0 = range_start(p.U, p.C, c_id);
    const int nst = range_start(p.U, p.C, c_id + 1) - S0;
    const int Gh = p.G >> 1;
    const int tS0 = S0 / Gh, kS0 = S0 - tS0 * Gh;      // tile and stage-in-tile of the first stage

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1 + kCW);           // the nibble boxes (with their bytes) + one per consumer warp
            mbar_init(&empty[s], kCW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) Q4_RTR(p, 4000);
    if (threadIdx.x == 0 && c_id < 300) Q4_GTR(p, 2000 + 3 * c_id);
#ifdef Q4_TRACE
    if (threadIdx.x == 0 && c_id < 300 && p.trace) {
        unsigned int smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        p.trace[2500 + 3 * c_id] = smid;
        p.trace[2501 + 3 * c_id] = nst;
        p.trace[2502 + 3 * c_id] = (unsigned long long)tS0 * 1000 + kS0;
    }
#endif

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&map_nib);
            const uint64_t pol = policy_evict_first();
            int tn = tS0, kn = kS0;                    // stage of the next nibble load
            auto issue_nibbles = [&](int slot) {
                uint8_t* sbase = smem + slot * kStageBytes;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)kNibStage);
                for (int b = 0; b < kBoxes; ++b)
                    tma_load_2d_hint(sbase + b * kBoxRows * 64, &map_nib, &full[slot], kn * 64,
                                     tn * kRowsTile + b * kBoxRows, pol);
                if (++kn == Gh) {
                    kn = 0;
                    ++tn;
                }
            };
            int slot = 0;
            uint32_t ph = 0;
            int si = 0;
            for (; si < nst; ++si) {
                if (si >= kStages && !wait_or_abort(p, &empty[slot], ph ^ 1u, 1u, abort_flag)) break;
                Q4_RTR(p, si);
                issue_nibbles(slot);
                if (++slot == kStages) {
                    slot = 0;
                    ph ^= 1u;
                }
            }
            // every issued copy must have landed before the CTA may exit
            for (int s2 = (si > kStages ? si - kStages : 0); s2 < si; ++s2)
                mbar_wait(&full[s2 % kStages], (s2 / kStages) & 1, kWaitLimit);
        }
        // (no griddepcontrol.wait in this warp: it would stall lane 0's weight stream behind the preceding kernel)
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - 1;                       // 0..14
        const int wbase = cw * kRowsW;                 // first tile row of this warp
        const int gid = lane >> 2, tig = lane & 3;
        const int ct = cw * 32 + lane;                 // 0..479 among the consumers
        const int t_first = S0 / Gh;
        float4* wscr = reinterpret_cast<float4*>(scratch + cw * kRowsW * 2 * 16);   // [32 rows][2 groups]
        [[maybe_unused]] const int tr = (threadIdx.x == 32) ? 1000 : 1 << 20;

        // scale and bias words of this lane's row: 16-byte blocks of 8 groups (four stages)
        const uint8_t* splane = p.W + p.N * (p.K / 2);
        const uint8_t* bplane = splane + p.N * p.G * 2;
        auto load_sb = [&](int t, int k, uint4& sv, uint4& bv) {   // block starting at stage-in-tile k of tile t
            const int64_t n = (int64_t)t * kRowsTile + wbase + lane;
            if (n < p.N) {
                const int64_t off = (n * p.G + 2 * k) * 2;
                sv = __ldg(reinterpret_cast<const uint4*>(splane + off));
                bv = __ldg(reinterpret_cast<const uint4*>(bplane + off));
            } else {
                sv = make_uint4(0, 0, 0, 0);
                bv = make_uint4(0, 0, 0, 0);
            }
        };
        uint4 cur_s, cur_b, nxt_s = make_uint4(0, 0, 0, 0), nxt_b = make_uint4(0, 0, 0, 0);
        int k_sb = kS0 - (kS0 & 3), t_sb = tS0;        // block of the next load
        int S_sb = S0 - (kS0 & 3);                     // its first stage
        auto sb_next = [&]() {
            k_sb += 4;
            if (k_sb >= Gh) {
                k_sb = 0;
                ++t_sb;
            }
            S_sb += 4;
        };
        load_sb(t_sb, k_sb, cur_s, cur_b);
        sb_next();
        if (S_sb < S0 + nst) load_sb(t_sb, k_sb, nxt_s, nxt_b);

        // x records: a stage's 256 16-byte blocks of x (group jj, row m, 8-block c) are
        // shared out over 256 consumer threads (the first 256 on even stages, the last
        // 256 on odd ones); each writes the four B fragment words of its block and the
        // rows' group sums, two stages ahead of their use
        auto x_task = [&](int st, int& jj, int& m, int& c) {
            const int ci = ct - ((st & 1) ? (kCW * 32 - 256) : 0);
            jj = ci >> 7;
            m = (ci >> 3) & 15;
            c = ci & 7;
            return ci >= 0 && ci < 256;                // uniform over each warp
        };
        auto x_load = [&](int st, int kx, uint4& v) {
            int jj, m, c;
            v = make_uint4(0, 0, 0, 0);
            if (x_task(st, jj, m, c) && m < p.M)
                v = __ldg(reinterpret_cast<const uint4*>(p.x + (int64_t)m * p.K + 128 * kx + 64 * jj + 8 * c));
        };
        auto x_write = [&](int st, int xslot, const uint4& v) {
            int jj, m, c;
            if (x_task(st, jj, m, c)) {
                uint32_t o[4];
                float s = x_block(v, o);
                // block c = inputs 16*tig + 8*h .. +7 of the group; word ((kk*2 + tt)*32 + lane)*2 + h
                const int tigc = c >> 1, h = c & 1, fl = (m & 7) * 4 + tigc, tt = m >> 3;
                uint32_t* rec = reinterpret_cast<uint32_t*>(smem + xslot * kStageBytes + kNibStage + jj * kRec);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) rec[((kk * 2 + tt) * 32 + fl) * 2 + h] = o[kk];
                // the 8 block sums of row m sit in 8 consecutive lanes: a fixed tree
                s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 1));
                s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 2));
                s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 4));
                if (c == 0) reinterpret_cast<float*>(rec + 512)[m] = s;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[xslot]);
        };

        pdl_wait();                                    // x, y and the split-K scratch belong to the preceding kernel until now
        if (ct == 0 && c_id < 300) Q4_GTR(p, 2001 + 3 * c_id);
        int kx = kS0;                                  // stage-in-tile of the next x load
        uint4 xv;
        for (int e = 0; e < 2 && e < nst; ++e) {
            x_load(e, kx, xv);
            x_write(e, e, xv);
            if (++kx == Gh) kx = 0;
        }
        if (nst > 2) {
            x_load(2, kx, xv);
            if (++kx == Gh) kx = 0;
        }
        int xslot = 2 % kStages;
        uint32_t xph = 0;                              // phase of the slot of stage si + 2

        float acc[2][NT][4];
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[sl][tt][i] = 0.0f;

        bool live = true;
        int slot = 0;
        uint32_t ph = 0;
        int kst = kS0, t = tS0;
        for (int si = 0; si < nst; ++si) {
            Q4_RTR(p, tr + 8 * si + 0);
            if (si > 0 && (kst & 3) == 0) {
                cur_s = nxt_s;
                cur_b = nxt_b;
                sb_next();
                if (S_sb < S0 + nst) load_sb(t_sb, k_sb, nxt_s, nxt_b);
            }
            // constants of this lane's row for both groups, shared through the warp's scratch
            {
                const int wsel = kst & 3;
                const uint32_t sw = wsel == 0 ? cur_s.x : wsel == 1 ? cur_s.y : wsel == 2 ? cur_s.z : cur_s.w;
                const uint32_t bw = wsel == 0 ? cur_b.x : wsel == 1 ? cur_b.y : wsel == 2 ? cur_b.z : cur_b.w;
                wscr[lane * 2 + 0] = group_constants(sw, bw);
                wscr[lane * 2 + 1] = group_constants(sw >> 16, bw >> 16);
            }
            live = __all_sync(0xFFFFFFFFu, live && wait_or_abort(p, &full[slot], ph, 8u, abort_flag));
            __syncwarp();
            Q4_RTR(p, tr + 8 * si + 1);
            const uint8_t* sbase = smem + slot * kStageBytes;
            if (live) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint8_t* rec = sbase + kNibStage + j * kRec;
                    uint2 bf[4][NT];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int tt = 0; tt < NT; ++tt)
                            bf[kk][tt] = *reinterpret_cast<const uint2*>(rec + ((kk * 2 + tt) * 32 + lane) * 8);
                    const float2 xa = *reinterpret_cast<const float2*>(rec + 2048 + 8 * tig);
                    const float2 xb = *reinterpret_cast<const float2*>(rec + 2048 + 32 + 8 * tig);
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        const int ra = 16 * sl + gid, rb = ra + 8;            // rows within the warp
                        const float4 ca = wscr[ra * 2 + j], cb = wscr[rb * 2 + j];
                        const int rowa = wbase + ra, rowb = wbase + rb;        // rows within the tile
                        const int chunk = 2 * j + (tig >> 1);
                        const uint2 na = *reinterpret_cast<const uint2*>(
                            sbase + rowa * 64 + ((chunk ^ ((rowa >> 1) & 3)) << 4) + 8 * (tig & 1));
                        const uint2 nbv = *reinterpret_cast<const uint2*>(
                            sbase + rowb * 64 + ((chunk ^ ((rowb >> 1) & 3)) << 4) + 8 * (tig & 1));
                        uint32_t A0[8], A1[8];
                        dequant16(na.x, na.y, __float_as_uint(ca.z), A0);
                        dequant16(nbv.x, nbv.y, __float_as_uint(cb.z), A1);
                        float P[NT][4];
#pragma unroll
                        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                            for (int i = 0; i < 4; ++i) P[tt][i] = 0.0f;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                            for (int tt = 0; tt < NT; ++tt)
                                mma16816(P[tt], A0[kk], A1[kk], A0[4 + kk], A1[4 + kk], bf[kk][tt].x, bf[kk][tt].y);
#pragma unroll
                        for (int tt = 0; tt < NT; ++tt) {
                            const float x0 = tt ? xb.x : xa.x, x1 = tt ? xb.y : xa.y;
                            acc[sl][tt][0] = __fmaf_rn(ca.x, P[tt][0], __fmaf_rn(ca.y, x0, acc[sl][tt][0]));
                            acc[sl][tt][1] = __fmaf_rn(ca.x, P[tt][1], __fmaf_rn(ca.y, x1, acc[sl][tt][1]));
                            acc[sl][tt][2] = __fmaf_rn(cb.x, P[tt][2], __fmaf_rn(cb.y, x0, acc[sl][tt][2]));
                            acc[sl][tt][3] = __fmaf_rn(cb.x, P[tt][3], __fmaf_rn(cb.y, x1, acc[sl][tt][3]));
                        }
                    }
                }
            }
            __syncwarp();
            Q4_RTR(p, tr + 8 * si + 2);
            if (lane == 0) mbar_arrive_relaxed(&empty[slot]);    // this warp's reads of the slot are consumed
            // the x records of the stage two ahead, into a slot every consumer warp has released
            if (si + 2 < nst) {
                if (si + 2 >= kStages) {
                    const bool fr = wait_or_abort(p, &empty[xslot], xph ^ 1u, 16u, abort_flag);
                    live = __all_sync(0xFFFFFFFFu, live && fr);
                }
                x_write(si + 2, xslot, xv);
                if (si + 3 < nst) {
                    x_load(si + 3, kx, xv);
                    if (++kx == Gh) kx = 0;
                }
                if (++xslot == kStages) {
                    xslot = 0;
                    xph ^= 1u;
                }
            }
            // a segment ends with the tile's last group or with this CTA's last unit
            if (kst == Gh - 1 || si == nst - 1) {
                const bool whole = (kst == Gh - 1) && t * Gh >= S0;
                end_segment<NT>(p, acc, t, whole, t == t_first ? 0 : 1, wbase, gid, tig, ct, c_id, bcast, !*abort_flag);
                Q4_RTR(p, tr + 8 * si + 3);
            }
            if (++slot == kStages) {
                slot = 0;
                ph ^= 1u;
            }
            if (++kst == Gh) {
                kst = 0;
                ++t;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) Q4_RTR(p, 4001);
    if (threadIdx.x == 0 && c_id < 300) Q4_GTR(p, 2002 + 3 * c_id);
}

inline int smem_bytes() { return kSmemBytes; }
inline size_t partial_floats(int C) { return (size_t)C * 2 * 16 * kRowsTile; }
inline size_t sem_ints(int C) { return (size_t)C; }

}  // namespace rk
}  // namespace q4
