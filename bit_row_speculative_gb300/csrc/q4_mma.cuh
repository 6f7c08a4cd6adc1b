// Register-operand Q4 verify-matmul kernel for sm_103a (K a multiple of 512).
//
// y[m,n] = sum_g ( s[n,g] * P[m,n,g] + r[n,g] * X[m,g] )
//   P[m,n,g] = sum_{k in g} (q[n,k] - c[n,g]) * x[m,k]     (tensor core, exact products)
//   X[m,g]   = sum_{k in g} x[m,k]                          (prepared once per call)
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
// exactly, and the fold applies s * 2^33.  Tensor-core products of subnormal
// bf16 operands are exact on this GPU (checked by the tests).
//
// One persistent CTA per SM, 16 warps, tiles of 480 rows; a stage is an
// aligned pair of groups (inputs 128k .. 128k+127) of one tile.
//   warp 0      TMA producer: four 120-row x 64-byte nibble boxes per stage
//               (64-byte swizzle) and one bulk copy of the two groups'
//               prepared x records.
//   warps 1..15 consumers, 32 rows each (two m16 slabs): per stage they derive
//               the groups' constants (one row per lane, shared through
//               shared memory), dequantize into mma.sync A fragments, run the
//               m16n8k16 MMAs against the prepared B fragments and fold P into
//               fp32 sums held in registers.
// Work split: stream-K over (tile, group) units, as in the tensor-memory
// kernel; a tile whose groups span several CTAs is finished by the last to
// arrive, adding the partial sums in increasing CTA order.  Nothing depends on
// M except how many n8 tiles run, and n8 tile 0 is computed identically for
// every M, so each row's result is independent of M and of the other rows.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "q4_prep.cuh"
#include "q4_sm100.cuh"

namespace q4 {
namespace rk {

constexpr int kThreads = 512;
constexpr int kCW = 15;                           // consumer warps
constexpr int kRowsW = 32;                        // rows per consumer warp
constexpr int kRowsTile = kCW * kRowsW;           // 480
constexpr int kBoxRows = 120;
constexpr int kBoxes = kRowsTile / kBoxRows;      // 4
constexpr int kStages = 5;
constexpr int kRec = q4::prep::kRecordBytes;      // 2112
constexpr int kNibStage = kRowsTile * 64;         // 30720 B: 480 rows x 64 B (two groups)
constexpr int kStageBytes = ((kNibStage + 2 * kRec + 1023) / 1024) * 1024;
constexpr int kScratchBytes = kCW * kRowsW * 2 * 16;   // per-warp constants (s*2^33, r, cc, -)
constexpr int kBarrierBytes = 512;
constexpr int kSmemBytes = kStages * kStageBytes + kScratchBytes + kBarrierBytes + 1024 /* alignment */;
constexpr long long kWaitLimit = 2000000000LL;   // cycles (about one second)
constexpr float kFoldScale = 8589934592.0f;      // 2^33: undoes 2^-133 (weights) * 2^100 (x)
static_assert(q4::prep::kFragScale == 100, "fold scale assumes x * 2^100");

struct Params {
    const uint8_t* W;           // packed weights (scales/biases read directly)
    const uint8_t* xt;          // prepared x records, [G][2112]
    float* y;                   // [M, N]
    float* partials;            // scratch: [C][2][16][480]
    int* sems;                  // scratch: [C], zero between launches
    unsigned int* error_word;   // set on a timed-out wait
    int64_t N;
    int64_t K;
    int M;
    int G;                      // K / 64 (a multiple of 8)
    int T;                      // tiles of 480 rows
    int U;                      // T * G units
    int C;                      // CTAs (grid size)
#ifdef Q4_TRACE
    unsigned long long* trace;  // developer timing trace of CTA 0 (compiled in only with Q4_TRACE)
#endif
};

#ifdef Q4_TRACE
#define Q4_RTR(p, idx)                                                                    \
    do {                                                                                  \
        if ((p).trace && blockIdx.x == 0 && (idx) < 4096) (p).trace[(idx)] = clock64(); \
    } while (0)
#else
#define Q4_RTR(p, idx) \
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

__device__ __forceinline__ uint32_t and32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, 0, 0xC0;" : "=r"(d) : "r"(a), "r"(b));
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

// End of this CTA's segment of tile t (run by all consumer threads together).
template <int NT>
__device__ void end_segment(const Params& p, float (&acc)[2][NT][4], int t, bool whole, int slot, int wbase, int gid,
                            int tig, int c_id, int* bcast, bool live) {
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
        named_barrier(1, kCW * 32);
        if (threadIdx.x == 32) {
            int last = 0;
            if (live) {
                const int tu = t * p.G;
                const int c_first = cta_of_unit(p.U, p.C, tu);
                const int c_last = cta_of_unit(p.U, p.C, tu + p.G - 1);
                int* sem = p.sems + c_first;
                int old;
                asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(sem) : "memory");
                if (old == c_last - c_first) {
                    asm volatile("st.relaxed.gpu.global.s32 [%0], 0;" ::"l"(sem) : "memory");
                    last = 1;
                }
            }
            *bcast = last;
        }
        named_barrier(1, kCW * 32);
        if (*bcast) {
            const int tu = t * p.G;
            const int c_first = cta_of_unit(p.U, p.C, tu), c_last = cta_of_unit(p.U, p.C, tu + p.G - 1);
            float sum[2][NT][4];
#pragma unroll
            for (int sl = 0; sl < 2; ++sl)
#pragma unroll
                for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) sum[sl][tt][i] = 0.0f;
            for (int c = c_first; c <= c_last; ++c) {
                const int cslot = (range_start(p.U, p.C, c) / p.G == t) ? 0 : 1;
                const float* src = p.partials + ((int64_t)c * 2 + cslot) * 16 * kRowsTile;
#pragma unroll
                for (int sl = 0; sl < 2; ++sl)
#pragma unroll
                    for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int row = wbase + 16 * sl + gid + 8 * (i >> 1);
                            const int m = 8 * tt + 2 * tig + (i & 1);
                            sum[sl][tt][i] = __fadd_rn(sum[sl][tt][i], __ldcg(src + m * kRowsTile + row));
                        }
            }
            store_rows<NT>(p, sum, t, wbase, gid, tig);
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
    uint64_t* full = reinterpret_cast<uint64_t*>(scratch + kScratchBytes);
    uint64_t* full_x = full + kStages;
    uint64_t* empty = full_x + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);
    int* bcast = const_cast<int*>(abort_flag) + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c_id = blockIdx.x;

    q4::prep::pdl_launch_dependents();

    const int u0 = range_start(p.U, p.C, c_id);
    const int u1 = range_start(p.U, p.C, c_id + 1);
    const int S0 = u0 >> 1;
    const int nst = ((u1 - 1) >> 1) - S0 + 1;
    const int Gh = p.G >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&full_x[s], 1);
            mbar_init(&empty[s], kCW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) Q4_RTR(p, 4000);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&map_nib);
            const uint64_t pol = policy_evict_first();
            bool x_ready = false;
            int early_n = 0;
            int t = S0 / Gh, k = S0 - (S0 / Gh) * Gh;
            int ke = k;
            auto issue_x = [&](int si, int kx) {
                mbar_arrive_expect_tx(&full_x[si % kStages], (uint32_t)(2 * kRec));
                bulk_copy_g2s(smem + (si % kStages) * kStageBytes + kNibStage, p.xt + (int64_t)(2 * kx) * kRec,
                              (uint32_t)(2 * kRec), &full_x[si % kStages]);
            };
            int si = 0;
            for (; si < nst; ++si) {
                const int slot = si % kStages;
                if (si >= kStages && !wait_or_abort(p, &empty[slot], ((si / kStages) - 1) & 1, 1u, abort_flag)) break;
                Q4_RTR(p, si);
                uint8_t* sbase = smem + slot * kStageBytes;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)kNibStage);
                for (int b = 0; b < kBoxes; ++b)
                    tma_load_2d_hint(sbase + b * kBoxRows * 64, &map_nib, &full[slot], k * 64,
                                     t * kRowsTile + b * kBoxRows, pol);
                if (!x_ready && (si + 1 == kStages || si + 1 == nst)) {
                    q4::prep::pdl_wait();        // the prep kernel (the preceding grid) has finished
                    Q4_RTR(p, 3999);
                    x_ready = true;
                    for (int e = 0; e < early_n; ++e) {
                        issue_x(e, ke);
                        if (++ke == Gh) ke = 0;
                    }
                }
                if (x_ready)
                    issue_x(si, k);
                else
                    ++early_n;
                if (++k == Gh) { k = 0; ++t; }
            }
            if (!x_ready) {
                q4::prep::pdl_wait();
                for (int e = 0; e < early_n; ++e) {
                    issue_x(e, ke);
                    if (++ke == Gh) ke = 0;
                }
            }
            for (int s2 = (si > kStages ? si - kStages : 0); s2 < si; ++s2) {
                mbar_wait(&full[s2 % kStages], (s2 / kStages) & 1, kWaitLimit);
                mbar_wait(&full_x[s2 % kStages], (s2 / kStages) & 1, kWaitLimit);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - 1;                       // 0..14
        const int wbase = cw * kRowsW;                 // first tile row of this warp
        const int gid = lane >> 2, tig = lane & 3;
        const int t_first = u0 / p.G;
        float4* wscr = reinterpret_cast<float4*>(scratch + cw * kRowsW * 2 * 16);   // [32 rows][2 groups]

        // scale/bias words (2 groups) of this lane's row, three stages ahead
        const uint32_t* scales = reinterpret_cast<const uint32_t*>(p.W + p.N * (p.K / 2));
        const uint32_t* biases = scales + p.N * (int64_t)Gh;
        int t_pf = S0 / Gh, k_pf = S0 - (S0 / Gh) * Gh;
        auto fetch_sb = [&](uint32_t& sw, uint32_t& bw) {
            const int64_t n = (int64_t)t_pf * kRowsTile + wbase + lane;
            if (n < p.N) {
                sw = __ldg(scales + n * Gh + k_pf);
                bw = __ldg(biases + n * Gh + k_pf);
            } else {
                sw = 0u;
                bw = 0u;
            }
            if (++k_pf == Gh) { k_pf = 0; ++t_pf; }
        };
        uint32_t sw0 = 0, bw0 = 0, sw1 = 0, bw1 = 0, sw2 = 0, bw2 = 0;
        if (nst > 0) fetch_sb(sw0, bw0);
        if (nst > 1) fetch_sb(sw1, bw1);
        if (nst > 2) fetch_sb(sw2, bw2);

        float acc[2][NT][4];
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[sl][tt][i] = 0.0f;

        bool live = true;
        bool pdl_done = false;
        int t = S0 / Gh, k = S0 - (S0 / Gh) * Gh;
        for (int si = 0; si < nst; ++si) {
            const int S = S0 + si;
            const int slot = si % kStages;
            const uint8_t* sbase = smem + slot * kStageBytes;
            [[maybe_unused]] const int tr = (threadIdx.x == 32) ? 1000 + 8 * si : 1 << 20;
            Q4_RTR(p, tr + 0);
            bool have = wait_or_abort(p, &full[slot], (si / kStages) & 1, 8u, abort_flag);
            Q4_RTR(p, tr + 1);
            have = have && wait_or_abort(p, &full_x[slot], (si / kStages) & 1, 8u, abort_flag);
            Q4_RTR(p, tr + 2);
            live = __all_sync(0xFFFFFFFFu, live && have);

            // constants of this lane's row for both groups (c, r, s * 2^33, the bf16 pair c * 2^-133)
            {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float s = __uint_as_float(j ? (sw0 & 0xFFFF0000u) : (sw0 << 16));
                    const float b = __uint_as_float(j ? (bw0 & 0xFFFF0000u) : (bw0 << 16));
                    float cf = rintf(__fdividef(-b, s));
                    cf = fminf(fmaxf(cf, 0.0f), 15.0f);            // NaN -> 0
                    const float r = __fmaf_rn(cf, s, b);
                    // c as an integer: the low bits of 2^23 + c
                    const uint32_t ci = __float_as_uint(__fadd_rn(8388608.0f, cf)) & 0xFu;
                    wscr[lane * 2 + j] = make_float4(s * kFoldScale, r, __uint_as_float(ci * 0x00010001u), 0.0f);
                }
            }
            sw0 = sw1; bw0 = bw1; sw1 = sw2; bw1 = bw2;
            if (si + 3 < nst) fetch_sb(sw2, bw2);
            __syncwarp();
            Q4_RTR(p, tr + 3);

            if (live) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int u = 2 * S + j;
                    if (u < u0 || u >= u1) continue;             // warp-uniform
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
                        const uint2 nb = *reinterpret_cast<const uint2*>(
                            sbase + rowb * 64 + ((chunk ^ ((rowb >> 1) & 3)) << 4) + 8 * (tig & 1));
                        uint32_t A0[8], A1[8];
                        dequant16(na.x, na.y, __float_as_uint(ca.z), A0);
                        dequant16(nb.x, nb.y, __float_as_uint(cb.z), A1);
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
            Q4_RTR(p, tr + 4);
            if (lane == 0) mbar_arrive_relaxed(&empty[slot]);    // this warp's reads of the slot are consumed
            if (k == Gh - 1 || si == nst - 1) {
                if (!pdl_done) {
                    q4::prep::pdl_wait();       // partial sums and y: only after the preceding grid finished
                    pdl_done = true;
                }
                const bool whole = (k == Gh - 1) && (t > t_first || u0 == t_first * p.G);
                end_segment<NT>(p, acc, t, whole, t == t_first ? 0 : 1, wbase, gid, tig, c_id, bcast,
                                !*abort_flag);
                Q4_RTR(p, tr + 5);
            }
            if (++k == Gh) { k = 0; ++t; }
        }
        if (!pdl_done) q4::prep::pdl_wait();
    }
    __syncthreads();
    if (threadIdx.x == 0) Q4_RTR(p, 4001);
}

inline int smem_bytes() { return kSmemBytes; }
inline size_t partial_floats(int C) { return (size_t)C * 2 * 16 * kRowsTile; }
inline size_t sem_ints(int C) { return (size_t)C; }

}  // namespace rk
}  // namespace q4
