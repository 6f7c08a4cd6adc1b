// Two-launch tensor-memory Q4 verify-matmul kernel for sm_103a (K a multiple
// of 512), used by q4_matmul_noalloc on its fixed scratch array.
//
// y[m,n] = sum_g ( s[n,g] * P[m,n,g] + r[n,g] * X[m,g] )
//   P[m,n,g] = sum_{k in g} (q[n,k] - c[n,g]) * x[m,k]      (tensor core, exact products)
//   X[m,g]   = sum_{k in g} x[m,k]                           (prepared once per call)
//   c[n,g]   = clamp(rint(-b/s), 0, 15),  r[n,g] = b + c*s
// which is w = s*q + b = s*(q - c) + r regrouped.  q - c is an exact small
// integer in bf16, and |r| <= s/2 whenever -b/s lies in [0,15], so s*P and r*X
// never cancel catastrophically: the error stays a small multiple of the fp32
// unit roundoff times sum_k |x_k w_k|, and an all-zero weight row (q == c,
// b == -c*s) gives exactly zero.
//
// One persistent CTA per SM, 16 warps.  A stage is an aligned pair of groups
// (inputs 128k .. 128k+127) of one 384-row tile.
//   warp 0      TMA producer: per stage three 128-row x 64-byte nibble boxes
//               (64-byte swizzle) and one bulk copy of the two groups'
//               prepared x records.
//   warps 1..3  MMA issuers, one per consumer group: per stage 8 MMAs
//               M128 N16 K16 (A = dequantized weights in tensor memory,
//               B = x from shared memory, D = P in tensor memory).
//   warps 4..15 three consumer groups of 4 warps; consumer group cg owns rows
//               128*cg .. 128*cg+127 of the tile, one row per thread.  Per
//               stage: dequantize 2 x 64 nibbles into (q - c) bf16 pairs and
//               store them to tensor memory, then fold the previous stage's P
//               into the fp32 sums with s and r, then hand the new A over.
// Work split: the T*G (tile, group) units are cut into equal contiguous
// ranges, one per CTA (stream-K).  A tile whose groups span several CTAs is
// finished by the last of them to arrive, which adds the partial sums in
// increasing CTA order; the split depends only on N, K and the grid size, so
// the result of every row is independent of M and of the other rows.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "q4_prep.cuh"
#include "q4_sm100.cuh"

namespace q4 {
namespace tc {

constexpr int kCG = 3;                      // consumer groups
constexpr int kRowsCG = 128;                // rows per consumer group (tensor-memory lanes)
constexpr int kRowsTile = kCG * kRowsCG;    // 384 rows per tile
constexpr int kStages = 7;
constexpr int kThreads = 512;
constexpr int kConsumerWarp0 = 4;
constexpr int kConsumerWarps = kCG * 4;
constexpr int kRegsControl = 80;
constexpr int kRegsConsumer = 144;
static_assert(128 * kRegsControl + 384 * kRegsConsumer <= kThreads * 128, "register split exceeds the launch");

constexpr int kRec = q4::prep::kRecordBytes;          // 2112 B of prepared x per group
constexpr int kNibBox = kRowsCG * 64;                 // 8 KB: 128 rows x 64 B (two groups)
constexpr int kNibStage = kCG * kNibBox;              // 24 KB
constexpr int kStageBytes = ((kNibStage + 2 * kRec + 1023) / 1024) * 1024;
constexpr int kBarrierBytes = 1024;
constexpr int kSmemBytes = kStages * kStageBytes + kBarrierBytes + 1024 /* alignment slack */;

// tensor-memory columns: A [cg][buffer 0/1][group 0/1] x 32, P [cg][group 0/1] x 16
constexpr uint32_t kColA = 0;
constexpr uint32_t kColP = kColA + kCG * 2 * 2 * 32;
constexpr uint32_t kTmemCols = 512;
static_assert(kColP + kCG * 2 * 16 <= kTmemCols, "tensor memory over-subscribed");

constexpr long long kWaitLimit = 2000000000LL;   // cycles (about one second)

struct Params {
    const uint8_t* W;           // packed weights (scales/biases read directly)
    const uint8_t* xt;          // prepared x records, [G][2112]
    float* y;                   // [M, N]
    float* partials;            // scratch: [C][2][kCG][16][128]
    int* sems;                  // scratch: [C][kCG], zero between launches
    unsigned int* error_word;   // set on a timed-out wait
    int64_t N;
    int64_t K;
    int M;
    int G;                      // K / 64 (a multiple of 8)
    int T;                      // tiles of 384 rows
    int U;                      // T * G units (groups of tiles)
    int C;                      // CTAs (grid size)
#ifdef Q4_TRACE
    unsigned long long* trace;  // developer timing trace of CTA 0 (compiled in only with Q4_TRACE)
#endif
};

#ifdef Q4_TRACE
#define Q4_TR(p, idx)                                                                     \
    do {                                                                                  \
        if ((p).trace && blockIdx.x == 0 && (idx) < 4096) (p).trace[(idx)] = clock64(); \
    } while (0)
#else
#define Q4_TR(p, idx) \
    do {              \
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

// (128 + q) as a bf16 pair for the nibbles in bits 0-3 and 16-19 of v.
__device__ __forceinline__ uint32_t nib_pair(uint32_t v) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "r"(0x000F000Fu), "r"(0x43004300u));   // (a & b) | c
    return d;
}

// acc0/acc1 = fma(a, b0/b1, acc0/acc1), one packed instruction (each lane an
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

// Fixed-order finish of one 128-row slice of a tile whose groups span CTAs
// [c_first, c_last]; run by the 128 threads of one consumer group of the last
// CTA to arrive.
template <int MT>
__device__ void finish_shared_slice(const Params& p, int t, int cg, int row, int c_first, int c_last) {
    const int64_t n = (int64_t)t * kRowsTile + cg * kRowsCG + row;
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
    for (int c = c_first; c <= c_last; ++c) {
        const int cs = range_start(p.U, p.C, c);
        const int slot = (cs / p.G == t) ? 0 : 1;      // the tile is c's first segment, or its last
        const float* src = p.partials + ((((int64_t)c * 2 + slot) * kCG + cg) * 16) * kRowsCG + row;
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = __fadd_rn(acc[m], __ldcg(src + m * kRowsCG));
    }
    if (n < p.N) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (m < p.M) p.y[(int64_t)m * p.N + n] = acc[m];
    }
}

// End of this CTA's segment of tile t for one consumer group: store the sums
// (whole tile), or publish them as a partial and let the last contributor add
// all partials of the tile slice in increasing CTA order.
template <int MT>
__device__ void end_segment(const Params& p, float (&acc)[MT], int t, bool whole, int slot, int cg, int row,
                            int cg_tid, int c_id, int* bcast, bool live) {
    const int64_t n = (int64_t)t * kRowsTile + cg * kRowsCG + row;
    if (whole) {
        if (live && n < p.N) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < p.M) p.y[(int64_t)m * p.N + n] = acc[m];
        }
    } else {
        float* dst = p.partials + ((((int64_t)c_id * 2 + slot) * kCG + cg) * 16) * kRowsCG + row;
        if (live) {
#pragma unroll
            for (int m = 0; m < MT; ++m) __stcg(dst + m * kRowsCG, acc[m]);
        }
        // the consumer group's partial stores are ordered before thread 0's
        // release by the barrier; the last contributor's acquire makes every
        // partial of the slice visible to its group after the second barrier
        named_barrier(1 + cg, kRowsCG);
        if (cg_tid == 0) {
            int last = 0;
            if (live) {
                const int tu = t * p.G;
                const int c_first = cta_of_unit(p.U, p.C, tu);
                const int c_last = cta_of_unit(p.U, p.C, tu + p.G - 1);
                int* sem = p.sems + c_first * kCG + cg;
                int old;
                asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(sem) : "memory");
                if (old == c_last - c_first) {
                    asm volatile("st.relaxed.gpu.global.s32 [%0], 0;" ::"l"(sem) : "memory");   // zero for the next launch
                    last = 1;
                }
            }
            bcast[cg] = last;
        }
        named_barrier(1 + cg, kRowsCG);
        if (bcast[cg]) {
            const int tu = t * p.G;
            finish_shared_slice<MT>(p, t, cg, row, cta_of_unit(p.U, p.C, tu), cta_of_unit(p.U, p.C, tu + p.G - 1));
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
}

// Dequantize the 64 nibbles of one row and group (two 16-byte chunks) into
// 32 bf16 pairs (q - c), word order (k0,k4) (k1,k5) (k2,k6) (k3,k7) per 8 inputs.
__device__ __forceinline__ void dequant64(const uint4& n0, const uint4& n1, uint32_t cc, uint32_t (&a)[32]) {
    const uint32_t wv[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
        const uint32_t v = wv[wi];
        a[4 * wi + 0] = bf16x2_sub(nib_pair(v), cc);
        a[4 * wi + 1] = bf16x2_sub(nib_pair(v >> 4), cc);
        a[4 * wi + 2] = bf16x2_sub(nib_pair(v >> 8), cc);
        a[4 * wi + 3] = bf16x2_sub(nib_pair(v >> 12), cc);
    }
}

// r = b + c*s and the bf16 pair (128 + c) of one group, c = clamp(rint(-b/s), 0, 15).
__device__ __forceinline__ void group_constants(float s, float b, float& r, uint32_t& cc) {
    float cf = rintf(__fdividef(-b, s));
    cf = fminf(fmaxf(cf, 0.0f), 15.0f);            // NaN -> 0
    r = __fmaf_rn(cf, s, b);
    // 128 + c is exact in bf16: its bits are the upper half of the fp32 value
    uint32_t f = __float_as_uint(__fadd_rn(128.0f, cf));
    asm("prmt.b32 %0, %1, %1, 0x3232;" : "=r"(cc) : "r"(f));
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
q4_tc_kernel(const __grid_constant__ CUtensorMap map_nib, const Params p) {
    using namespace q4::sm100;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);   // weights landed
    uint64_t* full_x = full + kStages;                 // prepared x landed
    uint64_t* empty = full_x + kStages;
    uint64_t* ready = empty + kStages;                 // [kCG][2]: A of group j of the stage stored
    uint64_t* done = ready + 2 * kCG;                  // [kCG][2]: MMAs of group j of the stage complete
    uint64_t* fin = done + 2 * kCG;                    // [kCG]
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(fin + kCG);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);
    int* bcast = const_cast<int*>(abort_flag) + 1;     // [kCG]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c_id = blockIdx.x;

    // the next kernel on the stream may start its own set-up now
    q4::prep::pdl_launch_dependents();

    // This CTA's groups [u0, u1) and stages S0 .. S0+nst-1 (stage S = groups 2S, 2S+1).
    const int u0 = range_start(p.U, p.C, c_id);
    const int u1 = range_start(p.U, p.C, c_id + 1);
    const int S0 = u0 >> 1;
    const int nst = ((u1 - 1) >> 1) - S0 + 1;
    const int Gh = p.G >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&full_x[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        for (int i = 0; i < 2 * kCG; ++i) {
            mbar_init(&ready[i], kRowsCG);
            mbar_init(&done[i], 1);
        }
        for (int i = 0; i < kCG; ++i) mbar_init(&fin[i], 1);
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
    if (threadIdx.x == 0) Q4_TR(p, 4000);

    // Register split: the producer/issuer warpgroup needs few registers, the
    // three consumer warpgroups many (128*80 + 384*144 = 512*128 at launch).
    if (warp < kConsumerWarp0)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    else
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsConsumer));

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            bool x_ready = false;
            int early_n = 0;             // first stages: weights issued before the prepared x exists
            auto issue_x = [&](int si, int k) {
                // records of groups 2k, 2k+1 (record index = group within K)
                mbar_arrive_expect_tx(&full_x[si % kStages], (uint32_t)(2 * kRec));
                bulk_copy_g2s(smem + (si % kStages) * kStageBytes + kNibStage, p.xt + (int64_t)(2 * k) * kRec,
                              (uint32_t)(2 * kRec), &full_x[si % kStages]);
            };
            int t = S0 / Gh, k = S0 - (S0 / Gh) * Gh;
            int te = t, ke = k;          // stage of the first pending x copy
            int si = 0;
            for (; si < nst; ++si) {
                const int slot = si % kStages;
                if (si >= kStages && !wait_or_abort(p, &empty[slot], ((si / kStages) - 1) & 1, 1u, abort_flag)) break;
                Q4_TR(p, 2 * si);
                uint8_t* sbase = smem + slot * kStageBytes;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)kNibStage);
                for (int cg = 0; cg < kCG; ++cg)
                    tma_load_2d_hint(sbase + cg * kNibBox, &map_nib, &full[slot], k * 64, t * kRowsTile + cg * kRowsCG,
                                     pol);
                if (!x_ready && (si + 1 == kStages || si + 1 == nst)) {
                    q4::prep::pdl_wait();        // the prep kernel (the preceding grid) has finished
                    x_ready = true;
                    for (int e = 0; e < early_n; ++e) {
                        issue_x(e, ke);
                        if (++ke == Gh) { ke = 0; ++te; }
                    }
                }
                if (x_ready)
                    issue_x(si, k);
                else
                    ++early_n;
                if (++k == Gh) { k = 0; ++t; }
            }
            if (!x_ready) {                      // aborted early: complete what was started
                q4::prep::pdl_wait();
                for (int e = 0; e < early_n; ++e) {
                    issue_x(e, ke);
                    if (++ke == Gh) { ke = 0; ++te; }
                }
            }
            // every issued stage must have landed before the CTA may exit
            for (int s2 = (si > kStages ? si - kStages : 0); s2 < si; ++s2) {
                mbar_wait(&full[s2 % kStages], (s2 / kStages) & 1, kWaitLimit);
                mbar_wait(&full_x[s2 % kStages], (s2 / kStages) & 1, kWaitLimit);
            }
        }
    } else if (warp <= kCG) {
        // ------------------------------------------------------------ MMA issuers
        const int cg = warp - 1;
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, 16);
            bool ok = true;
            for (int si = 0; si < nst && ok; ++si) {
                const int S = S0 + si;
                const int slot = si % kStages;
                const uint32_t xs = smem_u32(smem + slot * kStageBytes + kNibStage);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    if (!wait_or_abort(p, &ready[cg * 2 + jj], si & 1, 2u, abort_flag) ||
                        (jj == 0 && !wait_or_abort(p, &full_x[slot], (si / kStages) & 1, 2u, abort_flag))) {
                        ok = false;
                        break;
                    }
                    Q4_TR(p, 200 + 200 * cg + 4 * si + jj);
                    tc_fence_after();
                    const int u = 2 * S + jj;
                    if (u >= u0 && u < u1) {
                        const uint32_t dP = tmem + kColP + (uint32_t)((cg * 2 + jj) * 16);
                        const uint32_t aA = tmem + kColA + (uint32_t)(((cg * 2 + (si & 1)) * 2 + jj) * 32);
                        const uint32_t bx = xs + (uint32_t)(jj * kRec);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_ts(dP, aA + 8 * kk, smem_desc_noswizzle(bx + kk * 512, 256, 128), idesc, kk > 0);
                    }
                    tc_commit(&done[cg * 2 + jj]);
                    Q4_TR(p, 202 + 200 * cg + 4 * si + jj);
                }
            }
            // no MMA of this thread may still run when tensor memory is freed
            tc_commit(&fin[cg]);
            mbar_wait(&fin[cg], 0, kWaitLimit);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - kConsumerWarp0;          // 0..11
        const int cg = cw >> 2;
        const int q = warp & 3;                        // tensor-memory lane quarter of this warp
        const int row = q * 32 + lane;                 // row within the consumer group's 128
        const int cg_tid = (cw & 3) * 32 + lane;       // 0..127 within the consumer group
        const uint32_t lane_field = (uint32_t)(q * 32) << 16;
        const int t_first = u0 / p.G;
        [[maybe_unused]] const int tr = (lane == 0 && (cw & 3) == 0) ? 1000 + 1000 * cg : 1 << 20;

        // scale and bias words of a stage: the 2 bf16 of groups 2k, 2k+1 of this thread's row
        const uint32_t* scales = reinterpret_cast<const uint32_t*>(p.W + p.N * (p.K / 2));
        const uint32_t* biases = scales + p.N * (int64_t)(p.G / 2);
        int t_pf = S0 / Gh, k_pf = S0 - (S0 / Gh) * Gh;   // stage of the next prefetch
        auto fetch_sb = [&](uint32_t& sw, uint32_t& bw) {
            const int64_t n = (int64_t)t_pf * kRowsTile + cg * kRowsCG + row;
            if (n < p.N) {
                sw = __ldg(scales + n * Gh + k_pf);
                bw = __ldg(biases + n * Gh + k_pf);
            } else {
                sw = 0u;
                bw = 0u;
            }
            if (++k_pf == Gh) { k_pf = 0; ++t_pf; }
        };
        // three stages of scale/bias words in flight (weights do not depend on the preceding grid)
        uint32_t sw0 = 0, bw0 = 0, sw1 = 0, bw1 = 0, sw2 = 0, bw2 = 0;
        if (nst > 0) fetch_sb(sw0, bw0);
        if (nst > 1) fetch_sb(sw1, bw1);
        if (nst > 2) fetch_sb(sw2, bw2);

        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

        bool live = true;
        bool pdl_done = false;
        // the previous stage's groups, each folded just before its P buffer is reused
        float ps[2] = {0.f, 0.f}, pr[2] = {0.f, 0.f};
        int pv = 0;            // bit 0: group 0 valid, bit 1: group 1 valid, bit 2: ends a segment, bit 3: whole tile
        int pt = 0, pslot = 0;

        // fold group jj of the previous stage (si_prev): wait for its MMAs, read P, add s*P + r*X
        auto fold_group = [&](int si_prev, int jj) {
            const bool w = __all_sync(0xFFFFFFFFu, live && wait_or_abort(p, &done[cg * 2 + jj], si_prev & 1, 4u,
                                                                          abort_flag));
            if (w && (pv & (1 << jj))) {
                tc_fence_after();
                uint32_t P[16];
                tmem_ld_32x32b_x16(tmem + lane_field + kColP + (uint32_t)((cg * 2 + jj) * 16), P);
                const uint8_t* xsum = smem + pslot * kStageBytes + kNibStage + jj * kRec + 2048;
                float X[16];
#pragma unroll
                for (int v4 = 0; v4 < (MT + 3) / 4; ++v4) {
                    const float4 v = *reinterpret_cast<const float4*>(xsum + 16 * v4);
                    X[4 * v4 + 0] = v.x;
                    X[4 * v4 + 1] = v.y;
                    X[4 * v4 + 2] = v.z;
                    X[4 * v4 + 3] = v.w;
                }
                tmem_wait_ld();
                const float s = ps[jj], r = pr[jj];
                if (MT == 1) {
                    acc[0] = __fmaf_rn(s, __uint_as_float(P[0]), acc[0]);
                    acc[0] = __fmaf_rn(r, X[0], acc[0]);
                } else {
#pragma unroll
                    for (int m = 0; m + 1 < MT; m += 2) {
                        fma2(acc[m], acc[m + 1], s, __uint_as_float(P[m]), __uint_as_float(P[m + 1]));
                        fma2(acc[m], acc[m + 1], r, X[m], X[m + 1]);
                    }
                }
            }
        };
        // after both groups of the previous stage are folded: release its ring slot, close its segment
        auto close_stage = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(&empty[pslot]);   // the slot's reads are consumed
            if (pv & 4) {
                if (!pdl_done) {
                    // partial sums and y may be touched only after the preceding grid finished
                    q4::prep::pdl_wait();
                    pdl_done = true;
                }
                end_segment<MT>(p, acc, pt, (pv & 8) != 0, pt == t_first ? 0 : 1, cg, row, cg_tid, c_id, bcast,
                                !*abort_flag);
            }
        };

        int t = S0 / Gh, k = S0 - (S0 / Gh) * Gh;
        for (int si = 0; si < nst; ++si) {
            const int S = S0 + si;
            const int slot = si % kStages;
            Q4_TR(p, tr + 8 * si + 0);
            const bool have = wait_or_abort(p, &full[slot], (si / kStages) & 1, 8u, abort_flag);
            live = __all_sync(0xFFFFFFFFu, live && have);
            const int cur_v = (2 * S >= u0 ? 1 : 0) | (2 * S + 1 < u1 ? 2 : 0);
            float s01[2], r01[2];
            s01[0] = __uint_as_float(sw0 << 16);
            s01[1] = __uint_as_float(sw0 & 0xFFFF0000u);
            const float b0 = __uint_as_float(bw0 << 16), b1 = __uint_as_float(bw0 & 0xFFFF0000u);
            // rotate the scale/bias words; fetch three stages ahead
            sw0 = sw1; bw0 = bw1; sw1 = sw2; bw1 = bw2;
            if (si + 3 < nst) fetch_sb(sw2, bw2);
            const uint8_t* nb = smem + slot * kStageBytes + cg * kNibBox + row * 64;
            const int sx = (row >> 1) & 3;
            const uint32_t abase = tmem + lane_field + kColA + (uint32_t)((cg * 2 + (si & 1)) * 2 * 32);
            // both groups' constants and nibbles, dequantized together (64 independent chains)
            uint32_t cc0, cc1;
            group_constants(s01[0], b0, r01[0], cc0);
            group_constants(s01[1], b1, r01[1], cc1);
            Q4_TR(p, tr + 8 * si + 1);
            if (live) {
                uint32_t a0[32], a1[32];
                const uint4 n0 = *reinterpret_cast<const uint4*>(nb + ((0 ^ sx) << 4));
                const uint4 n1 = *reinterpret_cast<const uint4*>(nb + ((1 ^ sx) << 4));
                const uint4 n2 = *reinterpret_cast<const uint4*>(nb + ((2 ^ sx) << 4));
                const uint4 n3 = *reinterpret_cast<const uint4*>(nb + ((3 ^ sx) << 4));
                dequant64(n0, n1, cc0, a0);
                dequant64(n2, n3, cc1, a1);
                tmem_st_32x32b_x32(abase, a0);
                tmem_st_32x32b_x32(abase + 32, a1);
            }
            Q4_TR(p, tr + 8 * si + 2);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                // group jj of the previous stage, before its P buffer is reused
                if (si > 0) fold_group(si - 1, jj);
                Q4_TR(p, tr + 8 * si + 3 + jj);
                if (live) {
                    if (jj == 0) tmem_wait_st();     // A is in tensor memory
                    tc_fence_before();
                    mbar_arrive_relaxed(&ready[cg * 2 + jj]);
                }
            }
            if (si > 0) close_stage();
            ps[0] = s01[0];
            ps[1] = s01[1];
            pr[0] = r01[0];
            pr[1] = r01[1];
            pv = cur_v;
            if (k == Gh - 1 || si == nst - 1) pv |= 4;                         // the segment ends with this stage
            if (k == Gh - 1 && (t > t_first || u0 == t_first * p.G)) pv |= 8;   // ... and spans the whole tile
            pt = t;
            pslot = slot;
            if (++k == Gh) { k = 0; ++t; }
        }
        if (nst > 0) {
            fold_group(nst - 1, 0);
            fold_group(nst - 1, 1);
            close_stage();
        }
        if (!pdl_done) q4::prep::pdl_wait();
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) Q4_TR(p, 4001);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

inline int smem_bytes() { return kSmemBytes; }
inline size_t partial_floats(int C) { return (size_t)C * 2 * kCG * 16 * kRowsCG; }
inline size_t sem_ints(int C) { return (size_t)C * kCG; }

}  // namespace tc
}  // namespace q4
