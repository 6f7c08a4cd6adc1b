// Q4 verify-matmul kernel for sm_103a (K a multiple of 512): one launch per call.
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
// One persistent CTA per SM, 16 warps; tiles of 384 rows, a stage is an
// aligned pair of groups (inputs 128k .. 128k+127) of one tile.
//   x records   once per call, each group's x record -- the M <= 16 rows of x
//               for the group's 64 inputs in the tensor core's K-major
//               core-matrix layout (inputs of each 8-block in the dequantized
//               order k0 k4 k1 k5 k2 k6 k3 k7, scaled as above) and the group
//               sums X -- is written to global scratch by one CTA (group g by
//               CTA g mod C) and published with a per-launch epoch flag.  The
//               epoch lives in device memory and advances when the last CTA of
//               a launch finishes, so repeated launches (and graph replays)
//               never mistake an older record for the current one.
//   warp 0      producer: per stage three 128-row x 64-byte nibble boxes
//               (TMA, 64-byte swizzle) into a 7-stage ring, then, once each
//               group's flag shows the current epoch, a bulk copy of the
//               stage's two x records into the same slot.
//   warps 1..3  MMA issuers, one per consumer group: per stage 8 MMAs
//               M128 N16 K16 (A = dequantized weights in tensor memory, B = the
//               x records in shared memory, D = P in tensor memory).
//   warps 4..15 three consumer groups of 4 warps; consumer group cg owns rows
//               128*cg .. 128*cg+127 of the tile, one row per thread.  Per
//               stage they dequantize the 2 x 64 nibbles of their row and store
//               them to tensor memory (A double-buffered by stage), fold the
//               previous stage's P into fp32 sums with s, r and X, and then
//               hand the new A over (P has one buffer per group: the next MMAs
//               are issued only after the fold has read it).
// Work split: the T*G (tile, group) units are cut into equal contiguous
// ranges, one per CTA (stream-K).  A tile whose groups span several CTAs is
// finished by the last of them to arrive, which adds the partial sums in
// increasing CTA order.  The split depends only on N, K and the grid size, and
// nothing in the arithmetic of row m depends on the other rows, so every
// row's result is independent of M.
// Programmatic dependent launch: the kernel lets the next kernel on the stream
// start at once; the weight stream needs nothing from the preceding kernel.
// Everything that touches x, y, the records or the split-K scratch waits for
// the preceding kernel first (griddepcontrol.wait).  A CTA waits for another
// CTA of the same launch only for a record flag; all CTAs of a launch fit on
// the GPU at once, so such a wait ends unless other work holds the SMs, and it
// is bounded in any case.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "q4_sm100.cuh"

namespace q4 {
namespace tm {

constexpr int kCG = 3;                      // consumer groups
constexpr int kRowsCG = 128;                // rows per consumer group (tensor-memory lanes)
constexpr int kRowsTile = kCG * kRowsCG;    // 384 rows per tile
constexpr int kStages = 7;
constexpr int kThreads = 512;
constexpr int kConsumerWarp0 = 4;
constexpr int kConsumerWarps = kCG * 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kRegsControl = 56;
constexpr int kRegsConsumer = 152;
static_assert(128 * kRegsControl + kConsumerThreads * kRegsConsumer <= kThreads * 128,
              "register split exceeds the launch");

constexpr int kRec = 2112;                            // x record of one group: 2048 B operand + 16 fp32 sums
constexpr int kNibBox = kRowsCG * 64;                 // 8 KB: 128 rows x 64 B (two groups)
constexpr int kNibStage = kCG * kNibBox;              // 24 KB
constexpr int kStageBytes = ((kNibStage + 2 * kRec + 1023) / 1024) * 1024;
constexpr int kBarrierBytes = 1024;
constexpr int kSmemBytes = kStages * kStageBytes + kBarrierBytes + 1024 /* alignment slack */;

// tensor-memory columns: A [cg][stage parity][group] x 32, P [cg][group] x 16
constexpr uint32_t kColA = 0;
constexpr uint32_t kColP = kColA + kCG * 2 * 2 * 32;
constexpr uint32_t kTmemCols = 512;
static_assert(kColP + kCG * 2 * 16 <= kTmemCols, "tensor memory over-subscribed");

constexpr long long kWaitLimit = 2000000000LL;     // cycles (about one second)
constexpr float kFoldScale = 8589934592.0f;        // 2^33: undoes 2^-133 (weights) * 2^100 (x)
constexpr uint32_t kXScaleEven = 0x71807180u;      // bf16 pair (2^100, 2^100)
constexpr uint32_t kXScaleOdd = 0x6F806F80u;       // bf16 pair (2^96, 2^96)

struct Params {
    const uint8_t* W;           // packed weights
    const uint16_t* x;          // bf16 [M, K]
    float* y;                   // [M, N]
    float* partials;            // scratch: [C][2][kCG][16][128]
    int* sems;                  // scratch: [C][kCG], zero between launches
    uint8_t* xt;                // scratch: x records [G][2112]
    unsigned int* flags;        // scratch: [G] epoch of each group's record
    unsigned int* epoch;        // scratch: launches completed (advanced by the last CTA)
    unsigned int* finished;     // scratch: CTAs of the current launch that have finished
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
#define Q4_TMTR(p, idx)                                                                   \
    do {                                                                                  \
        if ((p).trace && blockIdx.x == 0 && (idx) < 4096) (p).trace[(idx)] = clock64(); \
    } while (0)
#else
#define Q4_TMTR(p, idx) \
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

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* ptr) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned int* ptr, unsigned int v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// Orders generic-proxy memory accesses with later async-proxy ones (TMA, bulk
// copies, the tensor core) in every state space.
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Bounded wait until the record flag of a group shows `target`.
__device__ __forceinline__ bool wait_flag(const Params& p, const unsigned int* flag, unsigned int target,
                                          volatile int* abort_flag) {
    if (ld_acquire_gpu(flag) == target) return true;
    const long long t0 = clock64();
    while (ld_acquire_gpu(flag) != target) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimit) {
            record_timeout(p, 32u, abort_flag);
            return false;
        }
        __nanosleep(256);
    }
    return true;
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

// One 8-input block of one row of x (natural order, bf16) into the tensor
// core's order (k0,k4) (k1,k5) (k2,k6) (k3,k7) with the even inputs scaled by
// 2^100 and the odd ones by 2^96 (exact); returns the fp32 sum of the 8
// unscaled inputs, added in increasing k.
__device__ __forceinline__ float x_block(const uint4& v, uint4& o) {
    o.x = bf16x2_mul(prmt(v.x, v.z, 0x5410u), kXScaleEven);    // (k0, k4)
    o.y = bf16x2_mul(prmt(v.x, v.z, 0x7632u), kXScaleOdd);     // (k1, k5)
    o.z = bf16x2_mul(prmt(v.y, v.w, 0x5410u), kXScaleEven);    // (k2, k6)
    o.w = bf16x2_mul(prmt(v.y, v.w, 0x7632u), kXScaleOdd);     // (k3, k7)
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        s = __fadd_rn(s, __uint_as_float(w[i] << 16));
        s = __fadd_rn(s, __uint_as_float(w[i] & 0xFFFF0000u));
    }
    return s;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
q4_tm_kernel(const __grid_constant__ CUtensorMap map_nib, const Params p) {
    using namespace q4::sm100;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);   // nibbles and x records landed
    uint64_t* empty = full + kStages;                  // stage consumed (nibbles, records, its folds): one arrival per issuer
    uint64_t* ready = empty + kStages;                 // [kCG]: A of a stage stored
    uint64_t* done = ready + kCG;                      // [kCG]: MMAs of a stage complete
    uint64_t* fin = done + kCG;                        // [kCG]
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(fin + kCG);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);
    int* bcast = const_cast<int*>(abort_flag) + 1;     // [kCG]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c_id = blockIdx.x;

    // the next kernel on the stream may start its own weight stream now
    pdl_launch_dependents();

    // This CTA's units [u0, u1) and stages S0 .. S0+nst-1 (stage S = units 2S, 2S+1).
    const int u0 = range_start(p.U, p.C, c_id);
    const int u1 = range_start(p.U, p.C, c_id + 1);
    const int S0 = u0 >> 1;
    const int nst = ((u1 - 1) >> 1) - S0 + 1;
    const int Gh = p.G >> 1;
    const int tS0 = S0 / Gh, kS0 = S0 - tS0 * Gh;      // tile and stage-in-tile of the first stage

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 2);
            mbar_init(&empty[s], kCG);
        }
        for (int i = 0; i < kCG; ++i) {
            mbar_init(&ready[i], 4);
            mbar_init(&done[i], 1);
            mbar_init(&fin[i], 1);
        }
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
    if (threadIdx.x == 0) Q4_TMTR(p, 4000);

    // Register split: the producer/issuer warpgroup needs few registers, the
    // three consumer warpgroups many (128*56 + 384*152 = 512*128 at launch).
    if (warp < kConsumerWarp0)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    else
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsConsumer));

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int tn = tS0, kn = kS0;                    // stage of the next nibble load
            // one barrier per stage, two arrivals: the nibble boxes and the two x records, each with its bytes
            auto issue_nibbles = [&](int slot) {
                uint8_t* sbase = smem + slot * kStageBytes;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)kNibStage);
                for (int cg = 0; cg < kCG; ++cg)
                    tma_load_2d_hint(sbase + cg * kNibBox, &map_nib, &full[slot], kn * 64,
                                     tn * kRowsTile + cg * kRowsCG, pol);
                if (++kn == Gh) {
                    kn = 0;
                    ++tn;
                }
            };
            // the weight stream needs nothing from the preceding kernel
            const int pre = nst < kStages ? nst : kStages;
            for (int si = 0; si < pre; ++si) issue_nibbles(si);
            int issued = pre, rec_issued = 0;
            pdl_wait();
            const unsigned int target = __ldcg(p.epoch) + 1u;
            int kr = kS0;                              // stage-in-tile of the next record copy
            int slot = 0;
            uint32_t ph = 0;
            for (int si = 0; si < nst; ++si) {
                if (si >= kStages) {
                    if (!wait_or_abort(p, &empty[slot], ph ^ 1u, 1u, abort_flag)) break;
                    Q4_TMTR(p, si);
                    issue_nibbles(slot);
                    ++issued;
                }
                // the stage's two x records, once their writers have published them
                const int g0 = 2 * kr;
                if (!wait_flag(p, p.flags + g0, target, abort_flag) || !wait_flag(p, p.flags + g0 + 1, target, abort_flag))
                    break;
                fence_proxy_async_all();
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(2 * kRec));
                bulk_copy_g2s(smem + slot * kStageBytes + kNibStage, p.xt + (int64_t)g0 * kRec, (uint32_t)(2 * kRec),
                              &full[slot]);
                ++rec_issued;
                if (++kr == Gh) kr = 0;
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
    } else if (warp <= kCG) {
        // ------------------------------------------------------------ MMA issuers (warp-uniform loop)
        const int cg = warp - 1;
        const uint32_t idesc = idesc_bf16_f32(128, 16);
        const uint64_t bdesc0 = smem_desc_noswizzle(smem_u32(smem + kNibStage), 256, 128);
        const uint32_t aA0 = tmem + kColA + (uint32_t)(cg * 4 * 32);
        const uint32_t dP0 = tmem + kColP + (uint32_t)(cg * 2 * 16);
        int slot = 0;
        uint32_t ph = 0;
        int uS = 2 * S0;
        for (int si = 0; si < nst; ++si) {
            if (!__all_sync(0xFFFFFFFFu, wait_or_abort(p, &full[slot], ph, 2u, abort_flag))) break;
            if (!__all_sync(0xFFFFFFFFu, wait_or_abort(p, &ready[cg], (uint32_t)(si & 1), 2u, abort_flag))) break;
            tc_fence_after();
            // the consumer group has folded the previous stage: its ring slot is free as far as this group goes
            if (si > 0 && lane == 0) mbar_arrive_relaxed(&empty[slot == 0 ? kStages - 1 : slot - 1]);
            // operands computed by the whole warp (warp-uniform values), issued by one lane
            const bool v0 = uS >= u0, v1 = uS + 1 < u1;
            const uint64_t bd0 = bdesc0 + (uint64_t)((slot * kStageBytes) >> 4);
            const uint64_t bd1 = bd0 + (uint64_t)(kRec >> 4);
            const uint32_t aS = aA0 + (uint32_t)((si & 1) * 64);
            if (lane == 0) {
                if (cg == 0) Q4_TMTR(p, 2000 + 2 * si);
                if (v0) {
                    tc_mma_ts(dP0, aS + 0u, bd0 + 0u, idesc, 0u);
                    tc_mma_ts(dP0, aS + 8u, bd0 + 32u, idesc, 1u);
                    tc_mma_ts(dP0, aS + 16u, bd0 + 64u, idesc, 1u);
                    tc_mma_ts(dP0, aS + 24u, bd0 + 96u, idesc, 1u);
                }
                if (v1) {
                    tc_mma_ts(dP0 + 16u, aS + 32u, bd1 + 0u, idesc, 0u);
                    tc_mma_ts(dP0 + 16u, aS + 40u, bd1 + 32u, idesc, 1u);
                    tc_mma_ts(dP0 + 16u, aS + 48u, bd1 + 64u, idesc, 1u);
                    tc_mma_ts(dP0 + 16u, aS + 56u, bd1 + 96u, idesc, 1u);
                }
                tc_commit(&done[cg]);
                if (cg == 0) Q4_TMTR(p, 2001 + 2 * si);
            }
            __syncwarp();
            if (++slot == kStages) {
                slot = 0;
                ph ^= 1u;
            }
            uS += 2;
        }
        // no MMA of this warp may still run when tensor memory is freed
        if (lane == 0) {
            tc_commit(&fin[cg]);
            mbar_wait(&fin[cg], 0, kWaitLimit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - kConsumerWarp0;          // 0..11
        const int cg = cw >> 2;
        const int q = warp & 3;                        // tensor-memory lane quarter of this warp
        const int row = q * 32 + lane;                 // row within the consumer group's 128
        const int ct = cw * 32 + lane;                 // 0..383 among the consumers
        const uint32_t lane_field = (uint32_t)(q * 32) << 16;
        const uint32_t aA0 = tmem + lane_field + kColA + (uint32_t)(cg * 4 * 32);
        const uint32_t dP0 = tmem + lane_field + kColP + (uint32_t)(cg * 2 * 16);
        const int t_first = u0 / p.G;
        [[maybe_unused]] const int tr = (lane == 0 && q == 0 && cg == 0) ? 1000 : 1 << 20;

        // scale and bias planes: per row 16-byte blocks of 8 groups (four stages)
        const uint8_t* splane = p.W + p.N * (p.K / 2);
        const uint8_t* bplane = splane + p.N * p.G * 2;
        const int rows_cg = cg * kRowsCG + row;
        auto load_sb = [&](int t, int k, uint4& sv, uint4& bv) {   // block starting at stage-in-tile k of tile t
            const int64_t n = (int64_t)t * kRowsTile + rows_cg;
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

        // x records of this CTA's groups (g = c_id, c_id + C, ...), published for every CTA
        pdl_wait();                                    // x, the records, y and the split-K scratch
        {
            const unsigned int target = __ldcg(p.epoch) + 1u;
            for (int g = c_id; g < p.G; g += p.C) {
                if (ct < 128) {                        // 16 rows x 8 blocks of 8 inputs
                    const int m = ct >> 3, c = ct & 7;
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (m < p.M) v = __ldg(reinterpret_cast<const uint4*>(p.x + (int64_t)m * p.K + 64 * g + 8 * c));
                    uint4 o;
                    float s = x_block(v, o);
                    uint8_t* rec = p.xt + (int64_t)g * kRec;
                    *reinterpret_cast<uint4*>(rec + c * 256 + (m >> 3) * 128 + (m & 7) * 16) = o;
                    // the 8 block sums of row m sit in 8 consecutive lanes: a fixed tree
                    s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 1));
                    s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 2));
                    s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 4));
                    if (c == 0) reinterpret_cast<float*>(rec + 2048)[m] = s;
                }
            }
            fence_proxy_async_all();                   // the records are read by bulk copies
            named_barrier(5, kConsumerThreads);
            if (ct == 0) {
                __threadfence();
                for (int g = c_id; g < p.G; g += p.C) st_release_gpu(p.flags + g, target);
            }
        }

        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
        bool live = true;

        // the previous stage, folded during this one
        int pslot = 0, pkst = 0, pt = 0, puS = -1;
        float ps0 = 0.f, ps1 = 0.f, pr0 = 0.f, pr1 = 0.f;
        auto fold_group = [&](int jj, const uint32_t* P, const float* xsum, float s, float r) {
            float X[MT];
            if (MT >= 4) {
#pragma unroll
                for (int v4 = 0; v4 < MT / 4; ++v4) {
                    const float4 v = reinterpret_cast<const float4*>(xsum)[v4];
                    X[4 * v4 + 0] = v.x;
                    X[4 * v4 + 1] = v.y;
                    X[4 * v4 + 2] = v.z;
                    X[4 * v4 + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int m = 0; m < MT; ++m) X[m] = xsum[m];
            }
            if (MT == 1) {
                acc[0] = __fmaf_rn(s, __uint_as_float(P[0]), __fmaf_rn(r, X[0], acc[0]));
            } else {
#pragma unroll
                for (int m = 0; m + 1 < MT; m += 2) {
                    fma2(acc[m], acc[m + 1], r, X[m], X[m + 1]);
                    fma2(acc[m], acc[m + 1], s, __uint_as_float(P[m]), __uint_as_float(P[m + 1]));
                }
            }
        };
        auto close_group = [&](int jj) {
            const int uf = puS + jj, gf = 2 * pkst + jj;
            if (uf >= u0 && uf < u1 && (uf == u1 - 1 || gf == p.G - 1)) {
                const bool whole = gf == p.G - 1 && pt * p.G >= u0;
                end_segment<MT>(p, acc, pt, whole, pt == t_first ? 0 : 1, cg, row, row, c_id, bcast, !*abort_flag);
            }
        };
        // fold the previous stage: wait for its MMAs, read both groups' P, add s*P + r*X
        auto fold_prev = [&]() {
            const bool v0 = puS >= u0 && puS < u1, v1 = puS + 1 >= u0 && puS + 1 < u1;
            const uint32_t par = (uint32_t)(((puS - 2 * S0) >> 1) & 1);
            const bool w = __all_sync(0xFFFFFFFFu, live && wait_or_abort(p, &done[cg], par, 4u, abort_flag));
            const float* xs0 = reinterpret_cast<const float*>(smem + pslot * kStageBytes + kNibStage + 2048);
            const float* xs1 = reinterpret_cast<const float*>(smem + pslot * kStageBytes + kNibStage + kRec + 2048);
            if (w) {
                tc_fence_after();
                if (MT <= 8) {
                    uint32_t P0[8], P1[8];
                    tmem_ld_32x32b_x8(dP0, P0);
                    tmem_ld_32x32b_x8(dP0 + 16u, P1);
                    tmem_wait_ld();
                    if (v0) fold_group(0, P0, xs0, ps0, pr0);
                    close_group(0);
                    if (v1) fold_group(1, P1, xs1, ps1, pr1);
                } else {
                    uint32_t P[32];
                    tmem_ld_32x32b_x32(dP0, P);
                    tmem_wait_ld();
                    if (v0) fold_group(0, P, xs0, ps0, pr0);
                    close_group(0);
                    if (v1) fold_group(1, P + 16, xs1, ps1, pr1);
                }
            } else {
                close_group(0);
            }
            close_group(1);
        };

        int slot = 0;
        uint32_t ph = 0;
        int kst = kS0, t = tS0;
        int uS = 2 * S0;
        // constants of the stage about to be dequantized, computed one iteration ahead
        float cs0, cs1, cr0, cr1;
        uint32_t cc0a, cc0b;
        auto stage_constants = [&](int k) {
            const int wsel = k & 3;
            const uint32_t sw = wsel == 0 ? cur_s.x : wsel == 1 ? cur_s.y : wsel == 2 ? cur_s.z : cur_s.w;
            const uint32_t bw = wsel == 0 ? cur_b.x : wsel == 1 ? cur_b.y : wsel == 2 ? cur_b.z : cur_b.w;
            group_constants(sw, bw, cs0, cr0, cc0a);
            group_constants(sw >> 16, bw >> 16, cs1, cr1, cc0b);
        };
        stage_constants(kst);
        for (int si = 0; si < nst; ++si) {
            Q4_TMTR(p, tr + 8 * si + 0);
            live = __all_sync(0xFFFFFFFFu, live && wait_or_abort(p, &full[slot], ph, 8u, abort_flag));
            Q4_TMTR(p, tr + 8 * si + 1);
            const uint8_t* nb = smem + slot * kStageBytes + cg * kNibBox + row * 64;
            const int sx = (row >> 1) & 3;
            const uint32_t aA = aA0 + (uint32_t)((si & 1) * 64);
            const bool g0 = live && uS >= u0, g1 = live && uS + 1 < u1;   // groups of the stage owned by this CTA
            const uint4 n0 = *reinterpret_cast<const uint4*>(nb + ((0 ^ sx) << 4));
            const uint4 n1 = *reinterpret_cast<const uint4*>(nb + ((1 ^ sx) << 4));
            const uint4 n2 = *reinterpret_cast<const uint4*>(nb + ((2 ^ sx) << 4));
            const uint4 n3 = *reinterpret_cast<const uint4*>(nb + ((3 ^ sx) << 4));
            if (g0) {
                uint32_t a[32];
                dequant64(n0, n1, cc0a, a);
                tmem_st_32x32b_x32(aA, a);
                tmem_wait_st();                        // the registers are reused next: store first
            }
            if (g1) {
                uint32_t a[32];
                dequant64(n2, n3, cc0b, a);
                tmem_st_32x32b_x32(aA + 32u, a);
                tmem_wait_st();
            }
            Q4_TMTR(p, tr + 8 * si + 2);
            if (puS >= 0) fold_prev();
            Q4_TMTR(p, tr + 8 * si + 3);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ready[cg]);
            pslot = slot;
            pkst = kst;
            pt = t;
            puS = uS;
            ps0 = cs0;
            ps1 = cs1;
            pr0 = cr0;
            pr1 = cr1;
            if (++slot == kStages) {
                slot = 0;
                ph ^= 1u;
            }
            if (++kst == Gh) {
                kst = 0;
                ++t;
            }
            uS += 2;
            if (si + 1 < nst) {
                if ((kst & 3) == 0) {
                    cur_s = nxt_s;
                    cur_b = nxt_b;
                    sb_next();
                    if (S_sb < S0 + nst) load_sb(t_sb, k_sb, nxt_s, nxt_b);
                }
                stage_constants(kst);
            }
        }
        if (puS >= 0) fold_prev();
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        Q4_TMTR(p, 4001);
        // the last CTA of the launch advances the epoch for the next launch's records
        __threadfence();
        const unsigned int prev = atomicAdd(p.finished, 1u);
        if (prev == (unsigned int)p.C - 1u) {
            *p.finished = 0u;
            __threadfence();
            atomicAdd(p.epoch, 1u);
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

inline int smem_bytes() { return kSmemBytes; }
inline size_t partial_floats(int C) { return (size_t)C * 2 * kCG * 16 * kRowsCG; }
inline size_t sem_ints(int C) { return (size_t)C * kCG; }

}  // namespace tm
}  // namespace q4
