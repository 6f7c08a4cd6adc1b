// Production Q4 verify-matmul kernel for sm_103a (K a multiple of 512).
//
// y[m,n] = sum_g ( s[n,g] * P[m,n,g] + r[n,g] * X[m,g] )
//   P[m,n,g] = sum_{k in g} (q[n,k] - c[n,g]) * x[m,k]      (tensor core, exact products)
//   X[m,g]   = sum_{k in g} x[m,k]                           (tensor core, A = ones)
//   c[n,g]   = clamp(rint(-b/s), 0, 15),  r[n,g] = b + c*s
// which is w = s*q + b = s*(q - c) + r regrouped.  q - c is an exact small
// integer in bf16, and |r| <= s/2 whenever -b/s lies in [0,15], so s*P and r*X
// never cancel catastrophically: the error stays a small multiple of the fp32
// unit roundoff times sum_k |x_k w_k|, and an all-zero weight row (q == c,
// b == -c*s) gives exactly zero.
//
// Structure (one persistent CTA per SM, 16 warps):
//   warp 0       TMA producer: per stage, the nibble tiles of SG groups for a
//                384-row tile (3 boxes of 128 rows x 32 B each, 32-byte swizzle)
//                and the raw x tile of each group (16 rows x 64 inputs).
//   warps 1..3   MMA issuers, one per consumer group: 4 MMAs M128 N16 K16 per
//                group (A = dequantized weights in tensor memory, B = x from
//                shared memory), plus the 4 X MMAs of every third group.
//   warps 4..15  three consumer groups of 4 warps; consumer group cg owns rows
//                128*cg .. 128*cg+127 of the tile, one row per thread.  Per
//                group: permute x for the tensor core (one group in three),
//                dequantize 64 nibbles into (q - c) bf16 pairs, store them to
//                tensor memory, and fold the previous group's P and X into the
//                fp32 accumulators with s and r.
// Work split: the T*G (tile, group) units are cut into equal contiguous
// ranges, one per CTA (stream-K).  A tile whose groups span several CTAs is
// finished by the last of them to arrive, which adds the partial sums in
// increasing CTA order; the split depends only on N, K and the grid size, so
// the result of every row is independent of M and of the other rows.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "q4_sm100.cuh"

namespace q4 {
namespace tc {

constexpr int kCG = 3;                      // consumer groups
constexpr int kRowsCG = 128;                // rows per consumer group (TMEM lanes)
constexpr int kRowsTile = kCG * kRowsCG;    // 384 rows per tile
constexpr int kSG = 2;                      // groups per pipeline stage
constexpr int kStages = 6;
constexpr int kNBUF = 2;                    // tensor-memory A/P buffers per consumer group
constexpr int kThreads = 512;
constexpr int kConsumerWarp0 = 4;

constexpr int kNibBox = kRowsCG * 32;                 // 4 KB: 128 rows x 32 B
constexpr int kNibGroup = kCG * kNibBox;              // 12 KB per group
constexpr int kXBytes = 16 * 64 * 2;                  // 2 KB raw x per group
constexpr int kStageBytes = kSG * (kNibGroup + 2 * kXBytes);
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /* barriers etc. */ + 1024 /* alignment slack */;

// tensor-memory columns
constexpr uint32_t kColOnes = 0;
constexpr uint32_t kColA = 32;
constexpr uint32_t kColP = kColA + kCG * kNBUF * 32;
constexpr uint32_t kColX = kColP + kCG * kNBUF * 16;
constexpr uint32_t kTmemCols = 512;
static_assert(kColX + kNBUF * 16 <= kTmemCols, "tensor memory over-subscribed");

constexpr long long kWaitLimit = 2000000000LL;   // cycles (about one second)

struct Params {
    const uint8_t* W;           // packed weights (scales/biases read directly)
    float* y;                   // [M, N]
    float* partials;            // scratch: [C][2][kCG][16][128]
    int* sems;                  // scratch: [C][kCG], zero between launches
    unsigned int* error_word;   // set on a timed-out wait
    int64_t N;
    int64_t K;
    int M;
    int G;                      // K / 64
    int T;                      // tiles of 384 rows
    int64_t U;                  // T * G units
    int C;                      // CTAs (grid size)
};

// Range of units owned by CTA c.
__device__ __forceinline__ int64_t range_start(int64_t U, int C, int c) { return (U * (int64_t)c) / C; }

// CTA that owns unit u.
__device__ __forceinline__ int cta_of_unit(int64_t U, int C, int64_t u) {
    int c = (int)((u * (int64_t)C) / U);
    while (c + 1 < C && range_start(U, C, c + 1) <= u) ++c;
    while (c > 0 && range_start(U, C, c) > u) --c;
    return c;
}

// Iterates the stages of one CTA's unit range: each stage is up to kSG
// consecutive groups of one tile.
struct StageIter {
    int64_t u, u_end;
    int G;
    __device__ void init(const Params& p, int c) {
        u = range_start(p.U, p.C, c);
        u_end = range_start(p.U, p.C, c + 1);
        G = p.G;
    }
    __device__ bool done() const { return u >= u_end; }
    // current stage: tile t, first group g0, count nv
    __device__ void current(int& t, int& g0, int& nv) const {
        t = (int)(u / G);
        g0 = (int)(u - (int64_t)t * G);
        int64_t lim = (int64_t)t * G + G;
        if (lim > u_end) lim = u_end;
        int64_t n = lim - u;
        nv = n < kSG ? (int)n : kSG;
    }
    __device__ void advance(int nv) { u += nv; }
};

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// (128 + q) as bf16 pairs for nibbles (lo half: bits 0-3, hi half: bits 16-19) of v.
__device__ __forceinline__ uint32_t nib_pair(uint32_t v) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "r"(0x000F000Fu), "r"(0x43004300u));   // (a & b) | c
    return d;
}

__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void record_timeout(const Params& p, unsigned int code, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(p.error_word, code);
}

template <int MT>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    q4::sm100::tmem_ld_32x32b_x16(taddr, r);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Fixed-order finish of one 128-row slice of a tile whose groups span CTAs
// [c_first, c_last]; called by the 128 threads of one consumer group of the
// last CTA to arrive.
template <int MT>
__device__ void finish_shared_slice(const Params& p, int t, int cg, int row, int c_first, int c_last) {
    const int64_t n = (int64_t)t * kRowsTile + cg * kRowsCG + row;
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
    for (int c = c_first; c <= c_last; ++c) {
        const int64_t cs = range_start(p.U, p.C, c);
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

// Bounded wait that also gives up at once when another role has already
// given up (the whole CTA then runs to its end without further waiting).
__device__ __forceinline__ bool wait_or_abort(const Params& p, uint64_t* bar, uint32_t parity, unsigned code,
                                              volatile int* abort_flag) {
    if (*abort_flag) return false;
    if (q4::sm100::mbar_wait(bar, parity, kWaitLimit)) return true;
    record_timeout(p, code, abort_flag);
    return false;
}

// End of this CTA's segment of tile t for one consumer group: store the sums
// (whole tile), or publish them as a partial and let the last contributor
// add all partials of the tile slice in increasing CTA order.
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
        __threadfence();
        named_barrier(1 + cg, kRowsCG);
        if (cg_tid == 0) {
            int last = 0;
            if (live) {
                const int64_t tu = (int64_t)t * p.G;
                const int c_first = cta_of_unit(p.U, p.C, tu);
                const int c_last = cta_of_unit(p.U, p.C, tu + p.G - 1);
                int* sem = p.sems + c_first * kCG + cg;
                const int old = atomicAdd(sem, 1);
                if (old == c_last - c_first) {
                    atomicExch(sem, 0);      // leave the counter at zero for the next launch
                    last = 1;
                }
            }
            bcast[cg] = last;
        }
        named_barrier(1 + cg, kRowsCG);
        if (bcast[cg]) {
            __threadfence();
            const int64_t tu = (int64_t)t * p.G;
            finish_shared_slice<MT>(p, t, cg, row, cta_of_unit(p.U, p.C, tu), cta_of_unit(p.U, p.C, tu + p.G - 1));
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
q4_tc_kernel(const __grid_constant__ CUtensorMap map_nib, const __grid_constant__ CUtensorMap map_x, const Params p) {
    using namespace q4::sm100;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* ready = empty + kStages;                 // [kNBUF]
    uint64_t* done = ready + kNBUF;                    // [kCG][kNBUF]
    uint64_t* fin = done + kCG * kNBUF;                // [kCG]
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(fin + kCG);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);
    int* bcast = const_cast<int*>(abort_flag) + 1;     // [kCG]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c_id = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCG);
        }
        for (int b = 0; b < kNBUF; ++b) mbar_init(&ready[b], kCG * kRowsCG);
        for (int i = 0; i < kCG * kNBUF; ++i) mbar_init(&done[i], 1);
        for (int i = 0; i < kCG; ++i) mbar_init(&fin[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_nib);
        prefetch_tensormap(&map_x);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            StageIter it;
            it.init(p, c_id);
            int st = 0;
            const uint64_t pol = policy_evict_first();
            while (!it.done()) {
                int t, g0, nv;
                it.current(t, g0, nv);
                const int slot = st % kStages;
                if (st >= kStages && !wait_or_abort(p, &empty[slot], ((st / kStages) - 1) & 1, 1u, abort_flag)) break;
                uint8_t* sbase = smem + slot * kStageBytes;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)nv * (kNibGroup + kXBytes));
                for (int j = 0; j < nv; ++j) {
                    const int g = g0 + j;
                    for (int cg = 0; cg < kCG; ++cg)
                        tma_load_2d_hint(sbase + j * kNibGroup + cg * kNibBox, &map_nib, &full[slot], g * 32,
                                         t * kRowsTile + cg * kRowsCG, pol);
                    tma_load_2d(sbase + kSG * kNibGroup + j * kXBytes, &map_x, &full[slot], g * 64, 0);
                }
                it.advance(nv);
                ++st;
            }
            // every issued stage must have landed before the CTA may exit
            for (int s = (st > kStages ? st - kStages : 0); s < st; ++s)
                mbar_wait(&full[s % kStages], (s / kStages) & 1, kWaitLimit);
        }
    } else if (warp <= kCG) {
        // ------------------------------------------------------------ MMA issuers
        const int cg = warp - 1;
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, 16);
            StageIter it;
            it.init(p, c_id);
            int st = 0, i = 0;
            bool live = true;
            while (!it.done() && live) {
                int t, g0, nv;
                it.current(t, g0, nv);
                const int slot = st % kStages;
                uint8_t* sbase = smem + slot * kStageBytes;
                for (int j = 0; j < nv; ++j, ++i) {
                    const int b = i % kNBUF;
                    if (!wait_or_abort(p, &ready[b], (i / kNBUF) & 1, 2u, abort_flag)) {
                        live = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t bperm = smem_u32(sbase + kSG * (kNibGroup + kXBytes) + j * kXBytes);
                    if (i % kCG == cg) {
                        const uint32_t dX = tmem + kColX + (uint32_t)(b * 16);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_ts(dX, tmem + kColOnes + 8 * kk, smem_desc_noswizzle(bperm + kk * 512, 256, 128),
                                      idesc, kk > 0);
                    }
                    const uint32_t dP = tmem + kColP + (uint32_t)((cg * kNBUF + b) * 16);
                    const uint32_t aA = tmem + kColA + (uint32_t)((cg * kNBUF + b) * 32);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_ts(dP, aA + 8 * kk, smem_desc_noswizzle(bperm + kk * 512, 256, 128), idesc, kk > 0);
                    tc_commit(&done[cg * kNBUF + b]);
                    if (j == nv - 1) tc_commit(&empty[slot]);
                }
                it.advance(nv);
                ++st;
            }
            // no MMA of this thread may still run when tensor memory is freed
            tc_commit(&fin[cg]);
            mbar_wait(&fin[cg], 0, kWaitLimit);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - kConsumerWarp0;          // 0..11
        const int cg = cw / 4;
        const int q = warp & 3;                        // tensor-memory lane quarter of this warp
        const int row = q * 32 + lane;                 // row within the consumer group's 128
        const int cg_tid = (cw & 3) * 32 + lane;       // 0..127 within the consumer group
        const uint32_t lane_field = (uint32_t)(q * 32) << 16;

        if (cg == 0) {
            uint32_t ones[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) ones[k] = 0x3F803F80u;      // bf16 1.0 pairs
            tmem_st_32x32b_x32(tmem + lane_field + kColOnes, ones);
            tmem_wait_st();
        }

        const uint16_t* scales = reinterpret_cast<const uint16_t*>(p.W + p.N * (p.K / 2));
        const uint16_t* biases = scales + p.N * (int64_t)p.G;
        const int64_t u0 = range_start(p.U, p.C, c_id);
        const int64_t u1 = range_start(p.U, p.C, c_id + 1);
        const int t_first = (int)(u0 / p.G);

        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

        // the previous group, folded one iteration later
        bool pv_valid = false, pv_last = false, pv_whole = false;
        float pv_s = 0.f, pv_r = 0.f;
        int pv_b = 0, pv_i = 0, pv_t = 0;

        int sb_t = -1, sb_blk = -1;
        uint4 sv = make_uint4(0, 0, 0, 0), bv = make_uint4(0, 0, 0, 0);

        StageIter it;
        it.init(p, c_id);
        int st = 0, i = 0;
        while (!it.done()) {
            int t, g0, nv;
            it.current(t, g0, nv);
            const int slot = st % kStages;
            uint8_t* sbase = smem + slot * kStageBytes;
            const bool have_stage = wait_or_abort(p, &full[slot], (st / kStages) & 1, 8u, abort_flag);
            for (int j = 0; j < nv; ++j, ++i) {
                const int g = g0 + j;
                const int b = i % kNBUF;
                const int64_t unit = (int64_t)t * p.G + g;
                const bool last_in_seg = (g == p.G - 1) || (unit == u1 - 1);
                const int seg_first = (t == t_first) ? (int)(u0 - (int64_t)t_first * p.G) : 0;
                const bool whole = (seg_first == 0) && (g == p.G - 1);
                float s = 0.f, rr = 0.f;
                // warp-uniform: tcgen05.st below is a warp-collective instruction
                const bool live = __all_sync(0xFFFFFFFFu, have_stage && !*abort_flag);
                if (live) {
                    // (1) x, permuted for the tensor core (one consumer group per group)
                    if (i % kCG == cg) {
                        const int e = cg_tid & 7, d = (cg_tid >> 3) & 7, mg = cg_tid >> 6;
                        const int r8 = (e + d) & 7, m = mg * 8 + r8;
                        const uint8_t* xr = sbase + kSG * kNibGroup + j * kXBytes;
                        uint8_t* bp = sbase + kSG * (kNibGroup + kXBytes) + j * kXBytes;
                        const uint4 w = *reinterpret_cast<const uint4*>(xr + m * 128 + e * 16);
                        uint4 o;
                        o.x = prmt(w.x, w.z, 0x5410u);
                        o.y = prmt(w.x, w.z, 0x7632u);
                        o.z = prmt(w.y, w.w, 0x5410u);
                        o.w = prmt(w.y, w.w, 0x7632u);
                        *reinterpret_cast<uint4*>(bp + e * 256 + mg * 128 + r8 * 16) = o;
                        fence_proxy_async_smem();
                    }
                    // (2) scale, bias and the centring integer c of this row and group
                    const int64_t n = (int64_t)t * kRowsTile + cg * kRowsCG + row;
                    const int blk = g >> 3;
                    if (t != sb_t || blk != sb_blk) {
                        sb_t = t;
                        sb_blk = blk;
                        if (n < p.N) {
                            sv = __ldg(reinterpret_cast<const uint4*>(scales + n * p.G + blk * 8));
                            bv = __ldg(reinterpret_cast<const uint4*>(biases + n * p.G + blk * 8));
                        } else {
                            sv = make_uint4(0, 0, 0, 0);
                            bv = make_uint4(0, 0, 0, 0);
                        }
                    }
                    const int gi = g & 7;
                    const uint32_t sw = gi < 2 ? sv.x : gi < 4 ? sv.y : gi < 6 ? sv.z : sv.w;
                    const uint32_t bw = gi < 2 ? bv.x : gi < 4 ? bv.y : gi < 6 ? bv.z : bv.w;
                    s = __uint_as_float((gi & 1) ? (sw & 0xFFFF0000u) : (sw << 16));
                    const float bb = __uint_as_float((gi & 1) ? (bw & 0xFFFF0000u) : (bw << 16));
                    float cf = rintf(__fdividef(-bb, s));
                    cf = fminf(fmaxf(cf, 0.0f), 15.0f);            // NaN -> 0
                    rr = __fmaf_rn(cf, s, bb);
                    const uint32_t cc = (0x4300u | (uint32_t)cf) * 0x00010001u;
                    // (3) the row's 64 nibbles (32-byte swizzle: 16-byte chunk ^= (row >> 2) & 1)
                    const uint8_t* nb = sbase + j * kNibGroup + cg * kNibBox + row * 32;
                    const int sx = (row >> 2) & 1;
                    const uint4 n0 = *reinterpret_cast<const uint4*>(nb + (sx << 4));
                    const uint4 n1 = *reinterpret_cast<const uint4*>(nb + ((sx ^ 1) << 4));
                    const uint32_t wv[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
                    uint32_t a[32];
#pragma unroll
                    for (int wi = 0; wi < 8; ++wi) {
                        const uint32_t v = wv[wi];
                        a[4 * wi + 0] = bf16x2_sub(nib_pair(v), cc);
                        a[4 * wi + 1] = bf16x2_sub(nib_pair(v >> 4), cc);
                        a[4 * wi + 2] = bf16x2_sub(nib_pair(v >> 8), cc);
                        a[4 * wi + 3] = bf16x2_sub(nib_pair(v >> 12), cc);
                    }
                    // (4) A to tensor memory; announce the group to the issuers
                    tmem_st_32x32b_x32(tmem + lane_field + kColA + (uint32_t)((cg * kNBUF + b) * 32), a);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&ready[b]);
                }
                // (5) fold the previous group's products into the sums
                if (pv_valid) {
                    const int xi = pv_i % kCG;
                    const uint32_t par = (pv_i / kNBUF) & 1;
                    bool w = wait_or_abort(p, &done[cg * kNBUF + pv_b], par, 4u, abort_flag);
                    if (w && xi != cg) w = wait_or_abort(p, &done[xi * kNBUF + pv_b], par, 4u, abort_flag);
                    w = __all_sync(0xFFFFFFFFu, w);          // tcgen05.ld is warp-collective
                    if (w) {
                        tc_fence_after();
                        float Pv[16], Xv[16];
                        tmem_load_cols<MT>(tmem + lane_field + kColP + (uint32_t)((cg * kNBUF + pv_b) * 16), Pv);
                        tmem_load_cols<MT>(tmem + lane_field + kColX + (uint32_t)(pv_b * 16), Xv);
                        tmem_wait_ld();
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            acc[m] = __fmaf_rn(pv_s, Pv[m], acc[m]);
                            acc[m] = __fmaf_rn(pv_r, Xv[m], acc[m]);
                        }
                    }
                    if (pv_last)
                        end_segment<MT>(p, acc, pv_t, pv_whole, pv_t == t_first ? 0 : 1, cg, row, cg_tid, c_id,
                                        bcast, !*abort_flag);
                }
                pv_valid = true;
                pv_last = last_in_seg;
                pv_whole = whole;
                pv_s = s;
                pv_r = rr;
                pv_b = b;
                pv_i = i;
                pv_t = t;
            }
            it.advance(nv);
            ++st;
        }
        if (pv_valid) {
            const int xi = pv_i % kCG;
            const uint32_t par = (pv_i / kNBUF) & 1;
            bool w = wait_or_abort(p, &done[cg * kNBUF + pv_b], par, 4u, abort_flag);
            if (w && xi != cg) w = wait_or_abort(p, &done[xi * kNBUF + pv_b], par, 4u, abort_flag);
            w = __all_sync(0xFFFFFFFFu, w);
            if (w) {
                tc_fence_after();
                float Pv[16], Xv[16];
                tmem_load_cols<MT>(tmem + lane_field + kColP + (uint32_t)((cg * kNBUF + pv_b) * 16), Pv);
                tmem_load_cols<MT>(tmem + lane_field + kColX + (uint32_t)(pv_b * 16), Xv);
                tmem_wait_ld();
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    acc[m] = __fmaf_rn(pv_s, Pv[m], acc[m]);
                    acc[m] = __fmaf_rn(pv_r, Xv[m], acc[m]);
                }
            }
            end_segment<MT>(p, acc, pv_t, pv_whole, pv_t == t_first ? 0 : 1, cg, row, cg_tid, c_id, bcast,
                            !*abort_flag);
        }
    }

    tc_fence_before();
    __syncthreads();
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
