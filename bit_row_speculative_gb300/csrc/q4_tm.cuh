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
// fold applies s * 2^33.  Range: |x| < 2^28 (x * 2^100 stays finite); a
// nonzero |x| below 2^-93 gives products below the fp32 normal range, which
// the tensor core may flush; s * 2^33 must stay finite (|s| < 2^95).
//
// x records.  Per group of 64 inputs: the fp32 group sums X[0..W-1], then the
// rows of x for the group's inputs as tensor-core core matrices (8 rows x 8
// inputs, 128 B each), 8-row blocks one after another (2112 bytes at W = 16,
// 4224 at W = 32; W = 16 for M <= 16, 32 for M <= 32).  Inputs of each 8-block
// are in the dequantized order k0 k4 k1 k5 k2 k6 k3 k7 and scaled as above;
// rows >= M are zero.  A call builds them into global scratch at its start: the
// MMA-issuer warps of CTA c build groups c, c + C, ... and count them on a device
// counter, and a team's producer lanes copy a stage's records only once the
// count says all are there.  Meanwhile each consumer team builds the records of
// its own first stages from x straight into its shared record slots, so it can
// start about one L2 latency after its predecessor finished.  Inside a chained
// pass the glue kernel has already written the records, and the call neither
// builds nor waits.
//
// One persistent CTA per SM, 16 warps; tiles of 128 rows (tensor-memory
// lanes), a stage is two groups (128 inputs) of one tile.  The T*G/2 (tile,
// group pair) units are cut into R = 3C equal contiguous ranges (stream-K),
// and consumer team j of CTA c works through range 3c + j on its own.
//   warp 0       producers.  One thread keeps only about one TMA operation in
//                flight at a time, so each team's streams are spread over
//                lanes: two issue its weights (a 128-row x 64-byte nibble box
//                per stage, L2 evict-first, into the team's nibble ring, and
//                at the first stage of each block of 8 groups a box of those
//                rows' scale and bias words), two copy its stages' records
//                into its record ring.  The lanes run one polling loop.  Two
//                stages of weights go out before the preceding kernel has
//                ended; the rest of the first ring-full only once every team
//                has loaded its x (which would otherwise queue behind them).
//   warps 1..3   MMA issuers, one per team: per stage 8 MMAs M128 N16 K16 (16
//                at W = 32: rows 0-15 and rows 16-31 as two N = 16 MMAs, so a
//                row's products never depend on the row width), A = the
//                dequantized weights in the team's tensor memory, B = the
//                stage's records in shared memory, D = the team's P; then a
//                commit to the team's "done" barrier.  Before that, their
//                share of the call's records.
//   warps 4..15  three consumer teams of 4 warps, one row per thread.  At
//                W = 16 a team keeps two A buffers: in its iteration for stage
//                k it dequantizes stage k into one while the MMAs of stage
//                k - 1 run on the other, loads that stage's P, hands stage k
//                to its issuer, then folds P into its fp32 sums with s, r and
//                X and frees stage k - 1's slots.  At W = 32 (one A buffer, to
//                fit tensor memory) it folds stage k - 1 first.
// Segment ends: a range covers at most two partial tiles (its first and last
// segments) and whole tiles between.  A warp stores a whole tile's 32 rows to
// y; for a partial tile it publishes its rows and counts them on the tile's
// quarter counter, and the last of the tile's contributors to arrive adds the
// partials in increasing range order and stores y.  No warp waits for another
// warp or CTA there.  The split depends only on N, K and the SM count, and
// nothing in the arithmetic of row m depends on the other rows, so every row's
// result is independent of M and of the run.
// Every barrier wait is bounded; a wait that runs out sets the error word and
// the CTA runs to its end without further waiting.  Counters return to zero
// within the call: a tile quarter's counter by its last contributor, the record
// counters by the last CTA whose record readers have all seen the records (so
// no CTA ends with a round trip to memory).  A call that gave up a wait may
// leave them set; the status query that reports the timeout clears them.  All
// CTAs of a call must be resident together (one per SM, as launched): a CTA
// waits for the records the others build.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "q4_sm100.cuh"

namespace q4 {
namespace tm {

constexpr int kRowsTile = 128;              // rows per tile (tensor-memory lanes)
constexpr int kTeams = 3;                   // consumer teams (one warpgroup each)
constexpr int kConsumerWarp0 = 4;           // warps 4.. (warp % 4 = tensor-memory lane quarter)
constexpr int kThreads = (kConsumerWarp0 + 4 * kTeams) * 32;   // 512
constexpr int kNibStage = kRowsTile * 64;   // 8 KB: 128 rows x 64 B (two groups)
constexpr int kRecHalf = 1088;              // W = 16: X and rows 0-7

template <int MT>
__host__ __device__ constexpr int width() { return MT > 16 ? 32 : 16; }
__host__ __device__ constexpr int rec_bytes(int W) { return 4 * W + (W / 8) * 1024; }   // X[W] fp32, then W/8 blocks of 8 rows
__host__ __device__ constexpr int rec_b(int W) { return 4 * W; }                        // offset of the core matrices
// Per team: a ring of nibble slots (one 128-row x 64-byte box each) and a ring
// of record slots (the stage's two x records; the group sums X in them are read
// by all four warps of the team), of the same depth: stage k uses slot k % depth
// of each.  One "full" barrier per slot counts the stage's weight box, its
// scale/bias box and its record copy together, and one "empty" barrier frees
// both slots once the stage's P is folded, so a consumer warp makes one wait
// and one arrival per stage on the ring (each costs a round trip).
__host__ __device__ constexpr int nib_slots(int W) { return W == 16 ? 5 : 4; }
__host__ __device__ constexpr int rec_slots(int W) { return nib_slots(W); }
__host__ __device__ constexpr int rec_stage_bytes(int W) { return ((2 * rec_bytes(W) + 127) / 128) * 128; }
// Stages whose records a team builds itself from x at its start (they do not
// wait for the call's shared records).
__host__ __device__ constexpr int local_stages(int W) { return W == 16 ? 3 : 2; }
// Weight stages per team issued before griddepcontrol.wait.  The rest of the
// ring's first fill waits until every team has loaded its x: x arrives after the
// preceding kernel ends and would otherwise queue behind a ring-full of weights
// on the way into the SM (measured: 0.8 us per attention call).
constexpr int kEarlyStages = 2;
static_assert(kEarlyStages <= nib_slots(16) && kEarlyStages <= nib_slots(32), "early stages must find free slots");
// Producer lanes per team and stream.  A lane issues every L-th stage of its
// team into a ring of S slots and waits, by phase parity, for the slot's previous
// user; that wait is unambiguous only while the lane cannot run more than one
// phase ahead of the slot, which L <= S guarantees (its own previous stage, L
// earlier, already waited for the stage S before that).
constexpr int kWeightLanes = 2;
constexpr int kRecordLanes = 2;
// Scale and bias words: per team two buffers (blocks of 8 groups = 4 stages),
// each a 128-row x 16-byte box of the scale plane and one of the bias plane.  A
// buffer is reloaded at the first stage of the block after next, which the
// producer issues only once the slots of the stage nib_slots earlier have been
// freed (that stage folded): at most 5 slots keep that stage at or after the
// last stage of the block the buffer held.
constexpr int kSbBuffers = 2;
static_assert((kSbBuffers & (kSbBuffers - 1)) == 0, "buffer index by mask");
constexpr int kSbBox = kRowsTile * 16;                          // 2 KB
constexpr int kSbBytes = kTeams * kSbBuffers * 2 * kSbBox;      // 24 KB
static_assert(nib_slots(16) <= 4 * (kSbBuffers - 1) + 1 && nib_slots(32) <= 4 * (kSbBuffers - 1) + 1,
              "a scale/bias buffer could be reloaded while a stage of its block is still unread");
constexpr int kBarrierBytes = 1024;
// full and empty per ring slot, ready/done/fin per team, x-ready; then the tensor-memory base and the
// abort flag
static_assert((kTeams * 2 * nib_slots(16) + 3 * kTeams + 1) * 8 + 8 <= kBarrierBytes &&
                  (kTeams * 2 * nib_slots(32) + 3 * kTeams + 1) * 8 + 8 <= kBarrierBytes,
              "barrier region");
__host__ __device__ constexpr int smem_bytes_w(int W) {
    return kTeams * (nib_slots(W) * kNibStage + rec_slots(W) * rec_stage_bytes(W)) + kSbBytes + kBarrierBytes +
           1024 /* alignment slack */;
}
static_assert(smem_bytes_w(16) <= 232448 && smem_bytes_w(32) <= 232448, "shared memory per CTA");
static_assert(kWeightLanes <= nib_slots(16) && kWeightLanes <= nib_slots(32) && kRecordLanes <= rec_slots(16) &&
                  kRecordLanes <= rec_slots(32),
              "a producer lane could wait on a slot two phases ahead");
static_assert(local_stages(16) <= rec_slots(16) && local_stages(32) <= rec_slots(32), "local stages fit the ring");

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

// Error-word codes of this kernel (a wait that ran out, by role).
constexpr unsigned kErrProducer = 1u, kErrIssuer = 2u, kErrConsumer = 4u, kErrRecords = 8u;

// Call counters in scratch (zero between launches).
constexpr int kCtlBuilt = 0;     // shared x records built in this call
constexpr int kCtlSeen = 1;      // CTAs whose record readers have all seen them complete
constexpr int kCtlWords = 4;

struct Params {
    const uint8_t* W;           // packed weights
    float* y;                   // [M, N]
    const uint16_t* x;          // bf16 [M, K]
    float* partials;            // scratch: [R][2][W][128]
    int* sems;                  // scratch: [R][4] tile-quarter counters, zero between launches
    uint8_t* xt;                // scratch: the call's x records [G][rec_bytes(W)]
    unsigned int* ctl;          // scratch: call counters [kCtlWords], zero between launches
    unsigned int* error_word;   // set on a timed-out wait
    int64_t N;
    int64_t K;
    int M;
    int G;                      // K / 64
    int GP;                     // G / 2 group pairs (stages per tile)
    int T;                      // tiles of 128 rows
    int U;                      // T * GP units
    int C;                      // CTAs (grid size)
    int R;                      // ranges (at most 3 * C; team j of CTA c runs range 3c + j)
    int S;                      // ranges per block of L units
    int L;                      // units per block (U: one block over all tiles; GP: one block per tile)
    int q_units;                // L / S: every range of a block has q_units units, the first rem_units one more
    int rem_units;              // L % S
    int build;                  // 1: build the x records here; 0: the preceding glue kernel wrote them
#ifdef Q4_TRACE
    unsigned long long* trace;  // developer timing trace (compiled in only with Q4_TRACE)
#endif
};

#ifdef Q4_TRACE
// globaltimer (ns) of event `ev` (0..15) of CTA c; slots 16..31 hold counters
#define Q4_TMGT(p, c, ev)                                                                \
    do {                                                                                 \
        if ((p).trace) {                                                                 \
            unsigned long long gt_;                                                      \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(gt_));                      \
            (p).trace[(c) * 32 + (ev)] = gt_;                                            \
        }                                                                                \
    } while (0)
#else
#define Q4_TMGT(p, c, ev) \
    do {                  \
    } while (0)
#endif

// Launch geometry: grid and range count from the unit count and the SM count only.
inline int grid_ctas(int U, int sm_count) {
    int c = U / kTeams;
    if (c < 1) c = 1;
    return c < sm_count ? c : sm_count;
}

// Ranges.  The U units (unit t*GP + gp: tile t, group pair gp) are cut into
// blocks of L consecutive units and every block into S ranges, the first rem of
// them q + 1 units long and the others q (q = L / S >= 1, rem = L % S): range
// r = b*S + j starts at unit b*L + j*q + min(j, rem), and ranges from R on are
// empty.  L = U, S = R is stream-K over all tiles (ranges cross tile
// boundaries); L = GP puts S ranges inside every tile.  32-bit arithmetic, at
// range boundaries only.
__host__ __device__ __forceinline__ int range_start(const Params& p, int r) {
    if (r >= p.R) return p.U;
    const int b = r / p.S, j = r - b * p.S;
    return b * p.L + j * p.q_units + (j < p.rem_units ? j : p.rem_units);
}

// The range that owns unit u (0 <= u < U).
__device__ __forceinline__ int range_of_unit(const Params& p, int u) {
    const int b = u / p.L, v = u - b * p.L;
    const int q = p.q_units, rem = p.rem_units;
    const int big = (q + 1) * rem;                  // units in the longer ranges of the block
    return b * p.S + (v < big ? v / (q + 1) : rem + (v - big) / q);
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

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned atom_add_relaxed_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_relaxed_gpu(unsigned* p, unsigned v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void record_timeout(const Params& p, unsigned int code, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(p.error_word, code);
}

#ifdef Q4_TRACE
__device__ unsigned long long q4_tm_spins[2];   // developer counters: wait-loop iterations
#endif

// Bounded wait that also gives up at once when another role has already
// given up (the whole CTA then runs to its end without further waiting).
__device__ __forceinline__ bool wait_or_abort(const Params& p, uint64_t* bar, uint32_t parity, unsigned code,
                                              volatile int* abort_flag, unsigned long long* spins = nullptr) {
    if (q4::sm100::mbar_try_wait(bar, parity)) return true;       // fast path: already complete
    if (*abort_flag) return false;
#ifdef Q4_TRACE
    if (spins) {
        const long long t0 = clock64();
        unsigned long long n = 0;
        bool ok = true;
        while (!q4::sm100::mbar_try_wait_sleep(bar, parity, 20000u)) {
            ++n;
            if (clock64() - t0 > kWaitLimit) {
                ok = false;
                break;
            }
        }
        *spins += n + 1;
        if (ok) return true;
        record_timeout(p, code, abort_flag);
        return false;
    }
#else
    (void)spins;
#endif
    // suspended in the hardware between checks; another role's abort ends the wait too
    const long long t0 = clock64();
    while (!q4::sm100::mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimit) {
            record_timeout(p, code, abort_flag);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ x records
// One item of a record: row m, 8-block kc of group g.  record_load fetches its
// 8 inputs (zero for rows past M); record_item permutes them to the dequantized
// order and scales them (o), and forms the row's group sum X over the 8 blocks (in
// 8 consecutive lanes, kc = lane % 8: the 8 inputs in increasing k, then a fixed
// xor tree) -- the same operations for every M.  All 32 lanes call record_item.
__device__ __forceinline__ uint4 record_load(const uint16_t* __restrict__ x, int M, int64_t K, int g, int m, int kc) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (m < M) v = __ldcg(reinterpret_cast<const uint4*>(x + (int64_t)m * K + (int64_t)g * 64 + kc * 8));
    return v;
}

__device__ __forceinline__ void record_item(const uint4& v, uint4& o, float& X) {
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
    s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 1));
    s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 2));
    s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, 4));
    X = s;
}

// Byte offset of item (m, kc) in a record.
template <int W>
__device__ __forceinline__ int record_item_offset(int m, int kc) { return rec_b(W) + (m >> 3) * 1024 + kc * 128 + (m & 7) * 16; }

// Group g's record into global scratch by one warp (W/4 passes of 4 rows, every
// load in flight together).
template <int W>
__device__ __forceinline__ void build_record_global(const uint16_t* __restrict__ x, int M, int64_t K, int g, int lane,
                                                    uint8_t* __restrict__ xt) {
    uint8_t* rec = xt + (int64_t)g * rec_bytes(W);
    const int kc = lane & 7;
    uint4 v[W / 4];
#pragma unroll
    for (int pass = 0; pass < W / 4; ++pass) v[pass] = record_load(x, M, K, g, (lane >> 3) + 4 * pass, kc);
#pragma unroll
    for (int pass = 0; pass < W / 4; ++pass) {
        const int m = (lane >> 3) + 4 * pass;
        uint4 o;
        float X;
        record_item(v[pass], o, X);
        *reinterpret_cast<uint4*>(rec + record_item_offset<W>(m, kc)) = o;
        if (kc == 0) reinterpret_cast<float*>(rec)[m] = X;
    }
}

// The records of NS consecutive stages (group pairs gp0, gp0 + 1, ... wrapping
// at GP) into shared record slots, by a team's 128 threads (thread t: rows t / 8
// (+ 16 at W = 32), 8-block t % 8, both groups), every load in flight together.
// slot(i): shared address of stage i's record slot.
template <int W, int NS, typename SlotFn>
__device__ __forceinline__ void build_records_smem(const uint16_t* __restrict__ x, int M, int64_t K, int gp0, int GP,
                                                   int n, int t, SlotFn slot) {
    const int kc = t & 7;
    uint4 v[NS][2][W / 16];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int gp = (gp0 + i) % GP;
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int h = 0; h < W / 16; ++h)
                v[i][g][h] = i < n ? record_load(x, M, K, 2 * gp + g, (t >> 3) + 16 * h, kc) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        if (i >= n) break;
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int h = 0; h < W / 16; ++h) {
                const int m = (t >> 3) + 16 * h;
                uint4 o;
                float X;
                record_item(v[i][g][h], o, X);
                const uint32_t r = slot(i) + (uint32_t)(g * rec_bytes(W));
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(r + (uint32_t)record_item_offset<W>(m, kc)),
                             "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                             : "memory");
                if (kc == 0) asm volatile("st.shared.f32 [%0], %1;" ::"r"(r + (uint32_t)(4 * m)), "f"(X) : "memory");
            }
    }
}

// Dequantize 32 nibbles of one row (four nibble words) into 16 bf16 pairs,
// (q - c) * 2^-133 for the even inputs and (q - c) * 2^-129 for the odd ones,
// word order (k0,k4) (k1,k5) (k2,k6) (k3,k7) per 8 inputs, and store them to
// tensor-memory columns taddr .. taddr + 15 of the thread's lane.  One PTX
// sequence -- shift, AND, bf16x2 subtraction, one 16-column store -- so the
// results are formed in the store's registers.  cc0 = c * 0x00010001 (c * 2^-133
// as a bf16 pair), cc1 = cc0 << 4.
__device__ __forceinline__ void dequant32_store(uint32_t taddr, const uint4& n, uint32_t cc0, uint32_t cc1) {
    asm volatile(
        "{\n\t"
        ".reg .b32 u0, u1, u2, u3, a0, a1, a2, a3, a4, a5, a6, a7, a8, a9, a10, a11, a12, a13, a14, a15;\n\t"
        "shr.b32 u0, %1, 8;\n\t"
        "shr.b32 u1, %2, 8;\n\t"
        "shr.b32 u2, %3, 8;\n\t"
        "shr.b32 u3, %4, 8;\n\t"
        "and.b32 a0, %1, 0x000F000F;\n\t"
        "and.b32 a1, %1, 0x00F000F0;\n\t"
        "and.b32 a2, u0, 0x000F000F;\n\t"
        "and.b32 a3, u0, 0x00F000F0;\n\t"
        "and.b32 a4, %2, 0x000F000F;\n\t"
        "and.b32 a5, %2, 0x00F000F0;\n\t"
        "and.b32 a6, u1, 0x000F000F;\n\t"
        "and.b32 a7, u1, 0x00F000F0;\n\t"
        "and.b32 a8, %3, 0x000F000F;\n\t"
        "and.b32 a9, %3, 0x00F000F0;\n\t"
        "and.b32 a10, u2, 0x000F000F;\n\t"
        "and.b32 a11, u2, 0x00F000F0;\n\t"
        "and.b32 a12, %4, 0x000F000F;\n\t"
        "and.b32 a13, %4, 0x00F000F0;\n\t"
        "and.b32 a14, u3, 0x000F000F;\n\t"
        "and.b32 a15, u3, 0x00F000F0;\n\t"
        "sub.rn.bf16x2 a0, a0, %5;\n\t"
        "sub.rn.bf16x2 a1, a1, %6;\n\t"
        "sub.rn.bf16x2 a2, a2, %5;\n\t"
        "sub.rn.bf16x2 a3, a3, %6;\n\t"
        "sub.rn.bf16x2 a4, a4, %5;\n\t"
        "sub.rn.bf16x2 a5, a5, %6;\n\t"
        "sub.rn.bf16x2 a6, a6, %5;\n\t"
        "sub.rn.bf16x2 a7, a7, %6;\n\t"
        "sub.rn.bf16x2 a8, a8, %5;\n\t"
        "sub.rn.bf16x2 a9, a9, %6;\n\t"
        "sub.rn.bf16x2 a10, a10, %5;\n\t"
        "sub.rn.bf16x2 a11, a11, %6;\n\t"
        "sub.rn.bf16x2 a12, a12, %5;\n\t"
        "sub.rn.bf16x2 a13, a13, %6;\n\t"
        "sub.rn.bf16x2 a14, a14, %5;\n\t"
        "sub.rn.bf16x2 a15, a15, %6;\n\t"
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {a0, a1, a2, a3, a4, a5, a6, a7, a8, a9, a10, a11, a12, a13, "
        "a14, a15};\n\t"
        "}" ::"r"(taddr),
        "r"(n.x), "r"(n.y), "r"(n.z), "r"(n.w), "r"(cc0), "r"(cc1)
        : "memory");
}

__device__ __forceinline__ void dequant64_store(const uint4& n0, const uint4& n1, uint32_t cc0, uint32_t taddr) {
    const uint32_t cc1 = cc0 << 4;
    dequant32_store(taddr, n0, cc0, cc1);
    dequant32_store(taddr + 16u, n1, cc0, cc1);
}

// Constants of one row and group from its bf16 scale and bias (the low 16
// bits of s_bits / b_bits): c = clamp(rint(-b/s), 0, 15) (NaN -> 0),
// r = b + c*s, s * 2^33 and the bf16 pair c * 2^-133.  t = 1.5 * 2^23 - b/s
// holds rint(-b/s) in its low mantissa bits (the fp32 addition rounds to the
// nearest integer, ties to even); clamped in that form, its low byte is c.
// Any c in 0..15 keeps q - c exact; rint(-b/s) only keeps s*P and r*X small.
__device__ __forceinline__ void group_constants(uint32_t s_bits, uint32_t b_bits, float& s_fold, float& r,
                                                uint32_t& cc0) {
    constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23
    const float s = __uint_as_float(s_bits << 16);
    const float b = __uint_as_float(b_bits << 16);
    float t = __fmaf_rn(-b, __fdividef(1.0f, s), kMagic);
    t = fminf(fmaxf(t, kMagic), kMagic + 15.0f);
    r = __fmaf_rn(t - kMagic, s, b);
    s_fold = s * kFoldScale;
    cc0 = prmt(__float_as_uint(t), 0u, 0x4040u);   // (c, c) as a bf16 pair of c * 2^-133
}

// acc[m] = fma(s, P[m], fma(r, X[m], acc[m])) for m < MT, the same two
// roundings in the same order for every MT.  X[m] are the record's fp32 group
// sums at shared address xs.
template <int MT>
__device__ __forceinline__ void fold_group(float (&acc)[MT], const uint32_t* P, uint32_t xs, float s, float r) {
    if (MT == 1) {
        acc[0] = __fmaf_rn(s, __uint_as_float(P[0]), __fmaf_rn(r, __uint_as_float(lds32(xs)), acc[0]));
    } else if (MT == 2) {
        const float x0 = __uint_as_float(lds32(xs)), x1 = __uint_as_float(lds32(xs + 4));
        fma2(acc[0], acc[1], r, x0, x1);
        fma2(acc[0], acc[1], s, __uint_as_float(P[0]), __uint_as_float(P[1]));
    } else {
#pragma unroll
        for (int m4 = 0; m4 < MT / 4; ++m4) {
            const uint4 v = lds128(xs + 16 * m4);
            const int m = 4 * m4;
            fma2(acc[m], acc[m + 1], r, __uint_as_float(v.x), __uint_as_float(v.y));
            fma2(acc[m], acc[m + 1], s, __uint_as_float(P[m]), __uint_as_float(P[m + 1]));
            fma2(acc[m + 2], acc[m + 3], r, __uint_as_float(v.z), __uint_as_float(v.w));
            fma2(acc[m + 2], acc[m + 3], s, __uint_as_float(P[m + 2]), __uint_as_float(P[m + 3]));
        }
    }
}

// The last contributor to a partial tile: add the partials of every
// contributing range in increasing range order and store the warp's 32 rows of
// y.  Kept out of line (rare); it takes no reference to the caller's sums.
template <int MT>
__device__ __noinline__ void finish_tile(const float* __restrict__ partials, float* __restrict__ y, int64_t N, int M,
                                         int t, int row, int r_first, int r_last, bool first_before) {
    constexpr int W = width<MT>();
    const int64_t n = (int64_t)t * kRowsTile + row;
    float v[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) v[m] = 0.0f;
    // ranges in increasing order, kB at a time with their loads in flight together
    constexpr int kB = MT <= 8 ? 4 : 2;
    for (int rb = r_first; rb <= r_last; rb += kB) {
        float pv[kB][MT];
#pragma unroll
        for (int i = 0; i < kB; ++i) {
            const int rr = rb + i;
            const bool use = rr <= r_last;
            // slot 0: the tile is rr's first segment; 1: its last (only r_first can
            // have started in an earlier tile)
            const int cslot = (rr == r_first && first_before) ? 1 : 0;
            const float* src = partials + (((int64_t)rr * 2 + cslot) * W) * kRowsTile + row;
#pragma unroll
            for (int m = 0; m < MT; ++m) pv[i][m] = use ? __ldcg(src + m * kRowsTile) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < kB; ++i) {
            if (rb + i > r_last) break;
#pragma unroll
            for (int m = 0; m < MT; ++m) v[m] = __fadd_rn(v[m], pv[i][m]);
        }
    }
    if (n < N) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (m < M) y[(int64_t)m * N + n] = v[m];
    }
}

// End of a tile segment for one warp (32 rows of tile t).  A whole tile goes
// straight to y.  A partial one is published in the range's slot (0: the
// range's first segment, 1: its last) and counted on the tile's quarter
// counter; the last contributor to arrive finishes the tile.  Warp-uniform
// arguments.
template <int MT>
__device__ __forceinline__ void end_segment(const Params& p, float (&acc)[MT], int t, bool whole, int slot, int r,
                                            int q, int lane, bool live) {
    constexpr int W = width<MT>();
    const int row = q * 32 + lane;
    const int64_t n = (int64_t)t * kRowsTile + row;
    if (whole) {
        if (live && n < p.N) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < p.M) p.y[(int64_t)m * p.N + n] = acc[m];
        }
    } else if (live) {
        float* dst = p.partials + (((int64_t)r * 2 + slot) * W) * kRowsTile + row;
#pragma unroll
        for (int m = 0; m < MT; ++m) __stcg(dst + m * kRowsTile, acc[m]);
        // the warp barrier orders every lane's partial stores before lane 0's
        // release (acq_rel) increment; the last contributor's acquire, followed
        // by the next warp barrier, orders the other ranges' partials before
        // every lane's reads in finish_tile
        __syncwarp();
        const int tu = t * p.GP;
        const int r_first = range_of_unit(p, tu);
        const int r_last = range_of_unit(p, tu + p.GP - 1);
        const int count = r_last - r_first + 1;        // ranges contributing to tile t (none of them empty)
        int last = 0;
        if (lane == 0) {
            int* sem = p.sems + r_first * 4 + q;
            int old;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(sem) : "memory");
            if (old == count - 1) {
                asm volatile("st.relaxed.gpu.global.s32 [%0], 0;" ::"l"(sem) : "memory");   // zero for the next launch
                last = 1;
            }
        }
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        __syncwarp();
        if (last) finish_tile<MT>(p.partials, p.y, p.N, p.M, t, row, r_first, r_last, range_start(p, r_first) < tu);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
q4_tm_kernel(const __grid_constant__ CUtensorMap map_nib, const __grid_constant__ CUtensorMap map_sb, const Params p) {
    using namespace q4::sm100;
    constexpr int W = width<MT>();
    constexpr int SN = nib_slots(W);
    constexpr int SR = rec_slots(W);
    constexpr int kRec = rec_bytes(W);
    constexpr int kRecB = rec_b(W);
    constexpr int kRecStage = rec_stage_bytes(W);
    constexpr int H = local_stages(W);
    constexpr uint32_t kColP = col_p(W);
    constexpr uint32_t kColsTeam = cols_team(W);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* nib = smem;                                      // [team][SN] nibble boxes
    uint8_t* rec = nib + kTeams * SN * kNibStage;             // [team][SR] two x records each
    uint8_t* sb = rec + kTeams * SR * kRecStage;              // [team][kSbBuffers][plane] scale/bias boxes
    static_assert(SN == SR, "one full barrier per stage serves both rings");
    uint64_t* fulln = reinterpret_cast<uint64_t*>(sb + kSbBytes);   // nibbles, scale/bias and records landed
    uint64_t* emptyr = fulln + kTeams * SN;                   // the stage's slots read (MMAs done, P folded)
    uint64_t* ready = emptyr + kTeams * SR;                   // [kTeams]: the team's A of a stage stored, its P free
    uint64_t* done = ready + kTeams;                          // [kTeams]: the team's MMAs of a stage complete
    uint64_t* fin = done + kTeams;                            // [kTeams]
    uint64_t* xrdy = fin + kTeams;                            // every team has loaded its first records' x
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(fin + kTeams + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c_id = blockIdx.x;

    if (threadIdx.x == 0) Q4_TMGT(p, c_id, 10);
#ifdef Q4_TRACE
    if (threadIdx.x == 0 && p.trace) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        p.trace[c_id * 32 + 25] = smid;
    }
#endif
    // the next kernel on the stream may start now
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTeams * SN; ++i) {
            mbar_init(&fulln[i], 1);
        }
        for (int i = 0; i < kTeams * SR; ++i) {
            mbar_init(&emptyr[i], 4);
        }
        for (int i = 0; i < kTeams; ++i) {
            mbar_init(&ready[i], 4);
            mbar_init(&done[i], 1);
            mbar_init(&fin[i], 1);
        }
        mbar_init(xrdy, kTeams);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_nib);
        prefetch_tensormap(&map_sb);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_slot;
    if (threadIdx.x == 0) Q4_TMGT(p, c_id, 0);

    if (warp == 0) {
        // ------------------------------------------------------------ producers
        // One thread keeps only about one TMA operation in flight at a time, so the
        // streams are spread over 12 lanes of this warp: kWeightLanes per team issue
        // its weights (the nibble box, and at the first stage of each block of 8
        // groups one box of its scale and bias words), kRecordLanes per team copy the
        // records of its stages from the call's shared records (all but the first
        // local_stages, which the team builds itself).  Lane p of a stream issues the
        // team's stages k with k % lanes = p.  All lanes run one polling loop (no lane
        // sleeps in a wait that would hold the others back): each tests its next slot
        // and issues when it is free.
        constexpr int kWL = kTeams * kWeightLanes;
        const bool active = lane < kWL + kTeams * kRecordLanes;
        const bool weights = lane < kWL;
        const int j = weights ? lane / kWeightLanes : (lane - kWL) / kRecordLanes;
        const int par = weights ? lane % kWeightLanes : (lane - kWL) % kRecordLanes;
        const int step = weights ? kWeightLanes : kRecordLanes;
        const int S = weights ? SN : SR;
        const int u0 = active ? range_start(p, kTeams * c_id + j) : 0;
        const int nst = active ? range_start(p, kTeams * c_id + j + 1) - u0 : 0;
        const int h_loc = p.build ? (nst < H ? nst : H) : 0;     // stages whose records the team builds
        uint64_t* fullb = fulln + j * SN;                    // weights and records of a stage land on one barrier
        uint64_t* emptyb = emptyr + j * SR;                  // both slots of a stage are freed together
        int k = weights ? par : h_loc + ((par - h_loc) % step + step) % step;
        if (!active) k = 0;
        // the tile and group pair of this lane's next stage, advanced by step (< GP)
        // per issue: no division in the loop
        int cur_t = (u0 + k) / p.GP, cur_gp = (u0 + k) - cur_t * p.GP;
        int slot = k % S;
        uint32_t ph = (uint32_t)((k / S) & 1);       // phase of this lane's next stage in its slot
        const uint64_t pol = policy_evict_first();
        auto issue = [&]() {
            const int t = cur_t, gp = cur_gp;
            if (weights) {
                const int u = u0 + k;
                const bool sb_new = k == 0 || (gp & 3) == 0;   // GP is a multiple of 4
                // the one arrival of the stage's phase; it also expects the record copy
                // (stages from h_loc on), which may land before or after it
                mbar_arrive_expect_tx(&fullb[slot], (uint32_t)(kNibStage + (sb_new ? 2 * kSbBox : 0) +
                                                               (k >= h_loc ? 2 * kRec : 0)));
                tma_load_2d_hint(nib + (j * SN + slot) * kNibStage, &map_nib, &fullb[slot], gp * 64, t * kRowsTile, pol);
                if (sb_new) {
                    const int buf = ((u >> 2) - (u0 >> 2)) & (kSbBuffers - 1);
                    tma_load_3d_hint(sb + (j * kSbBuffers + buf) * 2 * kSbBox, &map_sb, &fullb[slot], 8 * (gp >> 2),
                                     t * kRowsTile, 0, pol);
                }
            } else {
                (void)t;
                bulk_copy_g2s(rec + (j * SR + slot) * kRecStage, p.xt + (int64_t)(2 * gp) * kRec, (uint32_t)(2 * kRec),
                              &fullb[slot]);
            }
            k += step;
            cur_gp += step;
            if (cur_gp >= p.GP) {
                cur_gp -= p.GP;
                ++cur_t;
            }
            slot += step;
            if (slot >= S) {                          // step < S: one wrap at most
                slot -= S;
                ph ^= 1u;
            }
        };
        // the weights' first stages need nothing from the preceding kernel
        if (active && weights)
            while (k < nst && k < kEarlyStages) issue();
        bool x_loaded = false;                        // weight lanes: every team has loaded its x
        // the records come from this call (or from the preceding glue kernel)
        pdl_wait();
        if (lane == 0) Q4_TMGT(p, c_id, 1);
        bool ok = true;
        // The shared records of the call: every record lane, and one counting lane,
        // waits until they are complete; then the CTA counts itself once on
        // ctl[kCtlSeen], and the last CTA counted returns both counters to zero for
        // the next call -- all during the call, off its critical path.
        constexpr int kCountLane = 31;
        const bool poller = p.build && (lane == kCountLane || (active && !weights));
        bool records_ok = !poller;                    // this lane has seen the call's records complete
        bool counted = !p.build;                      // warp-uniform: this CTA is counted
        unsigned seen_before = 0xFFFFFFFFu;           // the counting lane's ticket
        long long idle_since = clock64();
        while (true) {
            const bool more = active && ok && k < nst;
            if (!__any_sync(0xFFFFFFFFu, more || (ok && !counted))) break;
            if (ok && !records_ok) {
                if (ld_acquire_gpu(p.ctl + kCtlBuilt) >= (unsigned)p.G) {
                    // written through the generic proxy, read by the bulk copies through the async one
                    fence_proxy_async_global();
                    records_ok = true;
                    if (lane == kWL) Q4_TMGT(p, c_id, 2);
                }
            }
            if (!counted && __all_sync(0xFFFFFFFFu, records_ok)) {
                if (lane == kCountLane) seen_before = atom_add_relaxed_gpu(p.ctl + kCtlSeen, 1u);
                counted = true;
            }
            if (weights && !x_loaded) x_loaded = mbar_test_wait(xrdy, 0u);
            bool issued = false;
            if (more && (weights ? (k < kEarlyStages || x_loaded) : records_ok) &&
                (k < S || mbar_test_wait(&emptyb[slot], ph ^ 1u))) {
                issue();
                issued = true;
            }
            if (__any_sync(0xFFFFFFFFu, issued)) {
                idle_since = clock64();
            } else {
                if (*abort_flag) {
                    ok = false;
                } else if (clock64() - idle_since > kWaitLimit) {
                    if (lane == 0) record_timeout(p, kErrProducer, abort_flag);
                    ok = false;
                } else {
                    __nanosleep(64);
                }
            }
        }
        // the ticket is read only now, so its round trip never held up a copy; every
        // other CTA counted has seen the records complete, so nothing reads or adds
        // to the counters again in this call
        if (lane == kCountLane && seen_before == (unsigned)p.C - 1) {
            st_relaxed_gpu(p.ctl + kCtlBuilt, 0u);
            st_relaxed_gpu(p.ctl + kCtlSeen, 0u);
        }
        if (!ok && active) {
            // every issued copy must land before the CTA may exit (a stage whose other
            // part was never issued keeps its phase open: the wait then runs to its limit)
            const int first = weights ? par : h_loc + ((par - h_loc) % step + step) % step;
            for (int k2 = k - step; k2 >= first && k2 + S >= k; k2 -= step)
                mbar_wait(&fullb[k2 % S], (uint32_t)((k2 / S) & 1), kWaitLimit);
        }
    } else if (warp <= kTeams) {
        // ------------------------------------------------------------ MMA issuers (warp-uniform loop)
        const int team = warp - 1;
        const int u0 = range_start(p, kTeams * c_id + team);
        const int nst = range_start(p, kTeams * c_id + team + 1) - u0;
        // first, this CTA's share of the call's x records (groups c, c + C, ...; this
        // warp takes every third of them), counted once written
        if (p.build) {
            pdl_wait();
            int nb = 0;
            for (int g = c_id + team * p.C; g < p.G; g += kTeams * p.C) {
                build_record_global<W>(p.x, p.M, p.K, g, lane, p.xt);
                ++nb;
            }
            __syncwarp();
            if (lane == 0 && nb > 0) {
                fence_proxy_async_global();
                red_release_gpu_add(p.ctl + kCtlBuilt, (unsigned)nb);
            }
        }
        const uint32_t idesc = idesc_bf16_f32(128, 16);
        // B: core matrices K-major, 128 B apart along K, 8-row blocks 1024 B apart
        const uint64_t bdesc0 = smem_desc_noswizzle(smem_u32(rec + team * SR * kRecStage + kRecB), 128, 1024);
        // the tensor-memory base is the same in every lane: take lane 0's, so the
        // operand arithmetic below is visibly warp-uniform
        const uint32_t tbase = __shfl_sync(0xFFFFFFFFu, tmem, 0) + (uint32_t)team * kColsTeam;
        const uint32_t leader = elect_one();           // the lane that issues (and commits) every MMA
        int rs = 0;
        for (int k = 0; k < nst; ++k) {
            // the team hands a stage over only once its records are in shared memory
            if (!__all_sync(0xFFFFFFFFu, wait_or_abort(p, &ready[team], (uint32_t)(k & 1), kErrIssuer, abort_flag)))
                break;
            tc_fence_after();
            const uint64_t bd = bdesc0 + (uint64_t)((rs * kRecStage) >> 4);
            const uint32_t aS = tbase + (a_buffers(W) == 2 ? (uint32_t)(k & 1) * kColsA : 0u);
            const uint32_t dS = tbase + kColP;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const uint64_t bg = bd + (uint64_t)((g * kRec) >> 4);
                // P of group g: columns W*g + m (rows 0-15 in one N = 16 MMA, rows 16-31 in another)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                    for (int h = 0; h < W / 16; ++h)
                        tc_mma_ts_if(leader, dS + (uint32_t)(W * g + 16 * h), aS + 32u * g + 8u * kk,
                                     bg + 16u * kk + (uint64_t)(h * (2048 >> 4)), idesc, kk > 0 ? 1u : 0u);
                }
            }
            tc_commit_if(leader, &done[team]);
            __syncwarp();
            if (++rs == SR) rs = 0;
        }
        // no MMA of this warp may still run when tensor memory is freed
        tc_commit_if(leader, &fin[team]);
        if (leader) mbar_wait(&fin[team], 0, kWaitLimit);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumer teams
        const int team = (warp - kConsumerWarp0) >> 2;
        const int q = warp & 3;                        // tensor-memory lane quarter of this warp
        const int row = q * 32 + lane;                 // row within the tile (and thread within the team)
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)team * kColsTeam;
        const uint32_t dP = tbase + kColP;
        const int r_id = kTeams * c_id + team;
        const int u0 = range_start(p, r_id);
        const int nst = range_start(p, r_id + 1) - u0;
        const int h_loc = p.build ? (nst < H ? nst : H) : 0;
        // shared addresses: this team's first nibble slot (its row), first record
        // slot, first scale/bias buffer (its row's 16 bytes)
        const uint32_t nib0 = smem_u32(nib) + (uint32_t)(team * SN * kNibStage + row * 64);
        const uint32_t rec0 = smem_u32(rec) + (uint32_t)(team * SR * kRecStage);
        const int sx = (row >> 1) & 3;                 // 64-byte swizzle: chunk index ^ bits 7-8 of the offset
        const uint32_t sb_row = smem_u32(sb) + (uint32_t)(team * kSbBuffers * 2 * kSbBox + row * 16);

        // the predecessor may still read y or the scratch, or produce x
        pdl_wait();
        if (team == 0 && q == 0 && lane == 0) Q4_TMGT(p, c_id, 14);
        if (h_loc > 0) {
            // the records of the team's first stages, from x, while the call's shared ones are built
            build_records_smem<W, H>(p.x, p.M, p.K, u0 % p.GP, p.GP, h_loc, row,
                                     [&](int i) { return rec0 + (uint32_t)(i * kRecStage); });
            fence_proxy_async_smem();                  // for the MMAs (async proxy)
            named_barrier(1 + team, 128);              // every row's X before any warp's fold
        }
        if (team == 0 && q == 0 && lane == 0) Q4_TMGT(p, c_id, 15);
        if (q == 0 && lane == 0) mbar_arrive(xrdy);   // this team's x loads are done (every team arrives once)

        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
        bool live = true;

        // cursor of the stage being dequantized: ring positions, tile, group pair
        int ns = 0, rs = 0;
        uint32_t nph = 0;
        int st_t = u0 / p.GP, st_gp = u0 - st_t * p.GP;
        int seg_first_gp = st_gp;                      // group pair at which the current segment started
        bool first_seg = true;

        // the stage handed over in the previous iteration, folded in this one
        int pend = -1, pend_t = 0, pend_gp = 0, pend_rs = 0;
        float s0 = 0.f, r0 = 0.f, s1 = 0.f, r1 = 0.f;  // constants of the stage being dequantized
        float ps0 = 0.f, pr0 = 0.f, ps1 = 0.f, pr1 = 0.f;

#ifdef Q4_TRACE
        const bool tr = team == 0 && q == 0 && lane == 0 && p.trace;
        unsigned long long tr_spin = 0, tr_c[6] = {0, 0, 0, 0, 0, 0};
        long long tr_t = clock64();
        auto tr_mark = [&](int i) {
            const long long t = clock64();
            tr_c[i] += (unsigned long long)(t - tr_t);
            tr_t = t;
        };
        unsigned long long* tr_sp = tr ? &tr_spin : nullptr;
#else
        auto tr_mark = [&](int) {};
        unsigned long long* tr_sp = nullptr;
#endif
        auto arrive_ready = [&]() {
            tc_fence_before();
            __syncwarp();
            mbar_arrive_elected(&ready[team]);
        };
        // fold the pending stage (signal_ready: hand the current stage over as
        // soon as P is in registers), free its record slot, close its segment if it ends one
        auto fold_pending = [&](bool signal_ready) {
            tr_mark(5);
            live = __all_sync(0xFFFFFFFFu, live && wait_or_abort(p, &done[team], (uint32_t)(pend & 1), kErrConsumer,
                                                                 abort_flag, tr_sp));
            tr_mark(2);
            if (live) {
                tc_fence_after();
                const uint32_t xs0 = rec0 + (uint32_t)(pend_rs * kRecStage);
                const uint32_t xs1 = xs0 + (uint32_t)kRec;
                if (MT <= 8) {
                    uint32_t P0[8], P1[8];
                    tmem_ld_32x32b_x8(dP, P0);
                    tmem_ld_32x32b_x8(dP + 16u, P1);
                    tmem_wait_ld();
                    if (signal_ready) arrive_ready();
                    fold_group<MT>(acc, P0, xs0, ps0, pr0);
                    fold_group<MT>(acc, P1, xs1, ps1, pr1);
                } else if (W == 32) {
                    uint32_t P[32];
                    tmem_ld_32x32b_x32(dP, P);
                    tmem_wait_ld();
                    fold_group<MT>(acc, P, xs0, ps0, pr0);
                    tmem_ld_32x32b_x32(dP + 32u, P);
                    tmem_wait_ld();
                    if (signal_ready) arrive_ready();
                    fold_group<MT>(acc, P, xs1, ps1, pr1);
                } else {
                    uint32_t P[32];                    // both groups' 16 columns, one load
                    tmem_ld_32x32b_x32(dP, P);
                    tmem_wait_ld();
                    if (signal_ready) arrive_ready();
                    fold_group<MT>(acc, P, xs0, ps0, pr0);
                    fold_group<MT>(acc, P + 16, xs1, ps1, pr1);
                }
            } else if (signal_ready) {
                arrive_ready();
            }
            // that stage's records have been read (by the MMAs and the fold: every value
            // it loaded has been used), and so has P
            tc_fence_before();
            __syncwarp();
            mbar_arrive_relaxed_elected(&emptyr[team * SR + pend_rs]);
            tr_mark(3);
            if (pend_gp == p.GP - 1 || pend == nst - 1) {
                const bool whole = seg_first_gp == 0 && pend_gp == p.GP - 1;
                end_segment<MT>(p, acc, pend_t, whole, first_seg ? 0 : 1, r_id, q, lane, live && !*abort_flag);
                if (first_seg && q == 0 && lane == 0) Q4_TMGT(p, c_id, 11 + team);
                first_seg = false;
                seg_first_gp = 0;
            }
        };

        for (int k = 0; k < nst; ++k) {
            tr_mark(5);
            live = __all_sync(0xFFFFFFFFu, live && wait_or_abort(p, &fulln[team * SN + ns], nph, kErrConsumer,
                                                                 abort_flag, tr_sp));
            tr_mark(0);
            if (k == 0 && q == 0 && lane == 0) Q4_TMGT(p, c_id, 3 + team);
            // scale and bias of this stage's two groups: word st_gp % 4 of the buffer of its block
            const int sbuf = (((u0 + k) >> 2) - (u0 >> 2)) & (kSbBuffers - 1);
            const uint32_t a = sb_row + (uint32_t)(sbuf * 2 * kSbBox + (st_gp & 3) * 4);
            const uint32_t sw = lds32(a), bw = lds32(a + kSbBox);
            uint32_t cc0, cc1;
            group_constants(sw, bw, s0, r0, cc0);
            group_constants(sw >> 16, bw >> 16, s1, r1, cc1);
            // one A buffer (W = 32): the previous stage's MMAs must have read it, so fold first
            if (a_buffers(W) == 1 && pend >= 0) fold_pending(false);
            const uint32_t nb = nib0 + (uint32_t)(ns * kNibStage);
            const uint4 w0 = lds128(nb + ((0 ^ sx) << 4)), w1 = lds128(nb + ((1 ^ sx) << 4));
            const uint4 w2 = lds128(nb + ((2 ^ sx) << 4)), w3 = lds128(nb + ((3 ^ sx) << 4));
            if (live) {
                const uint32_t aA = tbase + (a_buffers(W) == 2 ? (uint32_t)(k & 1) * kColsA : 0u);
                dequant64_store(w0, w1, cc0, aA);
                dequant64_store(w2, w3, cc1, aA + 32u);
                tmem_wait_st();
            }
            tr_mark(1);
            // (the stage's records -- copied ones landed on the same barrier as its
            // weights, built ones were written before the loop -- are in place)
            tr_mark(4);
            // fold the previous stage (its MMAs ran meanwhile); then P is free again
            const bool early = a_buffers(W) == 2 && pend >= 0;
            if (early) fold_pending(true);
            if (!early) arrive_ready();
            // this stage becomes the pending one
            pend = k;
            pend_t = st_t;
            pend_gp = st_gp;
            pend_rs = rs;
            ps0 = s0;
            pr0 = r0;
            ps1 = s1;
            pr1 = r1;
            if (++st_gp == p.GP) {
                st_gp = 0;
                ++st_t;
            }
            if (++ns == SN) {
                ns = 0;
                nph ^= 1u;
            }
            if (++rs == SR) rs = 0;
        }
        if (pend >= 0) fold_pending(false);
        if (q == 0 && lane == 0) Q4_TMGT(p, c_id, 6 + team);
#ifdef Q4_TRACE
        if (tr) {
            p.trace[c_id * 32 + 16] = tr_spin;
            for (int i = 0; i < 6; ++i) p.trace[c_id * 32 + 18 + i] = tr_c[i];
            p.trace[c_id * 32 + 24] = (unsigned long long)nst;
        }
#endif
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0) Q4_TMGT(p, c_id, 9);
}

template <int MT>
inline int smem_bytes() { return smem_bytes_w(width<MT>()); }
inline size_t partial_floats(int C) { return (size_t)kTeams * C * 2 * 32 * kRowsTile; }   // sized for W = 32
inline size_t sem_ints(int C) { return (size_t)kTeams * C * 4; }

}  // namespace tm
}  // namespace q4
