/*
 * q4.h -- C ABI of the GB300 Q4 verify-matmul library (libq4.so).
 *
 * The operation.  A speculative-decoding verify pass multiplies M = 1..32 draft
 * or tree rows against every quantized weight of a layer, reading the weights
 * from HBM once ("Faster, with the same words" (goinfer.dev), section "The
 * problem": a step that checks eight tokens costs much less than eight steps,
 * because the weights are read once; "qwen-spec" (jonasloos.github.io), Notes:
 * a 4-bit matmul that reads every weight tile once and multiplies all rows at
 * once).  For x[M,K] (bf16) and a packed Q4 matrix W[N,K]:
 *
 *     y[m,n] = sum_k x[m,k] * ( s[n,k/64] * q[n,k] + b[n,k/64] )
 *
 * Packed format ("Splash engine" analysis (ai.thesatyajit.com), section "The
 * engine hard-codes the model": nine bytes per sixteen weights -- 32 bytes of
 * unsigned nibbles plus a bf16 scale and a bf16 bias per group of 64 inputs).
 * Byte layout fixed by this library (planar, row-major), N*K/16*9 bytes:
 *     [nibbles: N rows x K/2 bytes; byte j of a row holds input 2j in bits 0-3
 *               and input 2j+1 in bits 4-7]
 *     [scales:  N rows x K/64 bf16, little-endian]
 *     [biases:  N rows x K/64 bf16, little-endian]
 *
 * Conventions for every call below:
 *   - All buffers are owned by the caller.  Device pointers must be device
 *     memory of the current CUDA device (or managed memory).
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Argument errors are detected on the host and returned before anything
 *     is launched; launch failures return Q4_ERR_CUDA.  A device-side wait
 *     that ran out of time is reported by q4_device_status().
 *   - On any status other than Q4_OK, q4_last_error() describes the failure
 *     (a thread-local string, valid until the next call on that thread).
 *   - Results are deterministic, and row m of y does not depend on M or on
 *     the contents of the other rows of x (bit-identical batched verify:
 *     "Faster, with the same words", section "How it works").
 */
#ifndef Q4_H
#define Q4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* q4_stream_t;

typedef enum {
    Q4_OK = 0,
    Q4_ERR_INVALID_ARG = 1,        /* null pointer, M out of 1..32, N < 1, ...     */
    Q4_ERR_UNSUPPORTED_SHAPE = 2,  /* K not a positive multiple of 64              */
    Q4_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned             */
    Q4_ERR_UNSUPPORTED_DEVICE = 4, /* the current device is not compute 10.3       */
    Q4_ERR_CUDA = 5,               /* a CUDA runtime call failed                   */
    Q4_ERR_TIMEOUT = 6,            /* a device-side wait gave up (q4_device_status) */
    Q4_ERR_OVERFLOW = 7,           /* a byte count does not fit in 64 bits          */
    Q4_ERR_INVALID_INDEX = 8       /* a codebook id was out of range (q4_device_status) */
} q4_status;

#define Q4_MAX_ROWS 32

/* Bytes of a packed N x K matrix: the page's q4PackedBytes -- an
 * overflow-checked (N*K/16)*9 ("Splash engine", section "The engine hard-codes
 * the model").  Returns 0 when N == 0, K is not a positive multiple of 64, or
 * the product overflows 64 bits.  Host only; never touches the GPU. */
uint64_t q4_packed_bytes(uint64_t N, uint64_t K);

/* y[M,N] = x[M,K] * W[N,K]^T with W dequantized as above.
 *   x : device, bf16, row-major [M, K], 16-byte aligned.
 *   W : device, packed buffer of exactly q4_packed_bytes(N, K) bytes, 16-byte aligned.
 *   M : 1..32 verify rows (the pages' kernels exist for 8, 16, 24 and 32 rows:
 *       up to four lanes of eight; "Splash engine", section "The decode step
 *       is one command buffer").   N : >= 1 outputs.   K : positive multiple of 64.
 *   y : device, fp32, row-major [M, N], 16-byte aligned; fully overwritten.
 * Row invariance: row m of y is bit-identical for every M (1..32) and every
 * other row's contents.
 * Device memory: the first call on each device (with that device current)
 * allocates the library's scratch -- split-K partial sums, per-tile and
 * per-call counters and the call's x records, about 25 MB on a 152-SM GPU --
 * and keeps it until the process exits; later calls allocate nothing.  Make
 * that first call outside any stream capture.  Every call on a device shares
 * this scratch, so calls that may run at the same time on one device (different
 * streams without an ordering between them) race and give wrong results: order
 * them on one stream or with events.
 * Ordering: the kernel is launched with programmatic dependent launch.  It
 * loads the first boxes of W before the preceding kernel on `stream` has
 * finished; x, y and the scratch only afterwards.  So W must not be written by
 * a preceding kernel that lets its dependents start early
 * (griddepcontrol.launch_dependents): ordinary kernels finish first.
 * Residency: the kernel runs one CTA per SM and its CTAs exchange the call's x
 * records, so all of them must be resident at once.  A context that gets fewer
 * SMs than the device reports (an MPS client limited to a share of the SMs, for
 * example) can leave a CTA waiting for one that never starts; the wait gives up
 * after about a second and q4_device_status() reports Q4_ERR_TIMEOUT.
 * Accuracy: |y - exact| <= 2e-3 * sum_k |x[m,k] w[n,k]| per output, for
 * activations with |x| < 2^28 whose nonzero values are at least 2^-93 in
 * magnitude, and scales with |s| < 2^95 (the tensor core sees x scaled by
 * 2^100 or 2^96 and products scaled by 2^-33: outside that range they overflow
 * or fall below the fp32 normal range). */
q4_status q4_matmul(const void* x, const void* W, int M, int64_t N, int64_t K, float* y,
                    q4_stream_t stream);

/* q4_matmul for callers that must not allocate device memory.  The pages have
 * no counterpart to this call; it exists for callers such as a serving
 * engine that hands all free HBM to its own pools at start-up, a plug-in
 * that runs inside a host application owning the device allocator, or a
 * latency-critical loop that cannot afford cudaMalloc's implicit device
 * synchronisation.
 *   Arguments, layout and the accuracy bound are those of q4_matmul, except
 *   that M is limited to 1..16; the caller still owns x, W and y.  Rows are
 *   bit-identical for every M and across runs, as with q4_matmul, but this call
 *   runs a different kernel, so its bits may differ from q4_matmul's.  K is
 *   limited to 20480 and the device to 160 SMs (larger:
 *   Q4_ERR_UNSUPPORTED_SHAPE / Q4_ERR_UNSUPPORTED_DEVICE, nothing launched).
 *   Scratch: a fixed array of 8,542,208 bytes inside the library's device
 *   image, which every device that loads the library holds until the process
 *   exits.  No call allocates or frees device memory, and neither does
 *   q4_device_status().  The first call on a device, with that device current,
 *   looks up the array's device address and sets kernel attributes; make that
 *   first call before any stream capture.
 *   Every call clears the counters it needs at zero (an asynchronous memset
 *   on `stream`) and overwrites the rest before reading it.
 *   All calls on one device share the one array, so calls that may run at the
 *   same time on the GPU (different streams with no ordering between them)
 *   race and give wrong results: order them on one stream or with events. */
q4_status q4_matmul_noalloc(const void* x, const void* W, int M, int64_t N, int64_t K, float* y,
                            q4_stream_t stream);

/* How the output y_j of one layer of a chained verify pass becomes the input
 * x_{j+1} of the next.  The pages' own between-layer operators (attention,
 * Gated DeltaNet, gated norms) are outside the matmul path; this library joins
 * layers with a fixed, bounded stand-in ("Splash engine" analysis, section
 * "The decode step is one command buffer": one submission runs every layer of
 * the step in order):
 *   RMSNORM:        v_k = y[m, k] for the first K_next columns (K_next <= N_prev)
 *   SWIGLU_RMSNORM: v_k = silu(y[m, k]) * y[m, K_next + k]       (N_prev == 2 K_next)
 *   x[m, k] = bf16_RNE( v_k / sqrt( mean_k v_k^2 + 1e-6 ) ),  silu(a) = a / (1 + e^-a)
 * Accuracy: the sum of squares is carried in about 48 bits and the scale formed
 * as a float pair (relative error below 3e-14).  RMSNORM: the one rounding to
 * bf16 matches an all-double evaluation except where the value lies within
 * about 1e-13 of a bf16 midpoint.
 * SWIGLU: silu(a) * b is formed in fp32 (within 9 float ulps), and recomputed in
 * float pairs (about 1e-14) near a bf16 midpoint; the scale agrees with an
 * all-double one to about 1e-8 (at worst 5e-7), so an output may differ by one
 * bf16 ulp where its value lies within that distance of a midpoint. */
typedef enum {
    Q4_GLUE_NONE = 0,              /* last layer: its y is the step's output  */
    Q4_GLUE_RMSNORM = 1,
    Q4_GLUE_SWIGLU_RMSNORM = 2
} q4_glue_kind;

/* One layer of a chained pass: packed W [N, K] (device, 16-byte aligned) and
 * the glue that turns its output into the next layer's input. */
typedef struct {
    const void* W;
    int64_t N;
    int64_t K;
    int glue;                      /* q4_glue_kind; ignored for the last layer */
} q4_layer;

/* The inter-layer step alone: x_next[M, K_next] (bf16, device) from y[M, N_prev]
 * (fp32, device), as described above.  Both 16-byte aligned.  K_next: a
 * multiple of 64 (the K of the next matmul), else Q4_ERR_UNSUPPORTED_SHAPE.
 * Asynchronous on `stream`; the kernel waits for the preceding kernel on the
 * stream (it may be the matmul that writes y).  Provided so that a chained
 * pass can be run and checked one layer at a time. */
q4_status q4_glue(const float* y, int M, int64_t N_prev, int64_t K_next, int glue, void* x_next,
                  q4_stream_t stream);

/* Bytes of workspace q4_decode_step needs for this layer list and M: one fp32
 * buffer for the widest intermediate output and one bf16 buffer for the widest
 * intermediate input.  0 for an invalid list (or a single layer). */
size_t q4_decode_step_workspace_bytes(const q4_layer* layers, int n_layers, int M);

/* One decode step of the chained verify pass in one submission ("Splash
 * engine", section "The decode step is one command buffer"): for j = 0..n-1,
 * y_j = x_j * W_j^T (as q4_matmul) and x_{j+1} = glue_j(y_j); the last layer
 * writes y_last [M, N_{n-1}] (fp32, device, 16-byte aligned).  x0 is bf16
 * [M, K_0] on the device.  Every kernel is chained with programmatic dependent
 * launch, so layer j+1 starts streaming its weights while layer j finishes.
 * The whole list is checked before anything is launched (Q4_ERR_INVALID_ARG
 * names the first bad layer); `workspace` (device, 16-byte aligned, at least
 * q4_decode_step_workspace_bytes) holds the intermediates and must not overlap
 * x0 or y_last.  Asynchronous on `stream`; the same scratch rules as q4_matmul
 * apply, and the call may be captured in a CUDA graph once the device has been
 * set up by an earlier call. */
q4_status q4_decode_step(const q4_layer* layers, int n_layers, const void* x0, int M, void* workspace,
                         size_t workspace_bytes, float* y_last, q4_stream_t stream);

/* Sampling epilogue of the LM head ("Splash engine" analysis, section "Exact,
 * up to top-32": the target's probabilities are the temperature softmax over
 * its first top_k entries, truncated by top_p, renormalized; top_k <= 32).
 *   logits : device, fp32 [M, N] row-major (e.g. the y of the LM-head matmul).
 *   M : 1..32.  N : top_k .. 1,048,576.  top_k : 1..32.  temperature > 0.
 *   top_p > 0 (>= 1 keeps all top_k entries).
 *   idx   : device, int32 [M, 32]: the top_k entries of each row by logit,
 *           largest first, equal logits by lower index first (so the result is
 *           unique); -1 past top_k.
 *   probs : device, fp32 [M, 32]: p_j = exp((l_j - l_0)/T) / sum over the
 *           top_k; the shortest prefix whose cumulative probability reaches
 *           top_p is kept and renormalized; 0 for the rest.  Computed in
 *           float pairs (about 48 significant bits, so they round as
 *           double-precision values would; an exponential below e^-60 in
 *           double).
 * All pointers 16-byte aligned.  Asynchronous on `stream`; uses the library's
 * per-device scratch (the same ordering rules as q4_matmul). */
q4_status q4_topk_probs(const float* logits, int M, int64_t N, int top_k, float temperature, float top_p,
                        int32_t* idx, float* probs, q4_stream_t stream);

/* The LM head with its sampling epilogue fused: q4_matmul of x[M,K] against
 * the packed head W[N,K] into the library's own logits scratch, then the
 * q4_topk_probs epilogue on those logits ("Splash engine" analysis, section
 * "Exact, up to top-32": top-32 sampling follows the head in the same step).
 * The logits never leave the GPU's L2: as each epilogue CTA finishes reading
 * its slice it invalidates those cache lines without writing them back, so the
 * M*N*4 bytes of logits are not written to HBM (when they are still resident).
 *   Arguments and results are those of q4_matmul (x, W, M, N, K) and of
 *   q4_topk_probs (top_k, temperature, top_p, idx, probs); idx and probs are
 *   bit-identical to q4_matmul followed by q4_topk_probs.
 * Device memory: the first call for a given N allocates a logits scratch of
 * 32*N*4 bytes on the current device (grown, never shrunk, held until exit);
 * make that call outside any stream capture.  The same scratch rules as
 * q4_matmul apply to concurrent calls. */
q4_status q4_lm_head_topk(const void* x, const void* W, int M, int64_t N, int64_t K, int top_k, float temperature,
                          float top_p, int32_t* idx, float* probs, q4_stream_t stream);

/* Edge scores of the draft selector ("Splash engine" analysis, section "The
 * draft is a small model with an unusual selector": the top 16 candidates of
 * each draft position are scored against 16 predecessors by a trilinear form
 * over two bf16 codebooks of vocabulary x 256).  For row r (one draft position
 * of one lane), predecessor i and candidate j:
 *   score[r][i][j] = sum_{d<R} pred_cb[pred_ids[r][i]][d] * hidden[r][d]
 *                                * succ_cb[cand_ids[r][j]][d]
 *   pred_cb, succ_cb : device, bf16 [V, R] row-major (the predecessor and the
 *                      successor codebook), read only at the ids' rows.
 *   V : 1 .. 2^31-1.   R : a multiple of 8 in 8..256 (256 on the pages).
 *   hidden   : device, fp32 [rows, R] (the position's rank-R projection).
 *   pred_ids, cand_ids : device, int32 [rows, 16].
 *   rows : 1 .. 2^20.
 *   score    : device, fp32 [rows, 16, 16] (written; caller-owned).
 * fp32 arithmetic: the context pred * hidden rounded once, then fused
 * multiply-adds in a fixed order; |error| <= (R/4 + 3) * 2^-24 * the sum over d
 * of |term|.  Each row's scores depend on that row's inputs only.  An id
 * outside 0..V-1 is not read (its codebook row counts as zeros) and the next
 * q4_device_status() returns Q4_ERR_INVALID_INDEX.  All pointers 16-byte
 * aligned.  Asynchronous on `stream`; no scratch. */
q4_status q4_draft_select_edges(const void* pred_cb, const void* succ_cb, int64_t V, int R, const float* hidden,
                                const int32_t* pred_ids, const int32_t* cand_ids, int rows, float* score,
                                q4_stream_t stream);

/* Self-check of the timeout reporting path.  Launches one thread on `stream`
 * that waits, with the same bounded wait every kernel of this library uses, on
 * a barrier that nothing signals; after `limit_cycles` SM clock cycles
 * (1..2^32) it records the timeout in the device error word, as a kernel whose
 * wait ran out does, and exits normally -- no trap, the context stays usable.
 * The next q4_device_status() then returns Q4_ERR_TIMEOUT and clears the
 * record.  Asynchronous; Q4_ERR_INVALID_ARG for a limit out of range. */
q4_status q4_check_wait_timeout(long long limit_cycles, q4_stream_t stream);

/* Synchronizes `stream` and reports whether any kernel of this library on the
 * current device recorded a device-side failure since the last query -- an
 * out-of-range codebook id (Q4_ERR_INVALID_INDEX, reported first) or a bounded
 * wait that gave up (Q4_ERR_TIMEOUT) -- then clears that record.  After a wait
 * that gave up it also returns the library's arrival counters to zero (a CTA
 * that gave up may have skipped its arrivals), so later calls start clean;
 * results of calls made on that device between the timed-out call and this
 * query are undefined.  Allocates no device memory.  Q4_OK otherwise. */
q4_status q4_device_status(q4_stream_t stream);

/* Thread-local description of the last failure on this thread ("" if none). */
const char* q4_last_error(void);

/* Constant name of a status code. */
const char* q4_status_string(q4_status s);

#ifdef __cplusplus
}
#endif

#endif /* Q4_H */
