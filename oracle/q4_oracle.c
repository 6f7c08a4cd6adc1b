/*
 * CPU oracle for the Q4 verify matmul -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * leg may load this code.  The product path (the CUDA library) never calls it
 * and shares no code, header or table with it.
 *
 * What it computes (plain definition, written out):
 *
 *   y[m,n] = sum_{k=0}^{K-1} x[m,k] * ( s[n, k/64] * q[n,k] + b[n, k/64] )
 *
 * - Weight format: "Splash engine" analysis (ai.thesatyajit.com/articles/
 *   splash-engine), section "The engine hard-codes the model": nine bytes per
 *   sixteen weights; every group of 64 inputs carries 32 bytes of unsigned
 *   nibbles, one bf16 scale and one bf16 bias; w = scale*q + bias.
 * - Nibble order (low nibble = even input) and the planar plane order
 *   [nibbles N x K/2][scales N x K/64][biases N x K/64] are the readings this
 *   project fixes for what the page leaves open.
 * - Arithmetic: every x, s, b (bf16) widens exactly to double; w = s*q + b is
 *   exact in double (at most 8+4 and 8 significant bits); each product x*w is
 *   exact in double; only the running sum over increasing k rounds.
 *
 * The packed-size function follows the page's q4PackedBytes: an
 * overflow-checked (elements / 16) * 9.
 *
 * Threads: contiguous ranges of output columns; the per-output order never
 * depends on the thread count.  Build with -O2, never -ffast-math.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>
#include <pthread.h>

#define Q4O_GROUP 64

/* bf16 bit pattern -> double, exactly (bf16 is the upper half of an IEEE fp32). */
static double bf16_to_f64(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp64 -> bf16 bit pattern, round to nearest, ties to even, computed from the
 * exact binary value (no intermediate fp32 rounding).  NaN -> quiet NaN. */
static uint16_t f64_to_bf16_rne(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    double fr = frexp(a, &e);          /* a = fr * 2^e, fr in [0.5, 1) */
    int exp_unbiased = e - 1;          /* a = 1.xxx * 2^(e-1) */
    if (exp_unbiased < -126) exp_unbiased = -126;      /* subnormal range: fixed quantum */
    /* quantum of bf16 at this exponent: 2^(exp_unbiased - 7) */
    double q = ldexp(1.0, exp_unbiased - 7);
    double t = a / q;                  /* exact: power-of-two division */
    double fl = floor(t);
    double rem = t - fl;               /* exact */
    double r;
    if (rem > 0.5) r = fl + 1.0;
    else if (rem < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double res = r * q;                /* exact */
    (void)fr;
    if (res >= ldexp(1.0, 128)) return sign | 0x7F80;   /* overflow to inf */
    float f = (float)res;              /* exact: res has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

uint64_t q4o_packed_bytes(uint64_t N, uint64_t K) {
    if (N == 0 || K == 0 || (K % Q4O_GROUP) != 0) return 0;
    /* elements = N * K, checked */
    if (K > UINT64_MAX / N) return 0;
    uint64_t elements = N * K;
    uint64_t sixteenths = elements / 16;
    if (sixteenths > UINT64_MAX / 9) return 0;
    return sixteenths * 9;
}

/* Readers of the documented planar layout.  W points at the first byte. */
static unsigned nib(const uint8_t* W, uint64_t K, uint64_t n, uint64_t k) {
    uint8_t byte = W[n * (K / 2) + k / 2];
    return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 0x0F);
}

static double scale_at(const uint8_t* W, uint64_t N, uint64_t K, uint64_t n, uint64_t g) {
    const uint8_t* plane = W + N * (K / 2);
    uint64_t off = 2 * (n * (K / Q4O_GROUP) + g);
    uint16_t h = (uint16_t)(plane[off] | ((uint16_t)plane[off + 1] << 8));
    return bf16_to_f64(h);
}

static double bias_at(const uint8_t* W, uint64_t N, uint64_t K, uint64_t n, uint64_t g) {
    const uint8_t* plane = W + N * (K / 2) + 2 * N * (K / Q4O_GROUP);
    uint64_t off = 2 * (n * (K / Q4O_GROUP) + g);
    uint16_t h = (uint16_t)(plane[off] | ((uint16_t)plane[off + 1] << 8));
    return bf16_to_f64(h);
}

/* Dequantized weight w[n,k] = s*q + b, exact in double. */
double q4o_weight(const uint8_t* W, uint64_t N, uint64_t K, uint64_t n, uint64_t k) {
    uint64_t g = k / Q4O_GROUP;
    return scale_at(W, N, K, n, g) * (double)nib(W, K, n, k) + bias_at(W, N, K, n, g);
}

typedef struct {
    const uint16_t* x;
    const uint8_t* W;
    int M;
    uint64_t N, K;
    const int64_t* cols;     /* NULL: all columns 0..N-1 */
    uint64_t ncols;
    double* y;               /* [M, ncols] */
    double* absy;            /* [M, ncols] or NULL */
    uint64_t c0, c1;         /* this worker's column range */
    double* wrow;            /* scratch, K doubles */
} job_t;

static void run_cols(job_t* j) {
    const uint64_t K = j->K;
    for (uint64_t c = j->c0; c < j->c1; ++c) {
        uint64_t n = j->cols ? (uint64_t)j->cols[c] : c;
        for (uint64_t k = 0; k < K; ++k) j->wrow[k] = q4o_weight(j->W, j->N, K, n, k);
        for (int m = 0; m < j->M; ++m) {
            const uint16_t* xr = j->x + (uint64_t)m * K;
            double acc = 0.0, aacc = 0.0;
            for (uint64_t k = 0; k < K; ++k) {
                double p = bf16_to_f64(xr[k]) * j->wrow[k];
                acc += p;
                aacc += fabs(p);
            }
            j->y[(uint64_t)m * j->ncols + c] = acc;
            if (j->absy) j->absy[(uint64_t)m * j->ncols + c] = aacc;
        }
    }
}

static void* worker(void* arg) {
    run_cols((job_t*)arg);
    return NULL;
}

#define Q4O_MAX_THREADS 256

/* y[M, ncols] (and optional absy = sum_k |x*w|) for the listed columns
 * (cols == NULL: every column, ncols must equal N).  Returns 0 on success,
 * -1 on invalid arguments, -2 on resource failure. */
int q4o_matmul_cols_f64(const uint16_t* x, const uint8_t* W, int M, uint64_t N, uint64_t K,
                        const int64_t* cols, uint64_t ncols, double* y, double* absy,
                        int n_threads) {
    if (!x || !W || !y || M < 1 || q4o_packed_bytes(N, K) == 0) return -1;
    if (!cols && ncols != N) return -1;
    if (cols)
        for (uint64_t c = 0; c < ncols; ++c)
            if (cols[c] < 0 || (uint64_t)cols[c] >= N) return -1;
    if (ncols == 0) return 0;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > Q4O_MAX_THREADS) n_threads = Q4O_MAX_THREADS;
    if ((uint64_t)n_threads > ncols) n_threads = (int)ncols;

    job_t jobs[Q4O_MAX_THREADS];
    pthread_t tids[Q4O_MAX_THREADS];
    double* scratch = (double*)calloc((size_t)n_threads * K, sizeof(double));
    if (!scratch) return -2;
    for (int t = 0; t < n_threads; ++t) {
        jobs[t].x = x; jobs[t].W = W; jobs[t].M = M; jobs[t].N = N; jobs[t].K = K;
        jobs[t].cols = cols; jobs[t].ncols = ncols; jobs[t].y = y; jobs[t].absy = absy;
        jobs[t].c0 = ncols * (uint64_t)t / (uint64_t)n_threads;
        jobs[t].c1 = ncols * (uint64_t)(t + 1) / (uint64_t)n_threads;
        jobs[t].wrow = scratch + (size_t)t * K;
    }
    int started = 0;
    for (int t = 1; t < n_threads; ++t) {
        if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0) break;
        started = t;
    }
    run_cols(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = started + 1; t < n_threads; ++t) run_cols(&jobs[t]);   /* not started: run here */
    free(scratch);
    return 0;
}

/*
 * Inter-layer glue of the chained verify pass (this project's reading: the
 * pages' real between-layer operators -- attention, Gated DeltaNet, norms --
 * are outside the matmul path, so a fixed, bounded stand-in joins layers).
 *
 *   kind 1 (RMSNORM):        v_k = y[m, k]                      k < K <= Nprev
 *   kind 2 (SWIGLU_RMSNORM): v_k = silu(y[m, k]) * y[m, K + k]  Nprev == 2K
 *   x[m, k] = bf16_RNE( v_k / sqrt( (1/K) sum_j v_j^2 + eps ) )
 *
 * silu(a) = a / (1 + exp(-a)).  Computed in double from the fp32 y, rounded
 * once to bf16.  Returns 0, or -1 on invalid arguments.
 */
int q4o_glue_f64(const float* y, int M, uint64_t Nprev, uint64_t K, int kind, double eps,
                 uint16_t* x_out) {
    if (!y || !x_out || M < 1 || K == 0) return -1;
    if (kind == 1 && K > Nprev) return -1;
    if (kind == 2 && Nprev != 2 * K) return -1;
    if (kind != 1 && kind != 2) return -1;
    double* v = (double*)calloc((size_t)K, sizeof(double));
    if (!v) return -1;
    for (int m = 0; m < M; ++m) {
        const float* yr = y + (uint64_t)m * Nprev;
        double ss = 0.0;
        for (uint64_t k = 0; k < K; ++k) {
            double a = (double)yr[k];
            if (kind == 2) a = a / (1.0 + exp(-a)) * (double)yr[K + k];
            v[k] = a;
            ss += a * a;
        }
        double inv = 1.0 / sqrt(ss / (double)K + eps);
        for (uint64_t k = 0; k < K; ++k) x_out[(uint64_t)m * K + k] = f64_to_bf16_rne(v[k] * inv);
    }
    free(v);
    return 0;
}

/* Exposed for the oracle's own pins (rounding helper and exact widening). */
uint16_t q4o_f64_to_bf16(double v) { return f64_to_bf16_rne(v); }
double q4o_bf16_to_f64(uint16_t h) { return bf16_to_f64(h); }
