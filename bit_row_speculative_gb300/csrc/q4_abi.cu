// Host side of the C ABI declared in include/q4.h: argument checks, the launch
// plan (chosen from N, K and the device's SM count only, never from M) and the
// kernel launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>
#include <algorithm>
#include <cstdlib>
#include <utility>

#include "q4.h"
#include "q4_generic.cuh"
#include "q4_tc.cuh"
#include "q4_tm.cuh"
#include "q4_glue.cuh"
#include "q4_topk.cuh"
#include "q4_edges.cuh"

// Set by a kernel whose bounded device-side wait ran out (never by a trap).
__device__ unsigned int q4_device_error_word = 0;

namespace {

constexpr unsigned int kErrWaitCheck = 0x80000000u;   // bit set by the wait self-check below

// One thread waits, with the kernels' own bounded wait, on an mbarrier that
// nothing arrives on; when the limit runs out it records a timeout in the
// error word exactly as a kernel would, and returns.
__global__ void wait_check_kernel(long long limit_cycles, unsigned int* error_word) {
    __shared__ uint64_t bar;
    q4::sm100::mbar_init(&bar, 1);
    q4::sm100::fence_mbar_init();
    if (!q4::sm100::mbar_wait(&bar, 0, limit_cycles)) atomicOr(error_word, kErrWaitCheck);
}

}  // namespace

namespace {

thread_local std::string g_last_error;

q4_status fail(q4_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

q4_status cuda_fail(cudaError_t e, const char* what) {
    return fail(Q4_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    q4_status status = Q4_OK;
    std::string error;
    int sm_count = 0;
    float* partials = nullptr;      // split-K partial sums of the tensor-core kernel
    int* sems = nullptr;            // per-tile arrival counters (zero between launches)
    size_t sem_bytes = 0;
    uint8_t* xt = nullptr;          // prepared x records (one per group of 64 inputs)
    unsigned int* ctl = nullptr;    // call counters of the tensor-memory kernel (zero between launches)
    uint64_t* topk_cand = nullptr;  // sampling epilogue: per-slice candidates [16][128][32]
    int* topk_tickets = nullptr;    // sampling epilogue: per-row arrival counters (zero between launches)
    unsigned int* error_word = nullptr;
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

#ifdef Q4_TRACE
unsigned long long* g_trace = nullptr;
#endif

// The tensor-core path serves K up to 64 * kTcMaxGroups (the prepared-x scratch).
constexpr int64_t kTcMaxGroups = 2048;

DeviceInfo g_devices[kMaxDevices];
std::mutex g_device_mutex;

template <int MT>
cudaError_t prepare_tc() {
    return cudaFuncSetAttribute(q4::tc::q4_tc_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                q4::tc::smem_bytes());
}

template <int MT>
cudaError_t prepare_tm() {
    return cudaFuncSetAttribute(q4::tm::q4_tm_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                q4::tm::smem_bytes<MT>());
}

template <int MT>
cudaError_t prepare_generic() {
    return cudaFuncSetAttribute(q4::generic::matmul_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)q4::generic::smem_bytes(MT));
}

// One-time per-device set-up: capability check and kernel attributes.
q4_status device_setup(int* dev_out, const DeviceInfo** info_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(Q4_ERR_UNSUPPORTED_DEVICE, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_device_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        if (prop.major != 10 || prop.minor != 3) {
            d.status = Q4_ERR_UNSUPPORTED_DEVICE;
            char buf[512];
            snprintf(buf, sizeof buf, "device %d (%s) is compute %d.%d; this library is built for 10.3 (sm_103a)",
                     dev, prop.name, prop.major, prop.minor);
            d.error = buf;
        } else {
            d.sm_count = prop.multiProcessorCount;
            cudaError_t a = prepare_generic<1>();
            if (a == cudaSuccess) a = prepare_generic<2>();
            if (a == cudaSuccess) a = prepare_generic<4>();
            if (a == cudaSuccess) a = prepare_generic<8>();
            if (a == cudaSuccess) a = prepare_generic<16>();
            if (a == cudaSuccess) a = prepare_generic<32>();
            if (a == cudaSuccess) a = prepare_tc<1>();
            if (a == cudaSuccess) a = prepare_tc<2>();
            if (a == cudaSuccess) a = prepare_tc<4>();
            if (a == cudaSuccess) a = prepare_tc<8>();
            if (a == cudaSuccess) a = prepare_tc<16>();
            if (a == cudaSuccess) a = prepare_tm<1>();
            if (a == cudaSuccess) a = prepare_tm<2>();
            if (a == cudaSuccess) a = prepare_tm<4>();
            if (a == cudaSuccess) a = prepare_tm<8>();
            if (a == cudaSuccess) a = prepare_tm<16>();
            if (a == cudaSuccess) a = prepare_tm<24>();
            if (a == cudaSuccess) a = prepare_tm<32>();
            if (a != cudaSuccess) return cuda_fail(a, "cudaFuncSetAttribute");
            if (!g_encode) {
                void* fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                a = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
                if (a != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                    return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
            }
            // scratch of the tensor-core kernel, sized for one CTA per SM
            const size_t pbytes = std::max(q4::tc::partial_floats(d.sm_count), q4::tm::partial_floats(d.sm_count)) *
                                  sizeof(float);
            const size_t sbytes = std::max(q4::tc::sem_ints(d.sm_count), q4::tm::sem_ints(d.sm_count)) *
                                  sizeof(int);
            d.sem_bytes = sbytes;
            a = cudaMalloc(&d.partials, pbytes);
            if (a == cudaSuccess) a = cudaMalloc(&d.sems, sbytes);
            if (a == cudaSuccess)
                a = cudaMalloc(&d.xt, (size_t)kTcMaxGroups * std::max(q4::prep::kRecordBytes, q4::tm::rec_bytes(32)));
            if (a == cudaSuccess)
                a = cudaMalloc(&d.topk_cand, (size_t)Q4_MAX_ROWS * q4::topk::kMaxSlices * q4::topk::kWidth * sizeof(uint64_t));
            if (a == cudaSuccess) a = cudaMalloc(&d.ctl, q4::tm::kCtlWords * sizeof(unsigned int));
            if (a == cudaSuccess) a = cudaMemset(d.ctl, 0, q4::tm::kCtlWords * sizeof(unsigned int));
            if (a == cudaSuccess) a = cudaMalloc(&d.topk_tickets, (size_t)Q4_MAX_ROWS * sizeof(int));
            if (a == cudaSuccess) a = cudaMemset(d.topk_tickets, 0, (size_t)Q4_MAX_ROWS * sizeof(int));
            if (a == cudaSuccess) a = cudaMemset(d.sems, 0, sbytes);
            if (a == cudaSuccess) a = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.error_word), q4_device_error_word);
            if (a == cudaSuccess) a = cudaDeviceSynchronize();
            if (a != cudaSuccess) return cuda_fail(a, "allocating the library scratch");
            d.status = Q4_OK;
        }
        d.ready = true;
    }
    if (d.status != Q4_OK) return fail(d.status, "%s", d.error.c_str());
    *dev_out = dev;
    *info_out = &d;
    return Q4_OK;
}

// Zero the arrival counters of the current device's scratch, if that device
// has been set up (nothing to do otherwise).  Synchronous; allocates nothing.
cudaError_t reset_counters(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
    std::lock_guard<std::mutex> lock(g_device_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready || d.status != Q4_OK) return cudaSuccess;
    cudaError_t e = cudaMemset(d.sems, 0, d.sem_bytes);
    if (e == cudaSuccess) e = cudaMemset(d.ctl, 0, q4::tm::kCtlWords * sizeof(unsigned int));
    if (e == cudaSuccess) e = cudaMemset(d.topk_tickets, 0, (size_t)Q4_MAX_ROWS * sizeof(int));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return e;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int rows_template(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : 32; }
// the tensor-memory kernel also has a 24-row instance (same 32-row layout, fewer live accumulators)
int tm_rows_template(int M) { return M <= 16 ? rows_template(M) : M <= 24 ? 24 : 32; }

q4_status launch_generic(const void* x, const void* W, int M, int64_t N, int64_t K, float* y,
                         cudaStream_t stream) {
    using namespace q4::generic;
    const int64_t blocks = (N + kRowsPerCta - 1) / kRowsPerCta;
    if (blocks > 0x7FFFFFFF) return fail(Q4_ERR_INVALID_ARG, "N = %lld needs too many blocks", (long long)N);
    const int MT = rows_template(M);
    const dim3 grid((unsigned)blocks), block(kWarps * 32);
    const size_t smem = smem_bytes(MT);
    auto xp = static_cast<const uint16_t*>(x);
    auto wp = static_cast<const uint8_t*>(W);
    switch (MT) {
        case 1: matmul_kernel<1><<<grid, block, smem, stream>>>(xp, wp, M, N, K, y); break;
        case 2: matmul_kernel<2><<<grid, block, smem, stream>>>(xp, wp, M, N, K, y); break;
        case 4: matmul_kernel<4><<<grid, block, smem, stream>>>(xp, wp, M, N, K, y); break;
        case 8: matmul_kernel<8><<<grid, block, smem, stream>>>(xp, wp, M, N, K, y); break;
        case 16: matmul_kernel<16><<<grid, block, smem, stream>>>(xp, wp, M, N, K, y); break;
        default: matmul_kernel<32><<<grid, block, smem, stream>>>(xp, wp, M, N, K, y); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launching the generic Q4 kernel");
    return Q4_OK;
}

q4_status encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return Q4_OK;
}

// Launch `kernel` on `stream` with programmatic stream serialization, so that
// it may start while the preceding kernel finishes (it waits on the device
// with griddepcontrol.wait before touching that kernel's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

q4_status launch_tc(const DeviceInfo& d, const void* x, const void* W, int M, int64_t N, int64_t K, float* y,
                    cudaStream_t stream) {
    using namespace q4::tc;
    CUtensorMap map_nib;
    q4_status s = encode_2d(&map_nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, (uint64_t)K / 2, (uint64_t)N,
                            (uint64_t)K / 2, 64, kRowsCG, CU_TENSOR_MAP_SWIZZLE_64B);
    if (s != Q4_OK) return s;
    Params p;
    p.W = static_cast<const uint8_t*>(W);
    p.xt = d.xt;
    p.y = y;
    p.partials = d.partials;
    p.sems = d.sems;
    p.error_word = d.error_word;
    p.N = N;
    p.K = K;
    p.M = M;
    p.G = (int)(K / 64);
    p.T = (int)((N + kRowsTile - 1) / kRowsTile);
    p.U = p.T * p.G;
    p.C = p.U < d.sm_count ? p.U : d.sm_count;
#ifdef Q4_TRACE
    p.trace = g_trace;
#endif
    cudaError_t e = launch_pdl(q4::prep::prep_x_kernel, dim3((unsigned)p.G), dim3(q4::prep::kThreads), 0, stream,
                               static_cast<const uint16_t*>(x), M, K, d.xt);
    if (e != cudaSuccess) return cuda_fail(e, "launching the x preparation kernel");
    const dim3 grid((unsigned)p.C), block(kThreads);
    const size_t smem = (size_t)smem_bytes();
    switch (rows_template(M)) {
        case 1: e = launch_pdl(q4_tc_kernel<1>, grid, block, smem, stream, map_nib, p); break;
        case 2: e = launch_pdl(q4_tc_kernel<2>, grid, block, smem, stream, map_nib, p); break;
        case 4: e = launch_pdl(q4_tc_kernel<4>, grid, block, smem, stream, map_nib, p); break;
        case 8: e = launch_pdl(q4_tc_kernel<8>, grid, block, smem, stream, map_nib, p); break;
        default: e = launch_pdl(q4_tc_kernel<16>, grid, block, smem, stream, map_nib, p); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "launching the tensor-core Q4 kernel");
    return Q4_OK;
}

// Work split of the tensor-memory kernel, from T, GP and the SM count only.
// Stream-K over all tiles by default: R = 3C ranges of about U / R units, which
// cross tile boundaries, so most ranges end two partial tiles.  Where the tiles
// divide among the teams (S = floor(3C / T) >= 2 ranges per tile, no longer than
// the stream-K ranges), every range lies inside one tile instead and ends just
// one partial tile: the attention and out-projection shapes.
void plan_ranges(q4::tm::Params& p, int sm_count) {
    using namespace q4::tm;
    const int C0 = grid_ctas(p.U, sm_count);
    const int R0 = kTeams * C0;
    const int q_stream = (p.U + R0 - 1) / R0;         // longest stream-K range
    int s = R0 / p.T;
    if (s > p.GP) s = p.GP;
    if (s >= 2 && (p.GP + s - 1) / s <= q_stream) {
        p.S = s;
        p.L = p.GP;
        p.R = p.T * s;
        p.C = (p.R + kTeams - 1) / kTeams;
    } else {
        p.S = R0;
        p.L = p.U;
        p.R = R0;
        p.C = C0;
    }
    p.q_units = p.L / p.S;
    p.rem_units = p.L % p.S;
}

q4_status launch_tm(const DeviceInfo& d, const void* x, const void* W, int M, int64_t N, int64_t K, float* y,
                    cudaStream_t stream, bool records_ready) {
    using namespace q4::tm;
    const int MT = tm_rows_template(M);
    CUtensorMap map_nib, map_sb;
    const uint8_t* w8 = static_cast<const uint8_t*>(W);
    const uint64_t G = (uint64_t)K / 64;
    q4_status s = encode_2d(&map_nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, (uint64_t)K / 2, (uint64_t)N,
                            (uint64_t)K / 2, 64, kRowsTile, CU_TENSOR_MAP_SWIZZLE_64B);
    // scale and bias planes as one 3-D tensor [2][N][G] of bf16 words; boxes of 8 groups x 128 rows x both planes
    if (s == Q4_OK) {
        const cuuint64_t dims[3] = {G, (cuuint64_t)N, 2};
        const cuuint64_t strides[2] = {G * 2, (cuuint64_t)N * G * 2};
        const cuuint32_t box[3] = {8, (cuuint32_t)kRowsTile, 2};
        const cuuint32_t estr[3] = {1, 1, 1};
        const CUresult r = g_encode(&map_sb, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                                    const_cast<uint8_t*>(w8 + (uint64_t)N * (uint64_t)K / 2), dims, strides, box, estr,
                                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) s = fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    if (s != Q4_OK) return s;
    Params p;
    p.W = w8;
    p.y = y;
    p.x = static_cast<const uint16_t*>(x);
    p.partials = d.partials;
    p.sems = d.sems;
    p.xt = d.xt;
    p.ctl = d.ctl;
    p.error_word = d.error_word;
    p.N = N;
    p.K = K;
    p.M = M;
    p.G = (int)(K / 64);
    p.GP = p.G / 2;
    p.T = (int)((N + kRowsTile - 1) / kRowsTile);
    p.U = p.T * p.GP;
    plan_ranges(p, d.sm_count);
    p.build = records_ready ? 0 : 1;   // else the preceding glue kernel wrote the records
#ifdef Q4_TRACE
    p.trace = g_trace;
#endif
    cudaError_t e = cudaSuccess;
    const dim3 grid((unsigned)p.C), block(kThreads);
    switch (MT) {
        case 1: e = launch_pdl(q4_tm_kernel<1>, grid, block, (size_t)smem_bytes<1>(), stream, map_nib, map_sb, p); break;
        case 2: e = launch_pdl(q4_tm_kernel<2>, grid, block, (size_t)smem_bytes<2>(), stream, map_nib, map_sb, p); break;
        case 4: e = launch_pdl(q4_tm_kernel<4>, grid, block, (size_t)smem_bytes<4>(), stream, map_nib, map_sb, p); break;
        case 8: e = launch_pdl(q4_tm_kernel<8>, grid, block, (size_t)smem_bytes<8>(), stream, map_nib, map_sb, p); break;
        case 16: e = launch_pdl(q4_tm_kernel<16>, grid, block, (size_t)smem_bytes<16>(), stream, map_nib, map_sb, p); break;
        case 24: e = launch_pdl(q4_tm_kernel<24>, grid, block, (size_t)smem_bytes<24>(), stream, map_nib, map_sb, p); break;
        default: e = launch_pdl(q4_tm_kernel<32>, grid, block, (size_t)smem_bytes<32>(), stream, map_nib, map_sb, p); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "launching the tensor-memory Q4 kernel");
    return Q4_OK;
}

// The launch plan depends on N, K and the device only -- never on M -- so a
// row's result is the same for every M.
bool use_tc(int64_t N, int64_t K) {
    // the kernel's schedule arithmetic is 32-bit: tiles x groups must fit
    return (K % 512) == 0 && K / 64 <= kTcMaxGroups &&
           ((N + q4::tc::kRowsTile - 1) / q4::tc::kRowsTile) * (K / 64) < ((int64_t)1 << 30);
}

// The kernel for a (validated) matmul: the tensor-memory kernel for K a
// multiple of 512, the generic kernel otherwise.
// records_ready: the x records of this call are already in the scratch (written by
// a glue kernel in record mode); only valid when use_tc(N, K).
q4_status dispatch_matmul(const DeviceInfo& d, const void* x, const void* W, int M, int64_t N, int64_t K, float* y,
                          cudaStream_t stream, bool records_ready = false) {
    if (use_tc(N, K)) return launch_tm(d, x, W, M, N, K, y, stream, records_ready);
    return launch_generic(x, W, M, N, K, y, stream);
}

// Argument checks shared by the matmul entry points (everything but the device).
q4_status check_matmul_args(const void* x, const void* W, int M, int64_t N, int64_t K, const void* y) {
    if (!x || !W || !y) return fail(Q4_ERR_INVALID_ARG, "null pointer argument (x=%p W=%p y=%p)", x, W, y);
    if (M < 1 || M > Q4_MAX_ROWS) return fail(Q4_ERR_INVALID_ARG, "M = %d is outside 1..%d", M, Q4_MAX_ROWS);
    if (N < 1) return fail(Q4_ERR_INVALID_ARG, "N = %lld must be >= 1", (long long)N);
    if (K < 64 || (K % 64) != 0)
        return fail(Q4_ERR_UNSUPPORTED_SHAPE, "K = %lld must be a positive multiple of 64", (long long)K);
    if (q4_packed_bytes((uint64_t)N, (uint64_t)K) == 0)
        return fail(Q4_ERR_OVERFLOW, "packed size of %lld x %lld overflows", (long long)N, (long long)K);
    if ((uint64_t)M * (uint64_t)N > (1ull << 40))
        return fail(Q4_ERR_INVALID_ARG, "output of %d x %lld is too large", M, (long long)N);
    if (!aligned16(x) || !aligned16(W) || !aligned16(y))
        return fail(Q4_ERR_MISALIGNED, "x, W and y must be 16-byte aligned (x=%p W=%p y=%p)", x, W, y);
    return Q4_OK;
}

constexpr double kGlueEps = 1e-6;

q4_status check_glue_args(const float* y, int M, int64_t n_prev, int64_t K, int kind, const void* x) {
    if (!y || !x) return fail(Q4_ERR_INVALID_ARG, "null pointer argument (y=%p x=%p)", (const void*)y, x);
    if (M < 1 || M > Q4_MAX_ROWS) return fail(Q4_ERR_INVALID_ARG, "M = %d is outside 1..%d", M, Q4_MAX_ROWS);
    if (K < 1 || n_prev < 1) return fail(Q4_ERR_INVALID_ARG, "glue widths must be >= 1 (N_prev=%lld K=%lld)",
                                         (long long)n_prev, (long long)K);
    if (kind == Q4_GLUE_RMSNORM) {
        if (K > n_prev)
            return fail(Q4_ERR_INVALID_ARG, "RMSNORM glue takes the first K=%lld of N_prev=%lld columns", (long long)K,
                        (long long)n_prev);
    } else if (kind == Q4_GLUE_SWIGLU_RMSNORM) {
        if (n_prev != 2 * K)
            return fail(Q4_ERR_INVALID_ARG, "SWIGLU_RMSNORM glue needs N_prev == 2K (N_prev=%lld K=%lld)",
                        (long long)n_prev, (long long)K);
    } else {
        return fail(Q4_ERR_INVALID_ARG, "unknown glue kind %d", kind);
    }
    // the kernel's slices are whole groups of 64 inputs (K_next is the K of a matmul)
    if (K % 64 != 0) return fail(Q4_ERR_UNSUPPORTED_SHAPE, "K_next = %lld must be a multiple of 64", (long long)K);
    if (!aligned16(y) || !aligned16(x))
        return fail(Q4_ERR_MISALIGNED, "y and x must be 16-byte aligned (y=%p x=%p)", (const void*)y, x);
    return Q4_OK;
}

// glue::slices(K) CTAs per row (a cluster, unless every CTA sums its row alone), chained by
// programmatic dependent launch.
// x mode (rec == nullptr): x_next bf16 [M, K] to x.  Record mode: the next
// matmul's x records (row width rec_w) to rec instead.
q4_status launch_glue(const float* y, int M, int64_t n_prev, int64_t K, int kind, void* x, cudaStream_t stream,
                      uint8_t* rec = nullptr, int rec_w = 16) {
    // rows every CTA sums alone: 8 CTAs (one per 640 inputs at K = 5120) spread the outputs widest
    // (measured: 1, 2, 5 and 16 per row were slower); otherwise slices(K), as a cluster
    const int S = q4::glue::one_cta_rows(kind, K) ? (int)std::min<int64_t>(q4::glue::kMaxSlices, K / 64)
                                                  : q4::glue::slices(K);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S, (unsigned)M);
    cfg.blockDim = dim3(q4::glue::kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = q4::glue::one_cta_rows(kind, K) ? 1 : 2;   // rows a CTA sums alone need no cluster
    const float eps_hi = (float)kGlueEps;
    const float eps_lo = (float)(kGlueEps - (double)eps_hi);
    cudaError_t e = cudaLaunchKernelEx(&cfg, q4::glue::glue_kernel, y, n_prev, K, kind, eps_hi, eps_lo,
                                       static_cast<uint16_t*>(x), rec, rec_w);
    if (e != cudaSuccess) return cuda_fail(e, "launching the glue kernel");
    return Q4_OK;
}

size_t round_up256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace of a decode step: one fp32 buffer for the widest intermediate y and
// one bf16 buffer for the widest intermediate x.
void decode_workspace_layout(const q4_layer* layers, int n_layers, int M, size_t* y_bytes, size_t* x_bytes) {
    int64_t max_n = 0, max_k = 0;
    for (int j = 0; j + 1 < n_layers; ++j) {
        max_n = std::max(max_n, layers[j].N);
        max_k = std::max(max_k, layers[j + 1].K);
    }
    *y_bytes = round_up256((size_t)M * (size_t)max_n * sizeof(float));
    *x_bytes = round_up256((size_t)M * (size_t)max_k * sizeof(uint16_t));
}

}  // namespace

// ---------------------------------------------------------------------------
// Scratch of q4_matmul_noalloc, for callers that may not allocate device
// memory at run time.  It lives in the library's own image: every device that
// loads the library holds kNoAllocScratchBytes of it until the process exits.
// Layout: [split-K partial sums][per-tile counters][prepared x records], each
// part 256-byte aligned, sized for the tensor-memory kernel with one CTA per
// SM on up to kNoAllocMaxSms SMs and K up to kNoAllocMaxK.
namespace {

constexpr int kNoAllocMaxSms = 160;
constexpr int kNoAllocMaxRows = 16;   // its two-launch kernel holds 16-row x records
constexpr int64_t kNoAllocMaxK = 20480;
constexpr size_t round256(size_t b) { return (b + 255) / 256 * 256; }
constexpr size_t kNoAllocPartialBytes =
    round256((size_t)kNoAllocMaxSms * 2 * q4::tc::kCG * 16 * q4::tc::kRowsCG * sizeof(float));
constexpr size_t kNoAllocSemBytes = round256((size_t)kNoAllocMaxSms * q4::tc::kCG * sizeof(int));
constexpr size_t kNoAllocXtBytes = round256((size_t)(kNoAllocMaxK / 64) * q4::prep::kRecordBytes);
constexpr size_t kNoAllocScratchBytes = kNoAllocPartialBytes + kNoAllocSemBytes + kNoAllocXtBytes;
static_assert(kNoAllocScratchBytes == 8542208, "the size q4.h states for q4_matmul_noalloc's scratch");

}  // namespace

static __device__ __align__(256) unsigned char q4_noalloc_scratch[kNoAllocScratchBytes];

namespace {

struct NoAllocDevice {
    bool ready = false;
    q4_status status = Q4_OK;
    std::string error;
    int sm_count = 0;
    uint8_t* scratch = nullptr;          // device address of q4_noalloc_scratch on this device
    unsigned int* error_word = nullptr;  // device address of q4_device_error_word
};

NoAllocDevice g_noalloc_devices[kMaxDevices];

// One-time set-up of the current device for q4_matmul_noalloc: capability
// check, kernel attributes and the device addresses of the static arrays.  In
// host code the array's name only stands for it; the address a kernel needs
// comes from cudaGetSymbolAddress with the device current.  Allocates nothing.
q4_status noalloc_setup(const NoAllocDevice** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(Q4_ERR_UNSUPPORTED_DEVICE, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_device_mutex);
    NoAllocDevice& d = g_noalloc_devices[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        char buf[512];
        if (prop.major != 10 || prop.minor != 3) {
            d.status = Q4_ERR_UNSUPPORTED_DEVICE;
            snprintf(buf, sizeof buf, "device %d (%s) is compute %d.%d; this library is built for 10.3 (sm_103a)",
                     dev, prop.name, prop.major, prop.minor);
            d.error = buf;
        } else if (prop.multiProcessorCount > kNoAllocMaxSms) {
            d.status = Q4_ERR_UNSUPPORTED_DEVICE;
            snprintf(buf, sizeof buf,
                     "device %d has %d SMs; the static scratch of q4_matmul_noalloc is sized for at most %d",
                     dev, prop.multiProcessorCount, kNoAllocMaxSms);
            d.error = buf;
        } else {
            d.sm_count = prop.multiProcessorCount;
            cudaError_t a = prepare_generic<1>();
            if (a == cudaSuccess) a = prepare_generic<2>();
            if (a == cudaSuccess) a = prepare_generic<4>();
            if (a == cudaSuccess) a = prepare_generic<8>();
            if (a == cudaSuccess) a = prepare_generic<16>();
            if (a == cudaSuccess) a = prepare_generic<32>();
            if (a == cudaSuccess) a = prepare_tc<1>();
            if (a == cudaSuccess) a = prepare_tc<2>();
            if (a == cudaSuccess) a = prepare_tc<4>();
            if (a == cudaSuccess) a = prepare_tc<8>();
            if (a == cudaSuccess) a = prepare_tc<16>();
            if (a != cudaSuccess) return cuda_fail(a, "cudaFuncSetAttribute");
            if (!g_encode) {
                void* fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                a = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
                if (a != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                    return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
            }
            void* ptr = nullptr;
            a = cudaGetSymbolAddress(&ptr, q4_noalloc_scratch);
            if (a != cudaSuccess) return cuda_fail(a, "cudaGetSymbolAddress(q4_noalloc_scratch)");
            d.scratch = static_cast<uint8_t*>(ptr);
            a = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.error_word), q4_device_error_word);
            if (a != cudaSuccess) return cuda_fail(a, "cudaGetSymbolAddress(q4_device_error_word)");
            d.status = Q4_OK;
        }
        d.ready = true;
    }
    if (d.status != Q4_OK) return fail(d.status, "%s", d.error.c_str());
    *out = &d;
    return Q4_OK;
}

}  // namespace

extern "C" {

uint64_t q4_packed_bytes(uint64_t N, uint64_t K) {
    if (N == 0 || K == 0 || (K % 64) != 0) return 0;
    if (K > UINT64_MAX / N) return 0;
    const uint64_t per16 = (N * K) / 16;
    if (per16 > UINT64_MAX / 9) return 0;
    return per16 * 9;
}

q4_status q4_matmul(const void* x, const void* W, int M, int64_t N, int64_t K, float* y,
                    q4_stream_t stream) {
    g_last_error.clear();
    q4_status cs = check_matmul_args(x, W, M, N, K, y);
    if (cs != Q4_OK) return cs;
    int dev = 0;
    const DeviceInfo* info = nullptr;
    q4_status s = device_setup(&dev, &info);
    if (s != Q4_OK) return s;
    return dispatch_matmul(*info, x, W, M, N, K, y, reinterpret_cast<cudaStream_t>(stream));
}

q4_status q4_matmul_noalloc(const void* x, const void* W, int M, int64_t N, int64_t K, float* y,
                            q4_stream_t stream) {
    g_last_error.clear();
    if (!x || !W || !y) return fail(Q4_ERR_INVALID_ARG, "null pointer argument (x=%p W=%p y=%p)", x, W, (void*)y);
    if (M < 1 || M > kNoAllocMaxRows)
        return fail(Q4_ERR_INVALID_ARG, "M = %d is outside 1..%d (q4_matmul_noalloc)", M, kNoAllocMaxRows);
    if (N < 1) return fail(Q4_ERR_INVALID_ARG, "N = %lld must be >= 1", (long long)N);
    if (K < 64 || (K % 64) != 0)
        return fail(Q4_ERR_UNSUPPORTED_SHAPE, "K = %lld must be a positive multiple of 64", (long long)K);
    if (K > kNoAllocMaxK)
        return fail(Q4_ERR_UNSUPPORTED_SHAPE,
                    "K = %lld is larger than the %lld inputs the static scratch of q4_matmul_noalloc holds; "
                    "use q4_matmul", (long long)K, (long long)kNoAllocMaxK);
    if (q4_packed_bytes((uint64_t)N, (uint64_t)K) == 0)
        return fail(Q4_ERR_OVERFLOW, "packed size of %lld x %lld overflows", (long long)N, (long long)K);
    if ((uint64_t)M * (uint64_t)N > (1ull << 40))
        return fail(Q4_ERR_INVALID_ARG, "output of %d x %lld is too large", M, (long long)N);
    if (!aligned16(x) || !aligned16(W) || !aligned16(y))
        return fail(Q4_ERR_MISALIGNED, "x, W and y must be 16-byte aligned (x=%p W=%p y=%p)", x, W, (void*)y);
    const NoAllocDevice* nd = nullptr;
    q4_status s = noalloc_setup(&nd);
    if (s != Q4_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!use_tc(N, K)) return launch_generic(x, W, M, N, K, y, st);   // this kernel needs no scratch
    DeviceInfo view;
    view.ready = true;
    view.sm_count = nd->sm_count;
    view.partials = reinterpret_cast<float*>(nd->scratch);
    view.sems = reinterpret_cast<int*>(nd->scratch + kNoAllocPartialBytes);
    view.xt = nd->scratch + kNoAllocPartialBytes + kNoAllocSemBytes;
    view.error_word = nd->error_word;
    // the counters must start at zero; a call that gave up a wait may have left them set
    cudaError_t e = cudaMemsetAsync(view.sems, 0, kNoAllocSemBytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the static scratch counters");
    return launch_tc(view, x, W, M, N, K, y, st);
}

q4_status q4_glue(const float* y, int M, int64_t n_prev, int64_t k_next, int kind, void* x_next,
                  q4_stream_t stream) {
    g_last_error.clear();
    q4_status s = check_glue_args(y, M, n_prev, k_next, kind, x_next);
    if (s != Q4_OK) return s;
    int dev = 0;
    const DeviceInfo* info = nullptr;
    s = device_setup(&dev, &info);
    if (s != Q4_OK) return s;
    return launch_glue(y, M, n_prev, k_next, kind, x_next, reinterpret_cast<cudaStream_t>(stream));
}

size_t q4_decode_step_workspace_bytes(const q4_layer* layers, int n_layers, int M) {
    if (!layers || n_layers < 1 || M < 1 || M > Q4_MAX_ROWS) return 0;
    size_t yb = 0, xb = 0;
    decode_workspace_layout(layers, n_layers, M, &yb, &xb);
    return yb + xb;
}

q4_status q4_decode_step(const q4_layer* layers, int n_layers, const void* x0, int M, void* workspace,
                         size_t workspace_bytes, float* y_last, q4_stream_t stream) {
    g_last_error.clear();
    if (!layers || n_layers < 1) return fail(Q4_ERR_INVALID_ARG, "empty layer list (layers=%p n=%d)", (const void*)layers,
                                            n_layers);
    // the whole list is checked before anything is launched
    for (int j = 0; j < n_layers; ++j) {
        const q4_layer& L = layers[j];
        // shapes and W of every layer; x0 and y_last stand in for the inner buffers (the workspace is checked below)
        q4_status s = check_matmul_args(x0, L.W, M, L.N, L.K, y_last);
        if (s != Q4_OK) {
            std::string msg = g_last_error;
            return fail(s, "layer %d: %s", j, msg.c_str());
        }
        if (j + 1 < n_layers) {
            const q4_layer& Nx = layers[j + 1];
            if (L.glue == Q4_GLUE_RMSNORM) {
                if (Nx.K > L.N)
                    return fail(Q4_ERR_INVALID_ARG, "layer %d: RMSNORM glue takes the first K=%lld of its N=%lld outputs",
                                j, (long long)Nx.K, (long long)L.N);
            } else if (L.glue == Q4_GLUE_SWIGLU_RMSNORM) {
                if (L.N != 2 * Nx.K)
                    return fail(Q4_ERR_INVALID_ARG, "layer %d: SWIGLU_RMSNORM glue needs N == 2 * next K (N=%lld K=%lld)",
                                j, (long long)L.N, (long long)Nx.K);
            } else {
                return fail(Q4_ERR_INVALID_ARG, "layer %d: glue kind %d does not chain to layer %d", j, L.glue, j + 1);
            }
        }
    }
    size_t yb = 0, xb = 0;
    decode_workspace_layout(layers, n_layers, M, &yb, &xb);
    if (n_layers > 1) {
        if (!workspace)
            return fail(Q4_ERR_INVALID_ARG, "a %d-layer step needs a workspace of %zu bytes", n_layers, yb + xb);
        if (!aligned16(workspace)) return fail(Q4_ERR_MISALIGNED, "workspace %p is not 16-byte aligned", workspace);
        if (workspace_bytes < yb + xb)
            return fail(Q4_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu bytes the step needs",
                        workspace_bytes, yb + xb);
    }
    int dev = 0;
    const DeviceInfo* info = nullptr;
    q4_status s = device_setup(&dev, &info);
    if (s != Q4_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* ybuf = static_cast<float*>(workspace);
    void* xbuf = static_cast<uint8_t*>(workspace) + yb;
    const void* xj = x0;
    bool records_ready = false;
    const int rec_w = tm_rows_template(M) > 16 ? 32 : 16;
    for (int j = 0; j < n_layers; ++j) {
        const q4_layer& L = layers[j];
        const bool last = j + 1 == n_layers;
        float* yj = last ? y_last : ybuf;
        s = dispatch_matmul(*info, xj, L.W, M, L.N, L.K, yj, st, records_ready);
        if (s != Q4_OK) return s;
        if (!last) {
            const q4_layer& Nx = layers[j + 1];
            // the next matmul on the tensor-memory kernel: the glue writes its x records directly
            records_ready = use_tc(Nx.N, Nx.K);
            s = launch_glue(yj, M, L.N, Nx.K, L.glue, xbuf, st, records_ready ? info->xt : nullptr, rec_w);
            if (s != Q4_OK) return s;
            xj = xbuf;
        }
    }
    return Q4_OK;
}

namespace {

// Argument checks of the sampling epilogue (everything but the device and the logits pointer).
q4_status check_topk_args(int M, int64_t N, int top_k, float temperature, float top_p, const int32_t* idx,
                          const float* probs) {
    using namespace q4::topk;
    if (!idx || !probs)
        return fail(Q4_ERR_INVALID_ARG, "null pointer argument (idx=%p probs=%p)", (const void*)idx, (const void*)probs);
    if (M < 1 || M > Q4_MAX_ROWS) return fail(Q4_ERR_INVALID_ARG, "M = %d is outside 1..%d", M, Q4_MAX_ROWS);
    if (top_k < 1 || top_k > kWidth) return fail(Q4_ERR_INVALID_ARG, "top_k = %d is outside 1..%d", top_k, kWidth);
    if (N < top_k) return fail(Q4_ERR_INVALID_ARG, "N = %lld is smaller than top_k = %d", (long long)N, top_k);
    if (N > (int64_t)kSlice * kMaxSlices)
        return fail(Q4_ERR_UNSUPPORTED_SHAPE, "N = %lld exceeds %lld", (long long)N, (long long)kSlice * kMaxSlices);
    if (!(temperature > 0.0f) || !(temperature < 3.0e38f))
        return fail(Q4_ERR_INVALID_ARG, "temperature must be positive and finite");
    if (!(top_p > 0.0f)) return fail(Q4_ERR_INVALID_ARG, "top_p must be positive");
    if (!aligned16(idx) || !aligned16(probs)) return fail(Q4_ERR_MISALIGNED, "idx and probs must be 16-byte aligned");
    return Q4_OK;
}

q4_status launch_topk(const DeviceInfo& d, const float* logits, int M, int64_t N, int top_k, float temperature,
                      float top_p, int32_t* idx, float* probs, cudaStream_t st, int discard) {
    using namespace q4::topk;
    const int S = (int)((N + kSlice - 1) / kSlice);
    // <= kSlice; a multiple of 32 floats, so slices start on 128-byte lines when each row does
    const int64_t L = ((N + S - 1) / S + 31) / 32 * 32;
    const cudaError_t e = launch_pdl(topk_kernel, dim3((unsigned)S, (unsigned)M), dim3(kThreads), 0, st, logits, N, L,
                                     top_k, temperature, top_p, d.topk_cand, d.topk_tickets, idx, probs, discard);
    if (e != cudaSuccess) return cuda_fail(e, "launching the top-k kernel");
    return Q4_OK;
}

// Logits scratch of q4_lm_head_topk, per device, grown on demand.
struct LogitsScratch {
    float* ptr = nullptr;
    size_t bytes = 0;
};
LogitsScratch g_logits[kMaxDevices];
std::mutex g_logits_mutex;

}  // namespace

q4_status q4_topk_probs(const float* logits, int M, int64_t N, int top_k, float temperature, float top_p,
                        int32_t* idx, float* probs, q4_stream_t stream) {
    g_last_error.clear();
    if (!logits) return fail(Q4_ERR_INVALID_ARG, "null pointer argument (logits)");
    q4_status s = check_topk_args(M, N, top_k, temperature, top_p, idx, probs);
    if (s != Q4_OK) return s;
    if (!aligned16(logits)) return fail(Q4_ERR_MISALIGNED, "logits, idx and probs must be 16-byte aligned");
    int dev = 0;
    const DeviceInfo* info = nullptr;
    s = device_setup(&dev, &info);
    if (s != Q4_OK) return s;
    return launch_topk(*info, logits, M, N, top_k, temperature, top_p, idx, probs,
                       reinterpret_cast<cudaStream_t>(stream), 0);
}

q4_status q4_lm_head_topk(const void* x, const void* W, int M, int64_t N, int64_t K, int top_k, float temperature,
                          float top_p, int32_t* idx, float* probs, q4_stream_t stream) {
    g_last_error.clear();
    q4_status s = check_matmul_args(x, W, M, N, K, probs);
    if (s != Q4_OK) return s;
    s = check_topk_args(M, N, top_k, temperature, top_p, idx, probs);
    if (s != Q4_OK) return s;
    int dev = 0;
    const DeviceInfo* info = nullptr;
    s = device_setup(&dev, &info);
    if (s != Q4_OK) return s;
    float* logits = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_logits_mutex);
        LogitsScratch& ls = g_logits[dev];
        const size_t need = (size_t)M * (size_t)N * sizeof(float);
        if (ls.bytes < need) {
            if (ls.ptr) {
                cudaError_t e = cudaDeviceSynchronize();   // earlier calls may still use the old buffer
                if (e == cudaSuccess) e = cudaFree(ls.ptr);
                if (e != cudaSuccess) return cuda_fail(e, "freeing the logits scratch");
                ls.ptr = nullptr;
                ls.bytes = 0;
            }
            const size_t grow = (size_t)Q4_MAX_ROWS * (size_t)N * sizeof(float);
            const cudaError_t e = cudaMalloc(&ls.ptr, grow);
            if (e != cudaSuccess) return cuda_fail(e, "allocating the logits scratch");
            ls.bytes = grow;
        }
        logits = ls.ptr;
    }
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    s = dispatch_matmul(*info, x, W, M, N, K, logits, st);
    if (s != Q4_OK) return s;
    return launch_topk(*info, logits, M, N, top_k, temperature, top_p, idx, probs, st, 1);
}

q4_status q4_draft_select_edges(const void* pred_cb, const void* succ_cb, int64_t V, int R, const float* hidden,
                                const int32_t* pred_ids, const int32_t* cand_ids, int rows, float* score,
                                q4_stream_t stream) {
    g_last_error.clear();
    using namespace q4::edges;
    if (!pred_cb || !succ_cb || !hidden || !pred_ids || !cand_ids || !score)
        return fail(Q4_ERR_INVALID_ARG, "null pointer argument");
    if (V < 1 || V > (int64_t)INT32_MAX) return fail(Q4_ERR_INVALID_ARG, "V = %lld is outside 1..2^31-1", (long long)V);
    if (R < 8 || R > kMaxRank || R % 8 != 0)
        return fail(Q4_ERR_UNSUPPORTED_SHAPE, "R = %d is not a multiple of 8 in 8..%d", R, kMaxRank);
    if (rows < 1 || rows > kMaxEdgeRows)
        return fail(Q4_ERR_INVALID_ARG, "rows = %d is outside 1..%d", rows, kMaxEdgeRows);
    if (!aligned16(pred_cb) || !aligned16(succ_cb) || !aligned16(hidden) || !aligned16(pred_ids) ||
        !aligned16(cand_ids) || !aligned16(score))
        return fail(Q4_ERR_MISALIGNED, "codebooks, hidden, ids and score must be 16-byte aligned");
    int dev = 0;
    const DeviceInfo* info = nullptr;
    q4_status s = device_setup(&dev, &info);
    if (s != Q4_OK) return s;
    const cudaError_t e =
        launch_pdl(edges_kernel, dim3((unsigned)rows), dim3(kThreads), 0, reinterpret_cast<cudaStream_t>(stream),
                   static_cast<const uint16_t*>(pred_cb), static_cast<const uint16_t*>(succ_cb), V, R, hidden,
                   pred_ids, cand_ids, score, info->error_word);
    if (e != cudaSuccess) return cuda_fail(e, "launching the edge-score kernel");
    return Q4_OK;
}

q4_status q4_check_wait_timeout(long long limit_cycles, q4_stream_t stream) {
    g_last_error.clear();
    if (limit_cycles < 1 || limit_cycles > (1ll << 32))
        return fail(Q4_ERR_INVALID_ARG, "limit_cycles must be in 1..2^32 (got %lld)", limit_cycles);
    int dev = 0;
    const DeviceInfo* info = nullptr;
    q4_status s = device_setup(&dev, &info);
    if (s != Q4_OK) return s;
    wait_check_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_cycles, info->error_word);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launching the wait check");
    return Q4_OK;
}

q4_status q4_device_status(q4_stream_t stream) {
    g_last_error.clear();
    // No set-up here: this call allocates nothing, so a caller of
    // q4_matmul_noalloc can use it too.  It reads the error word through the
    // symbol of the current device.
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, q4_device_error_word, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(q4_device_error_word, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
        if (word & ~q4::edges::kErrBadIndex) {
            // A CTA that gave up a wait skipped its arrivals on the split-K and
            // top-k counters, which the next launch expects at zero: clear them
            // (q4_matmul_noalloc clears its own on every call).
            e = reset_counters(dev);
            if (e != cudaSuccess) return cuda_fail(e, "clearing the library's arrival counters");
        }
        if (word & q4::edges::kErrBadIndex)
            return fail(Q4_ERR_INVALID_INDEX, "a codebook id was outside 0..V-1 (error word 0x%x)", word);
        return fail(Q4_ERR_TIMEOUT, "a device-side wait gave up (error word 0x%x)", word);
    }
    return Q4_OK;
}

const char* q4_last_error(void) { return g_last_error.c_str(); }

#ifdef Q4_TRACE
// Developer timing trace (only in builds made with -DQ4_TRACE).
void q4_debug_set_trace(void* device_buffer) { g_trace = static_cast<unsigned long long*>(device_buffer); }
#endif

const char* q4_status_string(q4_status s) {
    switch (s) {
        case Q4_OK: return "Q4_OK";
        case Q4_ERR_INVALID_ARG: return "Q4_ERR_INVALID_ARG";
        case Q4_ERR_UNSUPPORTED_SHAPE: return "Q4_ERR_UNSUPPORTED_SHAPE";
        case Q4_ERR_MISALIGNED: return "Q4_ERR_MISALIGNED";
        case Q4_ERR_UNSUPPORTED_DEVICE: return "Q4_ERR_UNSUPPORTED_DEVICE";
        case Q4_ERR_CUDA: return "Q4_ERR_CUDA";
        case Q4_ERR_TIMEOUT: return "Q4_ERR_TIMEOUT";
        case Q4_ERR_OVERFLOW: return "Q4_ERR_OVERFLOW";
        case Q4_ERR_INVALID_INDEX: return "Q4_ERR_INVALID_INDEX";
    }
    return "Q4_ERR_UNKNOWN";
}

}  // extern "C"
