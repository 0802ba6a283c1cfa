// api.cu -- the C ABI (include/fp8fg.h): argument validation, device checks,
// the library-owned device status word, and dispatch to the kernels.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/fp8fg.h"
#include "kernels.h"

namespace fp8fg {
namespace {

// Asynchronous errors recorded by kernels (bounded waits, grouped offsets).
__device__ int g_device_status;
// The value fp8fg_last_device_status took out of g_device_status, copied to
// the host from here.
__device__ int g_status_taken;

// Read and clear the status word in one atomic step, so that a kernel on
// another stream recording an error between a read and a separate clear
// cannot have it wiped.
__global__ void take_status_kernel() { g_status_taken = atomicExch(&g_device_status, 0); }
std::mutex g_take_mu;   // g_status_taken is one word per device: one reader at a time

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int ok = 0;             // 1 once probed successfully
    int supported = 0;      // compute capability 10.3
    int num_sms = 0;
    int* status_word = nullptr;
};

DeviceInfo g_dev[kMaxDevices];
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};
std::mutex g_dev_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Scale arrays are read and written one float at a time (except the GEMM's
// per-row B scales, read in 8-byte pairs): 4-byte alignment suffices.
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Probe the current device once; returns a library status.
int current_device(DeviceInfo** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kErrCuda;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ok) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return kErrCuda;
        d.supported = fp8fg_check_compute_capability(major, minor) == kOk;
        d.num_sms = sms;
        if (d.supported) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return kErrCuda;
            d.status_word = static_cast<int*>(addr);
        }
        d.ok = 1;
    }
    if (!d.supported) return kErrUnsupported;
    *out = &d;
    return kOk;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? kOk : kErrCuda; }

}  // namespace
}  // namespace fp8fg

using namespace fp8fg;

extern "C" {

int fp8_quant_act_1x128(const void* x_bf16, int64_t rows, int64_t cols, int axis, uint8_t* q, float* scales,
                        cudaStream_t stream) {
    if (rows < 0 || cols < 0) return kErrInvalidArg;
    if (axis != FP8FG_AXIS_COLS && axis != FP8FG_AXIS_ROWS) return kErrInvalidArg;
    if (axis == FP8FG_AXIS_COLS && cols % 128 != 0) return kErrInvalidArg;
    if (axis == FP8FG_AXIS_ROWS && (rows % 128 != 0 || cols % 8 != 0)) return kErrInvalidArg;
    if (rows == 0 || cols == 0) return kOk;
    if (!x_bf16 || !q || !scales) return kErrInvalidArg;
    if (rows > (int64_t(1) << 40) / cols) return kErrInvalidArg;
    // the 1x128 kernel's grid: (rows / 64) blocks by (cols / 128) group columns
    if (axis == FP8FG_AXIS_COLS && (cols / 128 > 65535 || rows / 64 >= (int64_t(1) << 31))) return kErrInvalidArg;
    if (!aligned16(x_bf16) || !aligned16(q) || !aligned4(scales)) return kErrMisaligned;
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != kOk) return st;
    if (axis == FP8FG_AXIS_COLS) return from_cuda(launch_quant_act_rows(x_bf16, rows, cols, q, scales, d->num_sms, stream));
    return from_cuda(launch_quant_act_cols(x_bf16, rows, cols, q, scales, d->num_sms, stream));
}

int fp8_quant_act_dual(const void* x_bf16, int64_t rows, int64_t cols, uint8_t* q_row, float* s_row,
                       uint8_t* q_col_t, float* s_col, cudaStream_t stream) {
    if (rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0) return kErrInvalidArg;
    if (rows == 0 || cols == 0) return kOk;
    if (!x_bf16 || !q_row || !s_row || !q_col_t || !s_col) return kErrInvalidArg;
    if (rows > (int64_t(1) << 40) / cols) return kErrInvalidArg;
    // grid: (rows / 128) x (cols / 128) tiles
    if (cols / 128 > 65535) return kErrInvalidArg;
    if (!aligned16(x_bf16) || !aligned16(q_row) || !aligned4(s_row) || !aligned16(q_col_t) || !aligned4(s_col))
        return kErrMisaligned;
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != kOk) return st;
    return from_cuda(launch_quant_act_dual(x_bf16, rows, cols, q_row, s_row, q_col_t, s_col, d->num_sms, stream));
}

int fp8_quant_w_128x128(const float* w, int64_t rows, int64_t cols, uint8_t* q, uint8_t* q_t, float* scales,
                        cudaStream_t stream) {
    if (rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0) return kErrInvalidArg;
    if (rows == 0 || cols == 0) return kOk;
    if (!w || !q || !scales) return kErrInvalidArg;
    if (rows > (int64_t(1) << 40) / cols) return kErrInvalidArg;
    if (!aligned16(w) || !aligned16(q) || !aligned4(scales) || (q_t && !aligned16(q_t))) return kErrMisaligned;
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != kOk) return st;
    return from_cuda(launch_quant_w(w, rows, cols, q, q_t, scales, d->num_sms, stream));
}

static int gemm_common(const GemmArgs& a, cudaStream_t stream) {
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != kOk) return st;
    if (a.K == 0) {
        const size_t elt = a.out_bf16 ? 2 : 4;
        return from_cuda(cudaMemsetAsync(a.d, 0, static_cast<size_t>(a.M) * a.N * elt, stream));
    }
    cudaError_t ce = cudaSuccess;
    GemmArgs b = a;
    b.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    return launch_gemm(b, d->num_sms, d->status_word, stream, &ce);
}

// Shape rules shared by the dense and grouped GEMMs.  TMA addresses rows of
// up to 2^32 elements per dimension; the limits below keep every index and
// byte count far inside int64 and the tensor-map ranges.
// ragged_m: M need not be a multiple of 128 (the last row tile is partial).
static int check_gemm_shape(int64_t M, int64_t N, int64_t K, int out_dtype, bool ragged_m = false) {
    if (M < 0 || N < 0 || K < 0) return kErrInvalidArg;
    if ((!ragged_m && M % 128 != 0) || N % 128 != 0 || K % 128 != 0) return kErrInvalidArg;
    if (out_dtype != FP8FG_OUT_F32 && out_dtype != FP8FG_OUT_BF16) return kErrInvalidArg;
    const int64_t lim = int64_t(1) << 31;
    if (M > lim || N > lim || K > lim) return kErrInvalidArg;
    // output tiles of 128 x 256 are numbered with 32-bit integers
    if (((M + 127) / 128) * ((N + 255) / 256) >= lim) return kErrInvalidArg;
    return kOk;
}

int fp8_gemm_blockscaled(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb, int bscale,
                         int64_t sb_stride_n, int64_t sb_stride_k, void* d, int out_dtype, int64_t M, int64_t N,
                         int64_t K, cudaStream_t stream) {
    if (bscale != FP8FG_BSCALE_BLOCK128 && bscale != FP8FG_BSCALE_ROW) return kErrInvalidArg;
    // block B scales (Fprop, Dgrad: M = tokens) take any M; per-row B scales
    // (Wgrad: M = output channels) need whole row tiles
    int st = check_gemm_shape(M, N, K, out_dtype, bscale == FP8FG_BSCALE_BLOCK128);
    if (st != kOk) return st;
    if (bscale == FP8FG_BSCALE_BLOCK128 && (sb_stride_n < 0 || sb_stride_k < 0)) return kErrInvalidArg;
    if (M == 0 || N == 0) return kOk;
    if (!d) return kErrInvalidArg;
    if (K > 0 && (!a || !sa || !b || !sb)) return kErrInvalidArg;
    // per-row B scales: both scale arrays 16-byte aligned (B scales are read in 8-byte pairs)
    const bool row = bscale == FP8FG_BSCALE_ROW;
    const bool sa_ok = row ? aligned16(sa) : aligned4(sa);
    const bool sb_ok = row ? aligned16(sb) : aligned4(sb);
    if (!aligned16(d) || (K > 0 && (!aligned16(a) || !sa_ok || !aligned16(b) || !sb_ok)))
        return kErrMisaligned;
    GemmArgs g{};
    g.a = a;
    g.sa = sa;
    g.b = b;
    g.sb = sb;
    g.bscale = bscale;
    g.sb_stride_n = sb_stride_n;
    g.sb_stride_k = sb_stride_k;
    g.d = d;
    g.out_bf16 = out_dtype == FP8FG_OUT_BF16;
    g.M = M;
    g.N = N;
    g.K = K;
    g.offsets = nullptr;
    g.G = 0;
    return gemm_common(g, stream);
}

int fp8_gemm_quant_a(const void* a_bf16, uint8_t* q_a, float* s_a, const uint8_t* b, const float* sb,
                     int64_t sb_stride_n, int64_t sb_stride_k, void* d, int out_dtype, int64_t M, int64_t N,
                     int64_t K, int32_t* band_flags, cudaStream_t stream) {
    int st = check_gemm_shape(M, N, K, out_dtype);
    if (st != kOk) return st;
    if (sb_stride_n < 0 || sb_stride_k < 0) return kErrInvalidArg;
    if (M == 0) return kOk;
    // with K == 0 there is nothing to read or quantize: only d is touched
    if ((K > 0 && (!a_bf16 || !q_a || !s_a || !band_flags)) || (N > 0 && (!d || (K > 0 && (!b || !sb)))))
        return kErrInvalidArg;
    if (M > (int64_t(1) << 40) / (K > 0 ? K : 1)) return kErrInvalidArg;
    if ((K > 0 && (!aligned16(a_bf16) || !aligned16(q_a) || !aligned4(s_a) || !aligned4(band_flags))) ||
        (N > 0 && (!aligned16(d) || (K > 0 && (!aligned16(b) || !aligned4(sb))))))
        return kErrMisaligned;
    DeviceInfo* dv = nullptr;
    st = current_device(&dv);
    if (st != kOk) return st;
    if (K == 0) {
        // no groups to quantize; D = 0
        if (N == 0) return kOk;
        const size_t elt = out_dtype == FP8FG_OUT_BF16 ? 2 : 4;
        return from_cuda(cudaMemsetAsync(d, 0, static_cast<size_t>(M) * N * elt, stream));
    }
    // the 1x128 quantizer's grid limits (a GEMM with no columns is that quantizer alone)
    if (K / 128 > 65535 || M / 64 >= (int64_t(1) << 31)) return kErrInvalidArg;
    if (N == 0) return from_cuda(launch_quant_act_rows(a_bf16, M, K, q_a, s_a, dv->num_sms, stream));
    GemmArgs g{};
    g.a = q_a;
    g.sa = s_a;
    g.b = b;
    g.sb = sb;
    g.bscale = FP8FG_BSCALE_BLOCK128;
    g.sb_stride_n = sb_stride_n;
    g.sb_stride_k = sb_stride_k;
    g.d = d;
    g.out_bf16 = out_dtype == FP8FG_OUT_BF16;
    g.M = M;
    g.N = N;
    g.K = K;
    g.offsets = nullptr;
    g.G = 0;
    g.xa = a_bf16;
    g.band_flags = band_flags;
    return gemm_common(g, stream);
}

int fp8_gemm_grouped(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                     const int32_t* group_offsets, int G, void* d, int out_dtype, int64_t M_total, int64_t N,
                     int64_t K, cudaStream_t stream) {
    int st = check_gemm_shape(M_total, N, K, out_dtype);
    if (st != kOk) return st;
    if (G < 1 || G > 4096) return kErrInvalidArg;
    if (!group_offsets) return kErrInvalidArg;
    if (M_total == 0 || N == 0) return kOk;
    if (!d) return kErrInvalidArg;
    if (K > 0 && (!a || !sa || !b || !sb)) return kErrInvalidArg;
    if (!aligned16(d) || (K > 0 && (!aligned16(a) || !aligned4(sa) || !aligned16(b) || !aligned4(sb))) ||
        (reinterpret_cast<uintptr_t>(group_offsets) & 3u))
        return kErrMisaligned;
    GemmArgs g{};
    g.a = a;
    g.sa = sa;
    g.b = b;
    g.sb = sb;
    g.bscale = FP8FG_BSCALE_BLOCK128;
    g.sb_stride_n = K / 128;
    g.sb_stride_k = 1;
    g.d = d;
    g.out_bf16 = out_dtype == FP8FG_OUT_BF16;
    g.M = M_total;
    g.N = N;
    g.K = K;
    g.offsets = group_offsets;
    g.G = G;
    return gemm_common(g, stream);
}

int fp8fg_check_compute_capability(int major, int minor) {
    return major == 10 && minor == 3 ? kOk : kErrUnsupported;
}

const char* fp8fg_status_string(int status) {
    switch (status) {
        case FP8FG_OK: return "FP8FG_OK";
        case FP8FG_ERR_INVALID_ARG: return "FP8FG_ERR_INVALID_ARG: invalid argument (null pointer, enum or shape)";
        case FP8FG_ERR_MISALIGNED: return "FP8FG_ERR_MISALIGNED: a pointer is not 16-byte aligned";
        case FP8FG_ERR_UNSUPPORTED_DEVICE: return "FP8FG_ERR_UNSUPPORTED_DEVICE: the current device is not sm_103";
        case FP8FG_ERR_CUDA: return "FP8FG_ERR_CUDA: a CUDA call or a kernel launch failed";
        case FP8FG_ERR_TIMEOUT: return "FP8FG_ERR_TIMEOUT: a bounded device wait ran out";
        case FP8FG_ERR_TEARDOWN: return "FP8FG_ERR_TEARDOWN: after a failed wait, a kernel's wait for its own copies "
                                        "or MMAs in flight also ran out before it released its resources";
        case FP8FG_ERR_TOO_LARGE:
            return "FP8FG_ERR_TOO_LARGE: the problem exceeds a fixed-size library buffer "
                   "(fp8_gemm_quant_a_noalloc: M must be <= 524288)";
        default: return "FP8FG: unknown status";
    }
}

int fp8fg_last_device_status(cudaStream_t stream) {
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != kOk) return st;
    int value = 0;
    std::lock_guard<std::mutex> lock(g_take_mu);
    take_status_kernel<<<1, 1, 0, stream>>>();
    if (cudaPeekAtLastError() != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&value, g_status_taken, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return kErrCuda;
    return value;
}

int fp8fg_set_wait_limit(int64_t limit_ns) {
    if (limit_ns < 0 || static_cast<uint64_t>(limit_ns) > kMaxWaitLimitNs) return kErrInvalidArg;
    g_wait_limit_ns.store(limit_ns == 0 ? kWaitLimitNs : static_cast<uint64_t>(limit_ns), std::memory_order_relaxed);
    return kOk;
}

int fp8fg_selftest_watchdog(int64_t timeout_ns, cudaStream_t stream) {
    if (timeout_ns < 1 || timeout_ns > 1000000000) return kErrInvalidArg;
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != kOk) return st;
    return from_cuda(launch_watchdog_selftest(static_cast<uint64_t>(timeout_ns), d->status_word, stream));
}

int fp8fg_probe_mma_rate(int64_t chunks, int* num_ctas, cudaStream_t stream) {
    if (chunks < 1 || chunks > (int64_t(1) << 24) || !num_ctas) return kErrInvalidArg;
    DeviceInfo* d = nullptr;
    int st = current_device(&d);
    if (st != kOk) return st;
    *num_ctas = d->num_sms;
    return from_cuda(launch_mma_rate_probe(chunks, d->num_sms, g_wait_limit_ns.load(std::memory_order_relaxed),
                                           d->status_word, stream));
}

}  // extern "C"
