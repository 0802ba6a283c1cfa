// kernels.h -- internal launchers behind the C ABI (host code only).
// Arguments are validated by the C ABI layer before any launcher runs.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace fp8fg {

// Library status codes (mirror fp8fg_status of the public header).
enum : int {
    kOk = 0,
    kErrInvalidArg = 1,
    kErrMisaligned = 2,
    kErrUnsupported = 3,
    kErrCuda = 4,
    kErrTimeout = 5,
    kErrTeardown = 6
};

// Bounded device waits give up after this long (nanoseconds) by default;
// fp8fg_set_wait_limit() changes it within [1, kMaxWaitLimitNs].
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kMaxWaitLimitNs = 10000000000ull;

cudaError_t launch_quant_act_rows(const void* x, int64_t rows, int64_t cols, uint8_t* q, float* scales, int num_sms,
                                  cudaStream_t stream);
cudaError_t launch_quant_act_cols(const void* x, int64_t rows, int64_t cols, uint8_t* q, float* scales, int num_sms,
                                  cudaStream_t stream);
cudaError_t launch_quant_act_dual(const void* x, int64_t rows, int64_t cols, uint8_t* q_row, float* s_row,
                                  uint8_t* q_col_t, float* s_col, int num_sms, cudaStream_t stream);
cudaError_t launch_quant_w(const float* w, int64_t rows, int64_t cols, uint8_t* q, uint8_t* q_t, float* scales,
                           int num_sms, cudaStream_t stream);

struct GemmArgs {
    const uint8_t* a;
    const float* sa;
    const uint8_t* b;
    const float* sb;
    int bscale;               // 0: 128x128 blocks, 1: per row of B per K chunk
    int64_t sb_stride_n;      // block mode strides, in elements
    int64_t sb_stride_k;
    void* d;
    int out_bf16;
    int64_t M, N, K;
    const int32_t* offsets;   // grouped: device int32[G+1]; nullptr for a dense GEMM
    int G;
    uint64_t wait_limit_ns;   // limit of the kernel's bounded waits
    // fused A quantization (block B scales, dense only): when xa is set the
    // kernel first writes the 1x128 codes of the BF16 xa[M, K] to a (as
    // uint8_t*) and their scales to sa, then runs the GEMM on them;
    // band_flags: device int32[M/128], zeroed by the launcher
    const void* xa;
    int32_t* band_flags;
};

// Returns a library status code; `cuda_err` receives the CUDA error when the
// status is kErrCuda.
int launch_gemm(const GemmArgs& args, int num_sms, int* status_word, cudaStream_t stream, cudaError_t* cuda_err);

cudaError_t launch_watchdog_selftest(uint64_t timeout_ns, int* status_word, cudaStream_t stream);

// One CTA per SM issuing `chunks` x 4 back-to-back FP8 MMAs (128 x 256 x 32).
cudaError_t launch_mma_rate_probe(int64_t chunks, int num_sms, uint64_t limit_ns, int* status_word,
                                  cudaStream_t stream);

}  // namespace fp8fg
