// noalloc.cu -- fp8_gemm_quant_a without a caller-provided workspace.
//
// fp8_gemm_quant_a needs a small device workspace (one int32 counter per
// 128-row band of A).  Some callers cannot provide it: code that owns no
// allocator (a C host program handed raw device pointers by another runtime,
// a plugin whose host framework forbids it to allocate device memory behind
// the framework's allocator), or code that must not allocate in its steady
// state (a serving loop with a fixed memory budget).  This file keeps the
// workspace in a fixed array in the library's own device memory instead: the
// array exists on every GPU that loads the library, from the load until the
// process exits, and this entry point allocates nothing.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fp8fg.h"
#include "kernels.h"

namespace {

// The shared workspace: band counters for A operands of up to
// kNoAllocMaxBands * 128 rows (16 KB per GPU).
constexpr int64_t kNoAllocMaxBands = 4096;
static __device__ __align__(256) int32_t g_noalloc_band_flags[kNoAllocMaxBands];

// The array's device address on each device.  In host code the array's name
// stands for a host-side shadow, not device memory, so the address is asked
// from the runtime once per device, with that device current.
constexpr int kMaxDevices = 64;
int32_t* g_flags_addr[kMaxDevices] = {};
std::mutex g_flags_mu;

// Device address of the array on the current device (looked up on the first
// call on that device); nullptr if the lookup failed.
int32_t* flags_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_flags_mu);
    if (!g_flags_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_band_flags) != cudaSuccess || !ptr) return nullptr;
        g_flags_addr[dev] = static_cast<int32_t*>(ptr);
    }
    return g_flags_addr[dev];
}

}  // namespace

extern "C" int fp8_gemm_quant_a_noalloc(const void* a_bf16, uint8_t* q_a, float* s_a, const uint8_t* b,
                                        const float* sb, int64_t sb_stride_n, int64_t sb_stride_k, void* d,
                                        int out_dtype, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    // the array holds one counter per 128-row band of A
    if (M > kNoAllocMaxBands * 128) return FP8FG_ERR_TOO_LARGE;
    int32_t* flags = nullptr;
    if (M > 0 && K > 0) {
        flags = flags_on_current_device();
        if (!flags) return FP8FG_ERR_CUDA;
    }
    // fp8_gemm_quant_a checks the rest and zeroes the counters on `stream`
    // before its kernel
    return fp8_gemm_quant_a(a_bf16, q_a, s_a, b, sb, sb_stride_n, sb_stride_k, d, out_dtype, M, N, K, flags, stream);
}
