// noalloc.cu -- fp8_linear_bwd_noalloc: the backward pass of the FP8 linear
// layer for callers that cannot allocate device memory.
//
// fp8_linear_bwd needs two FP8 work buffers (dY8 [M][N] and dY8t [N][M]) that
// live only for the duration of the call.  Some callers cannot provide them:
// a plugin that a host framework hands only the input and output tensors
// (the framework's allocator owns all device memory and offers no workspace
// hook), or code that must not call cudaMalloc / cudaFree because cudaFree
// waits for the whole device.  This variant keeps those two buffers in a
// fixed array in the library's own device memory instead, so the caller
// passes only inputs and outputs and nothing is allocated at call time.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (64 MiB) until the process exits.  In host code the
// array's name is only a host-side stand-in, not a device address, so its
// device address is looked up once per device with cudaGetSymbolAddress.
// That address belongs to the device's primary context: after a
// cudaDeviceReset of a device this entry point must not be called again on
// that device in the same process.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/fp8amax.h"
#include "kernels.h"

namespace {

// Largest dY this variant accepts: M * N <= 2^25 elements, i.e. two FP8
// copies of 32 MiB each (for example M = 4096 tokens, N = 8192 features).
constexpr int64_t kMaxElems = int64_t(1) << 25;

// dY8 in [0, kMaxElems), dY8t in [kMaxElems, 2 * kMaxElems).  Every call
// overwrites the part it uses before reading it, so nothing needs to start
// at zero; the previous call's bytes simply stay behind.
static __device__ __align__(256) uint8_t g_bwd_scratch[2 * kMaxElems];

constexpr int kMaxDevices = 64;
uint8_t *g_scratch_ptr[kMaxDevices] = {};
cudaError_t g_scratch_err[kMaxDevices] = {};
std::once_flag g_scratch_once[kMaxDevices];

}  // namespace

extern "C" {

fp8_status fp8_linear_bwd_noalloc(const void *dY, int64_t M, int64_t N, int64_t K,
                                  const fp8_meta *meta, const fp8_recipe *recipe,
                                  const uint8_t *X8t, const uint8_t *W8t, void *dX, void *dW,
                                  void *stream) {
    const fp8k::CallRange range("fp8_linear_bwd_noalloc");
    char msg[256];
    // Only the work-area limit is checked here; negative or misaligned sizes
    // and bad pointers are reported by fp8_linear_bwd's own checks below.
    if (M > 0 && N > 0 && N > kMaxElems / M) {
        snprintf(msg, sizeof msg,
                 "fp8_linear_bwd_noalloc: M=%lld x N=%lld exceeds the fixed work area of "
                 "%lld elements; use fp8_linear_bwd with caller-provided buffers",
                 (long long)M, (long long)N, (long long)kMaxElems);
        fp8k::set_last_error(msg);
        return FP8_ERR_ARG;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        fp8k::set_last_error("fp8_linear_bwd_noalloc: no usable current device");
        return FP8_ERR_CUDA;
    }
    // Set-up, once per device, with that device current: the device address
    // of the array.  The first call on a device does this, so make that first
    // call before any stream capture.
    std::call_once(g_scratch_once[dev], [dev] {
        void *p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_bwd_scratch);
        g_scratch_ptr[dev] = static_cast<uint8_t *>(p);
    });
    if (g_scratch_err[dev] != cudaSuccess || g_scratch_ptr[dev] == nullptr) {
        snprintf(msg, sizeof msg, "fp8_linear_bwd_noalloc: cudaGetSymbolAddress: %s",
                 cudaGetErrorString(g_scratch_err[dev]));
        fp8k::set_last_error(msg);
        return FP8_ERR_CUDA;
    }
    uint8_t *dY8 = g_scratch_ptr[dev];
    uint8_t *dY8t = g_scratch_ptr[dev] + kMaxElems;
    return fp8_linear_bwd(dY, M, N, K, meta, recipe, X8t, W8t, dY8, dY8t, dX, dW, stream);
}

}  // extern "C"
