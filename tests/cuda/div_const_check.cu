// Exhaustive check of the library's division by a divisor known in advance
// (div_by_const2 in common.cuh, used for Adam's bias corrections): for one
// divisor b, every binary32 bit pattern a is divided both ways, and the
// result must equal the IEEE division __fdiv_rn(a, b) bit for bit (any NaN
// for a NaN).  Test infrastructure: built and loaded only by the GPU tests.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../fp8_mixed_precision_amax_gb300/csrc/common.cuh"

namespace {

__device__ bool same(float x, float y) {
    return __float_as_uint(x) == __float_as_uint(y) || (x != x && y != y);
}

__global__ void check_kernel(float b, unsigned long long *bad, unsigned *first_bad) {
    const fp8k::DivConst d = fp8k::div_const(b);
    const uint64_t pairs = 1ull << 31;
    for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < pairs;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const uint32_t u0 = static_cast<uint32_t>(2 * i), u1 = u0 + 1;
        const float a0 = __uint_as_float(u0), a1 = __uint_as_float(u1);
        float q0, q1;
        fp8k::div_by_const2(a0, a1, d, q0, q1);
        const bool ok0 = same(q0, __fdiv_rn(a0, b)), ok1 = same(q1, __fdiv_rn(a1, b));
        if (!ok0) {
            atomicAdd(bad, 1ull);
            atomicMin(first_bad, u0);
        }
        if (!ok1) {
            atomicAdd(bad, 1ull);
            atomicMin(first_bad, u1);
        }
    }
}

__global__ void one_kernel(float a, float b, float *out) {
    const fp8k::DivConst d = fp8k::div_const(b);
    fp8k::div_by_const2(a, a, d, out[0], out[1]);
    out[2] = __fdiv_rn(a, b);
}

}  // namespace

// Returns 0 and the number of mismatches (and the smallest mismatching bit
// pattern, 0xFFFFFFFF if none), or a CUDA error code.
extern "C" int div_const_check(float b, int blocks, unsigned long long *bad_out,
                               unsigned *first_bad_out) {
    unsigned long long *bad = nullptr;
    unsigned *first = nullptr;
    cudaError_t e = cudaMalloc(&bad, sizeof *bad);
    if (e == cudaSuccess) e = cudaMalloc(&first, sizeof *first);
    if (e == cudaSuccess) e = cudaMemset(bad, 0, sizeof *bad);
    if (e == cudaSuccess) e = cudaMemset(first, 0xFF, sizeof *first);
    if (e == cudaSuccess) {
        check_kernel<<<blocks, 256>>>(b, bad, first);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(bad_out, bad, sizeof *bad, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(first_bad_out, first, sizeof *first, cudaMemcpyDeviceToHost);
    cudaFree(bad);
    cudaFree(first);
    return static_cast<int>(e);
}

// One quotient both ways: out[0], out[1] from div_by_const2, out[2] IEEE.
extern "C" int div_const_one(float a, float b, float *out_host) {
    float *out = nullptr;
    cudaError_t e = cudaMalloc(&out, 3 * sizeof(float));
    if (e == cudaSuccess) {
        one_kernel<<<1, 1>>>(a, b, out);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(out_host, out, 3 * sizeof(float), cudaMemcpyDeviceToHost);
    cudaFree(out);
    return static_cast<int>(e);
}
