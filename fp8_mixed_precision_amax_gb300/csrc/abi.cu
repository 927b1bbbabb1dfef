// abi.cu -- the exported C entry points (include/fp8amax.h): argument checks
// on the host, then the launches, in stream order, of the kernels in cast.cu
// and gemm.cu.  No device memory is allocated here and the stream is never
// synchronized (except by fp8_sync_status).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/fp8amax.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

fp8_status fail(fp8_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

fp8_status cuda_fail(cudaError_t e, const char *where) {
    return fail(FP8_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    int sm_count = 0;
    bool supported = false;
};
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

// SM count of the current device; FP8_ERR_UNSUPPORTED unless it is an sm_103 GPU.
fp8_status current_device(int *sm_count) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(FP8_ERR_UNSUPPORTED, "device index %d", dev);
    std::call_once(g_dev_once[dev], [dev] {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_dev[dev].sm_count = sms;
        g_dev[dev].supported = (major == 10 && minor == 3);
    });
    if (!g_dev[dev].supported)
        return fail(FP8_ERR_UNSUPPORTED, "device %d is not an sm_103 GPU", dev);
    *sm_count = g_dev[dev].sm_count;
    return FP8_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fp8_status check_dims16(const char *fn, int64_t a, const char *na, int64_t b, const char *nb) {
    if (a < 0 || b < 0) return fail(FP8_ERR_ARG, "%s: negative size (%s=%lld, %s=%lld)", fn, na,
                                    (long long)a, nb, (long long)b);
    if (a % 16 || b % 16)
        return fail(FP8_ERR_ALIGN, "%s: %s=%lld and %s=%lld must be multiples of 16", fn, na,
                    (long long)a, nb, (long long)b);
    if (a > (int64_t(1) << 31) || b > (int64_t(1) << 31))
        return fail(FP8_ERR_ARG, "%s: dimension above 2^31", fn);
    return FP8_OK;
}

fp8_status check_ptr(const char *fn, const void *p, const char *name, bool may_be_null) {
    if (p == nullptr) {
        if (may_be_null) return FP8_OK;
        return fail(FP8_ERR_ARG, "%s: %s is NULL", fn, name);
    }
    if (!aligned16(p)) return fail(FP8_ERR_ALIGN, "%s: %s is not 16-byte aligned", fn, name);
    return FP8_OK;
}

// A pointer to one fp32 scalar (scale, scale_inv, amax) needs 4-byte alignment.
fp8_status check_scalar(const char *fn, const void *p, const char *name, bool may_be_null) {
    if (p == nullptr) {
        if (may_be_null) return FP8_OK;
        return fail(FP8_ERR_ARG, "%s: %s is NULL", fn, name);
    }
    if (reinterpret_cast<uintptr_t>(p) & 3u)
        return fail(FP8_ERR_ALIGN, "%s: %s is not 4-byte aligned", fn, name);
    return FP8_OK;
}

#define FP8_TRY(expr)                       \
    do {                                    \
        fp8_status s_ = (expr);             \
        if (s_ != FP8_OK) return s_;        \
    } while (0)

#define FP8_CUDA(expr, where)                          \
    do {                                               \
        cudaError_t e_ = (expr);                       \
        if (e_ != cudaSuccess) return cuda_fail(e_, where); \
    } while (0)

fp8_status check_meta(const char *fn, const fp8_meta *m, const fp8_recipe *r) {
    if (m == nullptr || r == nullptr) return fail(FP8_ERR_ARG, "%s: meta or recipe is NULL", fn);
    if (m->history == nullptr || m->amax == nullptr || m->scale == nullptr ||
        m->scale_inv == nullptr)
        return fail(FP8_ERR_ARG, "%s: a meta buffer is NULL", fn);
    if ((reinterpret_cast<uintptr_t>(m->history) | reinterpret_cast<uintptr_t>(m->amax) |
         reinterpret_cast<uintptr_t>(m->scale) | reinterpret_cast<uintptr_t>(m->scale_inv)) & 3u)
        return fail(FP8_ERR_ALIGN, "%s: a meta buffer is not 4-byte aligned", fn);
    if (r->margin < 0 || r->margin > 64)
        return fail(FP8_ERR_ARG, "%s: margin %d outside [0, 64]", fn, r->margin);
    if (r->history_len < 1 || r->history_len > 8192 || m->history_len != r->history_len)
        return fail(FP8_ERR_ARG, "%s: history_len %d (meta %d) must match and lie in [1, 8192]",
                    fn, r->history_len, m->history_len);
    if (r->hybrid != 0 && r->hybrid != 1)
        return fail(FP8_ERR_ARG, "%s: hybrid must be 0 or 1", fn);
    if (r->scaling != FP8_SCALING_DELAYED && r->scaling != FP8_SCALING_CURRENT)
        return fail(FP8_ERR_ARG, "%s: scaling must be delayed (0) or current (1)", fn);
    return FP8_OK;
}

}  // namespace

void fp8k::set_last_error(const char *msg) { g_last_error = msg; }

extern "C" {

int32_t fp8_abi_version(void) { return FP8AMAX_ABI_VERSION; }

const char *fp8_last_error(void) { return g_last_error.c_str(); }

fp8_status fp8_sync_status(void *stream) {
    unsigned flags = 0;
    cudaError_t e = fp8k::read_and_clear_error_flag(&flags, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fp8_sync_status");
    if (flags & 1u) return fail(FP8_ERR_TIMEOUT, "a kernel gave up a bounded wait");
    return FP8_OK;
}

fp8_status fp8_selftest_wait_timeout(int64_t limit_ns, void *stream) {
    const char *fn = "fp8_selftest_wait_timeout";
    const fp8k::CallRange range(fn);
    if (limit_ns < 1 || limit_ns > 5000000000ll)
        return fail(FP8_ERR_ARG, "%s: limit_ns %lld outside [1, 5e9]", fn,
                    static_cast<long long>(limit_ns));
    FP8_CUDA(fp8k::launch_selftest_wait(static_cast<uint64_t>(limit_ns),
                                        static_cast<cudaStream_t>(stream)),
             fn);
    return FP8_OK;
}

fp8_status fp8_set_clock_probe(uint64_t *acc) {
    const fp8k::CallRange range("fp8_set_clock_probe");
    if (acc != nullptr && (reinterpret_cast<uintptr_t>(acc) & 7u) != 0)
        return fail(FP8_ERR_ALIGN, "fp8_set_clock_probe: acc must be 8-byte aligned");
    fp8k::set_clock_probe(reinterpret_cast<unsigned long long *>(acc));
    return FP8_OK;
}

fp8_status fp8_amax(const void *x, int64_t n, float *amax, void *stream) {
    const char *fn = "fp8_amax";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, n, "n", 0, "-"));
    FP8_TRY(check_ptr(fn, x, "x", n == 0));
    FP8_TRY(check_scalar(fn, amax, "amax", false));
    int sms;
    FP8_TRY(current_device(&sms));
    FP8_CUDA(fp8k::launch_amax(x, n, amax, sms, static_cast<cudaStream_t>(stream)), fn);
    return FP8_OK;
}

fp8_status fp8_quantize_f32(const float *x, int64_t n, const float *scale, int32_t fmt,
                            uint8_t *out, float *amax, void *stream) {
    const char *fn = "fp8_quantize_f32";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, n, "n", 0, "-"));
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(FP8_ERR_ARG, "%s: bad format %d", fn, fmt);
    FP8_TRY(check_ptr(fn, x, "x", n == 0));
    FP8_TRY(check_scalar(fn, scale, "scale", false));
    FP8_TRY(check_ptr(fn, out, "out", n == 0));
    FP8_TRY(check_scalar(fn, amax, "amax", true));
    int sms;
    FP8_TRY(current_device(&sms));
    FP8_CUDA(fp8k::launch_quantize_f32(x, n, scale, fmt, out, amax, sms,
                                       static_cast<cudaStream_t>(stream)),
             fn);
    return FP8_OK;
}

fp8_status fp8_quantize_transpose(const void *x, int64_t rows, int64_t cols, const float *scale,
                                  int32_t fmt, uint8_t *out, uint8_t *out_t, float *amax,
                                  void *stream) {
    const char *fn = "fp8_quantize_transpose";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, rows, "rows", cols, "cols"));
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(FP8_ERR_ARG, "%s: bad format %d", fn, fmt);
    const bool empty = rows == 0 || cols == 0;
    if (!empty && out == nullptr && out_t == nullptr)
        return fail(FP8_ERR_ARG, "%s: out and out_t are both NULL", fn);
    FP8_TRY(check_ptr(fn, x, "x", empty));
    FP8_TRY(check_scalar(fn, scale, "scale", false));
    FP8_TRY(check_ptr(fn, out, "out", true));
    FP8_TRY(check_ptr(fn, out_t, "out_t", true));
    FP8_TRY(check_scalar(fn, amax, "amax", true));
    int sms;
    FP8_TRY(current_device(&sms));
    FP8_CUDA(fp8k::launch_quantize_transpose(x, rows, cols, scale, fmt, out, out_t, amax, true, sms,
                                             static_cast<cudaStream_t>(stream)),
             fn);
    return FP8_OK;
}

fp8_status fp8_quantize_transpose_current(const void *x, int64_t rows, int64_t cols, int32_t fmt,
                                          int32_t margin, uint8_t *out, uint8_t *out_t,
                                          float *amax, float *scale, float *scale_inv,
                                          void *stream) {
    const char *fn = "fp8_quantize_transpose_current";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, rows, "rows", cols, "cols"));
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(FP8_ERR_ARG, "%s: bad format %d", fn, fmt);
    if (margin < 0 || margin > 64)
        return fail(FP8_ERR_ARG, "%s: margin %d outside [0, 64]", fn, margin);
    const bool empty = rows == 0 || cols == 0;
    if (!empty && out == nullptr && out_t == nullptr)
        return fail(FP8_ERR_ARG, "%s: out and out_t are both NULL", fn);
    FP8_TRY(check_ptr(fn, x, "x", empty));
    FP8_TRY(check_ptr(fn, out, "out", true));
    FP8_TRY(check_ptr(fn, out_t, "out_t", true));
    FP8_TRY(check_scalar(fn, amax, "amax", false));
    FP8_TRY(check_scalar(fn, scale, "scale", false));
    FP8_TRY(check_scalar(fn, scale_inv, "scale_inv", false));
    int sms;
    FP8_TRY(current_device(&sms));
    FP8_CUDA(fp8k::launch_quantize_transpose_current(x, rows, cols, fmt, margin, out, out_t, amax,
                                                     scale, scale_inv, sms,
                                                     static_cast<cudaStream_t>(stream)),
             fn);
    return FP8_OK;
}

fp8_status fp8_scale_update(float *history, const float *amax, float *scale, float *scale_inv,
                            int32_t num_tensors, int32_t history_len, uint32_t format_mask,
                            int32_t margin, void *stream) {
    const char *fn = "fp8_scale_update";
    const fp8k::CallRange range(fn);
    if (num_tensors < 1 || num_tensors > 32)
        return fail(FP8_ERR_ARG, "%s: num_tensors %d outside [1, 32]", fn, num_tensors);
    if (history_len < 1 || history_len > 8192)
        return fail(FP8_ERR_ARG, "%s: history_len %d outside [1, 8192]", fn, history_len);
    if (margin < 0 || margin > 64)
        return fail(FP8_ERR_ARG, "%s: margin %d outside [0, 64]", fn, margin);
    FP8_TRY(check_scalar(fn, history, "history", false));
    FP8_TRY(check_scalar(fn, amax, "amax", false));
    FP8_TRY(check_scalar(fn, scale, "scale", false));
    FP8_TRY(check_scalar(fn, scale_inv, "scale_inv", false));
    int sms;
    FP8_TRY(current_device(&sms));
    FP8_CUDA(fp8k::launch_scale_update(history, const_cast<float *>(amax), scale, scale_inv,
                                       num_tensors, history_len, format_mask, margin, false,
                                       static_cast<cudaStream_t>(stream)),
             fn);
    return FP8_OK;
}

fp8_status fp8_amax_scale_update(const fp8_meta *meta, const fp8_recipe *recipe, void *stream) {
    const char *fn = "fp8_amax_scale_update";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_meta(fn, meta, recipe));
    const uint32_t mask = recipe->hybrid ? ((1u << FP8_SLOT_DY) | (1u << FP8_SLOT_DX)) : 0u;
    int sms;
    FP8_TRY(current_device(&sms));
    // the five amax slots are consumed here and cleared for the next step
    FP8_CUDA(fp8k::launch_scale_update(meta->history, meta->amax, meta->scale, meta->scale_inv,
                                       FP8_NUM_SLOTS, meta->history_len, mask, recipe->margin,
                                       true, static_cast<cudaStream_t>(stream)),
             fn);
    return FP8_OK;
}

static fp8_status gemm_checked(const char *fn, const uint8_t *A, int32_t fa, const uint8_t *B,
                               int32_t fb, int64_t M, int64_t N, int64_t K, const float *sa,
                               const float *sb, void *D, float *d_amax, bool zero_amax, int sms,
                               cudaStream_t st) {
    const char *what = nullptr;
    cudaError_t e =
        fp8k::launch_gemm_tn(A, fa, B, fb, M, N, K, sa, sb, D, d_amax, zero_amax, sms, st, &what);
    if (e != cudaSuccess)
        return what ? fail(FP8_ERR_CUDA, "%s: %s", fn, what) : cuda_fail(e, fn);
    return FP8_OK;
}

fp8_status fp8_gemm_tn(const uint8_t *A, int32_t fa, const uint8_t *B, int32_t fb, int64_t M,
                       int64_t N, int64_t K, const float *a_scale_inv, const float *b_scale_inv,
                       void *D, float *d_amax, void *stream) {
    const char *fn = "fp8_gemm_tn";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, M, "M", N, "N"));
    FP8_TRY(check_dims16(fn, K, "K", 16, "-"));
    if (M < 16 || N < 16 || K < 16) return fail(FP8_ERR_ARG, "%s: M, N, K must be >= 16", fn);
    if ((fa != FP8_E4M3 && fa != FP8_E5M2) || (fb != FP8_E4M3 && fb != FP8_E5M2))
        return fail(FP8_ERR_ARG, "%s: bad operand format", fn);
    FP8_TRY(check_ptr(fn, A, "A", false));
    FP8_TRY(check_ptr(fn, B, "B", false));
    FP8_TRY(check_ptr(fn, D, "D", false));
    FP8_TRY(check_scalar(fn, a_scale_inv, "a_scale_inv", false));
    FP8_TRY(check_scalar(fn, b_scale_inv, "b_scale_inv", false));
    FP8_TRY(check_scalar(fn, d_amax, "d_amax", true));
    int sms;
    FP8_TRY(current_device(&sms));
    return gemm_checked(fn, A, fa, B, fb, M, N, K, a_scale_inv, b_scale_inv, D, d_amax, true, sms,
                        static_cast<cudaStream_t>(stream));
}

static fp8_status check_gemm(const char *fn, const fp8_gemm_desc &d) {
    FP8_TRY(check_dims16(fn, d.M, "M", d.N, "N"));
    FP8_TRY(check_dims16(fn, d.K, "K", 16, "-"));
    if (d.M < 16 || d.N < 16 || d.K < 16) return fail(FP8_ERR_ARG, "%s: M, N, K must be >= 16", fn);
    if ((d.fa != FP8_E4M3 && d.fa != FP8_E5M2) || (d.fb != FP8_E4M3 && d.fb != FP8_E5M2))
        return fail(FP8_ERR_ARG, "%s: bad operand format", fn);
    FP8_TRY(check_ptr(fn, d.A, "A", false));
    FP8_TRY(check_ptr(fn, d.B, "B", false));
    FP8_TRY(check_ptr(fn, d.D, "D", false));
    FP8_TRY(check_scalar(fn, d.a_scale_inv, "a_scale_inv", false));
    FP8_TRY(check_scalar(fn, d.b_scale_inv, "b_scale_inv", false));
    FP8_TRY(check_scalar(fn, d.d_amax, "d_amax", true));
    return FP8_OK;
}

fp8_status fp8_gemm_tn_grouped(const fp8_gemm_desc *descs, int32_t n, void *stream) {
    const char *fn = "fp8_gemm_tn_grouped";
    const fp8k::CallRange range(fn);
    if (descs == nullptr || n < 1 || n > 2) return fail(FP8_ERR_ARG, "%s: n must be 1 or 2", fn);
    fp8k::GemmSpec g[2];
    for (int i = 0; i < n; ++i) {
        FP8_TRY(check_gemm(fn, descs[i]));
        const fp8_gemm_desc &d = descs[i];
        g[i] = fp8k::GemmSpec{d.A, d.fa, d.B, d.fb, d.M, d.N, d.K, d.a_scale_inv, d.b_scale_inv,
                              d.D, d.d_amax, true};
    }
    int sms;
    FP8_TRY(current_device(&sms));
    const char *what = nullptr;
    cudaError_t e = fp8k::launch_gemm_group(g, n, sms, static_cast<cudaStream_t>(stream), &what);
    if (e != cudaSuccess)
        return what ? fail(FP8_ERR_CUDA, "%s: %s", fn, what) : cuda_fail(e, fn);
    return FP8_OK;
}

fp8_status fp8_quantize_transpose_grouped(const fp8_cast_desc *descs, int32_t n, int32_t fmt,
                                          void *stream) {
    const char *fn = "fp8_quantize_transpose_grouped";
    const fp8k::CallRange range(fn);
    if (descs == nullptr || n < 1 || n > 2) return fail(FP8_ERR_ARG, "%s: n must be 1 or 2", fn);
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(FP8_ERR_ARG, "%s: bad format %d", fn, fmt);
    fp8k::CastSpec c[2];
    for (int i = 0; i < n; ++i) {
        const fp8_cast_desc &d = descs[i];
        FP8_TRY(check_dims16(fn, d.rows, "rows", d.cols, "cols"));
        const bool empty = d.rows == 0 || d.cols == 0;
        if (!empty && d.out == nullptr && d.out_t == nullptr)
            return fail(FP8_ERR_ARG, "%s: out and out_t are both NULL", fn);
        FP8_TRY(check_ptr(fn, d.x, "x", empty));
        FP8_TRY(check_scalar(fn, d.scale, "scale", false));
        FP8_TRY(check_ptr(fn, d.out, "out", true));
        FP8_TRY(check_ptr(fn, d.out_t, "out_t", true));
        FP8_TRY(check_scalar(fn, d.amax, "amax", true));
        c[i] = fp8k::CastSpec{d.x, d.rows, d.cols, const_cast<float *>(d.scale), nullptr, d.out,
                              d.out_t, d.amax, true, nullptr, nullptr, nullptr, nullptr};
    }
    int sms;
    FP8_TRY(current_device(&sms));
    FP8_CUDA(fp8k::launch_cast_group(c, n, fmt, false, 0, sms, static_cast<cudaStream_t>(stream)),
             fn);
    return FP8_OK;
}

fp8_status fp8_dequant_sum(const uint8_t *parts, int32_t nranks, int64_t n, int32_t fmt,
                           const float *scale, void *out, void *stream) {
    const char *fn = "fp8_dequant_sum";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, n, "n", 0, "-"));
    if (nranks < 1 || nranks > 65536) return fail(FP8_ERR_ARG, "%s: nranks %d", fn, nranks);
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(FP8_ERR_ARG, "%s: bad format %d", fn, fmt);
    FP8_TRY(check_ptr(fn, parts, "parts", n == 0));
    FP8_TRY(check_ptr(fn, out, "out", n == 0));
    FP8_TRY(check_scalar(fn, scale, "scale", false));
    int sms;
    FP8_TRY(current_device(&sms));
    FP8_CUDA(fp8k::launch_dequant_sum(parts, nranks, n, fmt, scale, out, sms,
                                      static_cast<cudaStream_t>(stream)),
             fn);
    return FP8_OK;
}

fp8_status fp8_adam_step(const void *grad, int64_t n, uint8_t *m1, float *m1_scale,
                         float *m1_scale_inv, uint16_t *m2, uint16_t *w16, float *w_scale,
                         float *w_scale_inv, void *w_bf16, float *amax, const fp8_adam_hyper *hp,
                         void *stream) {
    const char *fn = "fp8_adam_step";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, n, "n", 0, "-"));
    if (hp == nullptr) return fail(FP8_ERR_ARG, "%s: hyper-parameters are NULL", fn);
    if (hp->margin < 0 || hp->margin > 64)
        return fail(FP8_ERR_ARG, "%s: margin %d outside [0, 64]", fn, hp->margin);
    if (!(hp->bias_correction1 > 0.0f) || !(hp->bias_correction2 > 0.0f))
        return fail(FP8_ERR_ARG, "%s: bias corrections must be > 0 (step >= 1)", fn);
    const bool empty = n == 0;
    FP8_TRY(check_ptr(fn, grad, "grad", empty));
    FP8_TRY(check_ptr(fn, m1, "m1", empty));
    FP8_TRY(check_ptr(fn, m2, "m2", empty));
    FP8_TRY(check_ptr(fn, w16, "w16", empty));
    FP8_TRY(check_ptr(fn, w_bf16, "w_bf16", empty));
    FP8_TRY(check_scalar(fn, m1_scale, "m1_scale", false));
    FP8_TRY(check_scalar(fn, m1_scale_inv, "m1_scale_inv", false));
    FP8_TRY(check_scalar(fn, w_scale, "w_scale", false));
    FP8_TRY(check_scalar(fn, w_scale_inv, "w_scale_inv", false));
    FP8_TRY(check_scalar(fn, amax, "amax", false));
    int sms;
    FP8_TRY(current_device(&sms));
    const fp8k::AdamSpec a{grad, n, m1, m1_scale, m1_scale_inv, m2, w16, w_scale, w_scale_inv,
                           w_bf16, amax, hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay,
                           hp->bias_correction1, hp->bias_correction2, hp->margin};
    FP8_CUDA(fp8k::launch_adam_step(a, sms, static_cast<cudaStream_t>(stream)), fn);
    return FP8_OK;
}

fp8_status fp8_adam_init(const void *w, int64_t n, int32_t margin, uint8_t *m1, float *m1_scale,
                         float *m1_scale_inv, uint16_t *m2, uint16_t *w16, float *w_scale,
                         float *w_scale_inv, float *amax, void *stream) {
    const char *fn = "fp8_adam_init";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, n, "n", 0, "-"));
    if (margin < 0 || margin > 64) return fail(FP8_ERR_ARG, "%s: margin %d outside [0, 64]", fn, margin);
    const bool empty = n == 0;
    FP8_TRY(check_ptr(fn, w, "w", empty));
    FP8_TRY(check_ptr(fn, m1, "m1", empty));
    FP8_TRY(check_ptr(fn, m2, "m2", empty));
    FP8_TRY(check_ptr(fn, w16, "w16", empty));
    FP8_TRY(check_scalar(fn, m1_scale, "m1_scale", false));
    FP8_TRY(check_scalar(fn, m1_scale_inv, "m1_scale_inv", false));
    FP8_TRY(check_scalar(fn, w_scale, "w_scale", false));
    FP8_TRY(check_scalar(fn, w_scale_inv, "w_scale_inv", false));
    FP8_TRY(check_scalar(fn, amax, "amax", false));
    int sms;
    FP8_TRY(current_device(&sms));
    const fp8k::AdamInitSpec a{w, n, margin, m1, m1_scale, m1_scale_inv, m2, w16, w_scale,
                               w_scale_inv, amax};
    FP8_CUDA(fp8k::launch_adam_init(a, sms, static_cast<cudaStream_t>(stream)), fn);
    return FP8_OK;
}

fp8_status fp8_layernorm_quantize_transpose(const void *x, const void *gamma, const void *beta,
                                            int64_t rows, int64_t cols, float eps,
                                            const float *scale, int32_t fmt, uint8_t *out,
                                            uint8_t *out_t, float *amax, float *mean, float *rstd,
                                            void *stream) {
    const char *fn = "fp8_layernorm_quantize_transpose";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, rows, "rows", cols, "cols"));
    if (cols < 16) return fail(FP8_ERR_ARG, "%s: cols must be >= 16", fn);
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(FP8_ERR_ARG, "%s: bad format %d", fn, fmt);
    if (!(eps >= 0.0f)) return fail(FP8_ERR_ARG, "%s: eps must be >= 0", fn);
    const bool empty = rows == 0;
    if (!empty && out == nullptr && out_t == nullptr)
        return fail(FP8_ERR_ARG, "%s: out and out_t are both NULL", fn);
    FP8_TRY(check_ptr(fn, x, "x", empty));
    FP8_TRY(check_ptr(fn, gamma, "gamma", false));
    FP8_TRY(check_ptr(fn, beta, "beta", false));
    FP8_TRY(check_scalar(fn, scale, "scale", false));
    FP8_TRY(check_ptr(fn, out, "out", true));
    FP8_TRY(check_ptr(fn, out_t, "out_t", true));
    FP8_TRY(check_scalar(fn, amax, "amax", true));
    FP8_TRY(check_scalar(fn, mean, "mean", empty));
    FP8_TRY(check_scalar(fn, rstd, "rstd", empty));
    int sms;
    FP8_TRY(current_device(&sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (out != nullptr && fp8k::ln_cast_rows_fits(rows, cols)) {
        // one pass over x; the transposed copy from the codes just written
        FP8_CUDA(fp8k::launch_ln_cast_rows(x, gamma, beta, rows, cols, eps, scale, fmt, out, amax,
                                           true, mean, rstd, sms, st),
                 fn);
        if (out_t != nullptr)
            FP8_CUDA(fp8k::launch_transpose_u8(out, rows, cols, out_t, sms, st), fn);
        return FP8_OK;
    }
    FP8_CUDA(fp8k::launch_ln_stats(x, gamma, beta, rows, cols, eps, mean, rstd, nullptr, sms, st),
             fn);
    const fp8k::CastSpec c{x, rows, cols, const_cast<float *>(scale), nullptr, out, out_t, amax,
                           true, mean, rstd, gamma, beta};
    FP8_CUDA(fp8k::launch_cast_group(&c, 1, fmt, false, 0, sms, st), fn);
    return FP8_OK;
}

fp8_status fp8_layernorm_stats(const void *x, const void *gamma, const void *beta, int64_t rows,
                               int64_t cols, float eps, float *mean, float *rstd, float *amax,
                               void *stream) {
    const char *fn = "fp8_layernorm_stats";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_dims16(fn, rows, "rows", cols, "cols"));
    if (cols < 16) return fail(FP8_ERR_ARG, "%s: cols must be >= 16", fn);
    if (!(eps >= 0.0f)) return fail(FP8_ERR_ARG, "%s: eps must be >= 0", fn);
    const bool empty = rows == 0;
    FP8_TRY(check_ptr(fn, x, "x", empty));
    // gamma and beta enter only max |y|
    FP8_TRY(check_ptr(fn, gamma, "gamma", amax == nullptr));
    FP8_TRY(check_ptr(fn, beta, "beta", amax == nullptr));
    FP8_TRY(check_scalar(fn, amax, "amax", true));
    FP8_TRY(check_scalar(fn, mean, "mean", empty));
    FP8_TRY(check_scalar(fn, rstd, "rstd", empty));
    int sms;
    FP8_TRY(current_device(&sms));
    FP8_CUDA(fp8k::launch_ln_stats(x, gamma, beta, rows, cols, eps, mean, rstd, amax, sms,
                                   static_cast<cudaStream_t>(stream)),
             fn);
    return FP8_OK;
}

static fp8_status linear_fwd_impl(const char *fn, const void *X, const void *gamma,
                                  const void *beta, float eps, const void *W, int64_t M, int64_t N,
                                  int64_t K, const fp8_meta *meta, const fp8_recipe *recipe,
                                  uint8_t *X8, uint8_t *X8t, uint8_t *W8, uint8_t *W8t, void *Y,
                                  float *mean, float *rstd, void *stream);

fp8_status fp8_layernorm_linear_fwd(const void *X, const void *gamma, const void *beta, float eps,
                                    const void *W, int64_t M, int64_t N, int64_t K,
                                    const fp8_meta *meta, const fp8_recipe *recipe, uint8_t *X8,
                                    uint8_t *X8t, uint8_t *W8, uint8_t *W8t, void *Y, float *mean,
                                    float *rstd, void *stream) {
    const char *fn = "fp8_layernorm_linear_fwd";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_ptr(fn, gamma, "gamma", false));
    FP8_TRY(check_ptr(fn, beta, "beta", false));
    FP8_TRY(check_scalar(fn, mean, "mean", false));
    FP8_TRY(check_scalar(fn, rstd, "rstd", false));
    if (!(eps >= 0.0f)) return fail(FP8_ERR_ARG, "%s: eps must be >= 0", fn);
    return linear_fwd_impl(fn, X, gamma, beta, eps, W, M, N, K, meta, recipe, X8, X8t, W8, W8t, Y,
                           mean, rstd, stream);
}

fp8_status fp8_linear_fwd(const void *X, const void *W, int64_t M, int64_t N, int64_t K,
                          const fp8_meta *meta, const fp8_recipe *recipe, uint8_t *X8,
                          uint8_t *X8t, uint8_t *W8, uint8_t *W8t, void *Y, void *stream) {
    return linear_fwd_impl("fp8_linear_fwd", X, nullptr, nullptr, 0.0f, W, M, N, K, meta, recipe,
                           X8, X8t, W8, W8t, Y, nullptr, nullptr, stream);
}

static fp8_status linear_fwd_impl(const char *fn, const void *X, const void *gamma,
                                  const void *beta, float eps, const void *W, int64_t M, int64_t N,
                                  int64_t K, const fp8_meta *meta, const fp8_recipe *recipe,
                                  uint8_t *X8, uint8_t *X8t, uint8_t *W8, uint8_t *W8t, void *Y,
                                  float *mean, float *rstd, void *stream) {
    FP8_TRY(check_meta(fn, meta, recipe));
    FP8_TRY(check_dims16(fn, M, "M", N, "N"));
    FP8_TRY(check_dims16(fn, K, "K", 16, "-"));
    if (M < 16 || N < 16 || K < 16) return fail(FP8_ERR_ARG, "%s: M, N, K must be >= 16", fn);
    FP8_TRY(check_ptr(fn, X, "X", false));
    FP8_TRY(check_ptr(fn, W, "W", false));
    FP8_TRY(check_ptr(fn, X8, "X8", false));
    FP8_TRY(check_ptr(fn, X8t, "X8t", false));
    FP8_TRY(check_ptr(fn, W8, "W8", false));
    FP8_TRY(check_ptr(fn, W8t, "W8t", false));
    FP8_TRY(check_ptr(fn, Y, "Y", false));
    int sms;
    FP8_TRY(current_device(&sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *am = meta->amax;
    // amax of X, W and Y are max-combined into their slots, which the
    // previous fp8_amax_scale_update cleared (a fresh meta starts at 0).
    const bool cur = recipe->scaling == FP8_SCALING_CURRENT;
    const fp8k::CastSpec c[2] = {
        {X, M, K, meta->scale + FP8_SLOT_X, meta->scale_inv + FP8_SLOT_X, X8, X8t,
         am + FP8_SLOT_X, false, mean, rstd, gamma, beta},
        {W, N, K, meta->scale + FP8_SLOT_W, meta->scale_inv + FP8_SLOT_W, W8, W8t,
         am + FP8_SLOT_W, false, nullptr, nullptr, nullptr, nullptr}};
    if (mean != nullptr && !cur && fp8k::ln_cast_rows_fits(M, K)) {
        // LN(X) in one pass over X, X8t transposed from X8, then W on its own
        FP8_CUDA(fp8k::launch_ln_cast_rows(X, gamma, beta, M, K, eps, meta->scale + FP8_SLOT_X,
                                           FP8_E4M3, X8, am + FP8_SLOT_X, false, mean, rstd, sms,
                                           st),
                 fn);
        FP8_CUDA(fp8k::launch_transpose_u8(X8, M, K, X8t, sms, st), fn);
        FP8_CUDA(fp8k::launch_cast_group(c + 1, 1, FP8_E4M3, false, recipe->margin, sms, st), fn);
    } else {
        if (mean != nullptr)   // LayerNorm statistics (and, for current scaling, amax of LN(X))
            FP8_CUDA(fp8k::launch_ln_stats(X, gamma, beta, M, K, eps, mean, rstd,
                                           cur ? am + FP8_SLOT_X : nullptr, sms, st),
                     fn);
        // X (or LN(X)) and W (both E4M3) in one cast launch
        FP8_CUDA(fp8k::launch_cast_group(c, 2, FP8_E4M3, cur, recipe->margin, sms, st), fn);
    }
    return gemm_checked(fn, X8, FP8_E4M3, W8, FP8_E4M3, M, N, K, meta->scale_inv + FP8_SLOT_X,
                        meta->scale_inv + FP8_SLOT_W, Y, am + FP8_SLOT_Y, false, sms, st);
}

fp8_status fp8_linear_bwd(const void *dY, int64_t M, int64_t N, int64_t K, const fp8_meta *meta,
                          const fp8_recipe *recipe, const uint8_t *X8t, const uint8_t *W8t,
                          uint8_t *dY8, uint8_t *dY8t, void *dX, void *dW, void *stream) {
    const char *fn = "fp8_linear_bwd";
    const fp8k::CallRange range(fn);
    FP8_TRY(check_meta(fn, meta, recipe));
    FP8_TRY(check_dims16(fn, M, "M", N, "N"));
    FP8_TRY(check_dims16(fn, K, "K", 16, "-"));
    if (M < 16 || N < 16 || K < 16) return fail(FP8_ERR_ARG, "%s: M, N, K must be >= 16", fn);
    FP8_TRY(check_ptr(fn, dY, "dY", false));
    FP8_TRY(check_ptr(fn, X8t, "X8t", false));
    FP8_TRY(check_ptr(fn, W8t, "W8t", false));
    FP8_TRY(check_ptr(fn, dY8, "dY8", false));
    FP8_TRY(check_ptr(fn, dY8t, "dY8t", false));
    FP8_TRY(check_ptr(fn, dX, "dX", false));
    FP8_TRY(check_ptr(fn, dW, "dW", false));
    int sms;
    FP8_TRY(current_device(&sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *am = meta->amax;
    const int32_t fg = recipe->hybrid ? FP8_E5M2 : FP8_E4M3;
    // amax of dY and dX are max-combined into their slots (see fp8_linear_fwd)
    if (recipe->scaling == FP8_SCALING_CURRENT)
        FP8_CUDA(fp8k::launch_quantize_transpose_current(
                     dY, M, N, fg, recipe->margin, dY8, dY8t, am + FP8_SLOT_DY,
                     meta->scale + FP8_SLOT_DY, meta->scale_inv + FP8_SLOT_DY, sms, st),
                 fn);
    else
        FP8_CUDA(fp8k::launch_quantize_transpose(dY, M, N, meta->scale + FP8_SLOT_DY, fg, dY8,
                                                 dY8t, am + FP8_SLOT_DY, false, sms, st),
                 fn);
    // One launch for both GEMMs, dgrad's (longer-K) tiles first:
    //   dgrad: dX[M][K] = dY8[M][N] . W8t[K][N]^T
    //   wgrad: dW[N][K] = dY8t[N][M] . X8t[K][M]^T
    const fp8k::GemmSpec g[2] = {
        {dY8, fg, W8t, FP8_E4M3, M, K, N, meta->scale_inv + FP8_SLOT_DY,
         meta->scale_inv + FP8_SLOT_W, dX, am + FP8_SLOT_DX, false},
        {dY8t, fg, X8t, FP8_E4M3, N, K, M, meta->scale_inv + FP8_SLOT_DY,
         meta->scale_inv + FP8_SLOT_X, dW, nullptr, false}};
    const char *what = nullptr;
    cudaError_t e = fp8k::launch_gemm_group(g, 2, sms, st, &what);
    if (e != cudaSuccess)
        return what ? fail(FP8_ERR_CUDA, "%s: %s", fn, what) : cuda_fail(e, fn);
    return FP8_OK;
}

}  // extern "C"
