// kernels.h -- host-side launchers of the sm_103a kernels (internal to the
// library; the public C ABI is include/fp8amax.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include <nvtx3/nvToolsExt.h>

namespace fp8k {

// An NVTX range around each C-ABI call (a pointer check when no profiler is
// attached), so a profile can attribute kernels to the calls that launched
// them.
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

// Tiled 2-D TMA descriptor of a row-major [outer][inner] tensor of 1- or
// 2-byte elements with a box of box_outer x box_inner elements, optionally
// with 128-byte swizzling (tmap.cu).  False if cuTensorMapEncodeTiled rejects it.
bool encode_tmap_2d(CUtensorMap *map, const void *base, bool two_byte, int64_t inner,
                    int64_t outer, uint32_t box_inner, uint32_t box_outer, bool swizzle128);

// amax of n BF16 values into *amax (zeroed first).
cudaError_t launch_amax(const void *x, int64_t n, float *amax, int sm_count, cudaStream_t st);
cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t st);
cudaError_t launch_quantize_f32(const float *x, int64_t n, const float *scale, int fmt,
                                uint8_t *out, float *amax, int sm_count, cudaStream_t st);

// Fused scaled cast + transposed copy + amax.  fmt: 0 = E4M3, 1 = E5M2.
// With zero_amax the amax word is cleared first; otherwise the tensor's amax
// is max-combined into it.  Returns cudaErrorInvalidValue when the input's
// TMA descriptor cannot be built.
cudaError_t launch_quantize_transpose(const void *x, int64_t rows, int64_t cols,
                                      const float *scale, int fmt, uint8_t *out, uint8_t *out_t,
                                      float *amax, bool zero_amax, int sm_count, cudaStream_t st);

// One tensor of a grouped cast: x [rows][cols] BF16 -> out / out_t (FP8),
// scale (read; in just-in-time mode replaced, with scale_inv, from the amax),
// amax (max-combined; cleared first when zero_amax; always overwritten in
// just-in-time mode).
struct CastSpec {
    const void *x;
    int64_t rows, cols;
    float *scale;
    float *scale_inv;
    uint8_t *out, *out_t;
    float *amax;
    bool zero_amax;
    // LayerNorm in front of the cast (all null for a plain cast): per-row
    // mean / rstd from launch_ln_stats, per-column gamma / beta (BF16).
    const float *ln_mean, *ln_rstd;
    const void *ln_gamma, *ln_beta;
};

// LayerNorm statistics of x [rows][cols] (BF16): fp32 mean and rstd per row;
// with amax, also max |y| of the LayerNorm output (cleared first).
cudaError_t launch_ln_stats(const void *x, const void *gamma, const void *beta, int64_t rows,
                            int64_t cols, float eps, float *mean, float *rstd, float *amax,
                            int sm_count, cudaStream_t st);

// LayerNorm statistics, normalisation and the row-major cast in one pass over
// x (delayed scaling: the scale is given; no transposed copy).  Only where
// ln_cast_rows_fits(rows, cols): cols a multiple of 16 of at most 4096.  max
// |y| is max-combined into amax (optional), cleared first when zero_amax.
bool ln_cast_rows_fits(int64_t rows, int64_t cols);
cudaError_t launch_ln_cast_rows(const void *x, const void *gamma, const void *beta, int64_t rows,
                                int64_t cols, float eps, const float *scale, int fmt,
                                uint8_t *out, float *amax, bool zero_amax, float *mean,
                                float *rstd, int sm_count, cudaStream_t st);

// out_t[c][r] = in[r][c] for a [rows][cols] byte array (FP8 codes); rows
// and cols multiples of 16.
cudaError_t launch_transpose_u8(const uint8_t *in, int64_t rows, int64_t cols, uint8_t *out_t,
                                int sm_count, cudaStream_t st);

// Up to two tensors of one format in one persistent cast launch (tiles form
// one list).  current = just-in-time scaling (an amax pass per tensor first).
cudaError_t launch_cast_group(const CastSpec *specs, int n, int fmt, bool current, int margin,
                              int sm_count, cudaStream_t st);

// Just-in-time scaling: amax of x into *amax (overwritten), then the cast
// with scale = recipe formula of that amax (history of one), written back to
// *scale / *scale_inv (both kept when the amax is 0 or not finite).
cudaError_t launch_quantize_transpose_current(const void *x, int64_t rows, int64_t cols, int fmt,
                                              int margin, uint8_t *out, uint8_t *out_t,
                                              float *amax, float *scale, float *scale_inv,
                                              int sm_count, cudaStream_t st);

// History shift + scale / scale_inv update of num_tensors states; with
// clear_amax the amax words are set to 0 once pushed into the history.
cudaError_t launch_scale_update(float *history, float *amax, float *scale, float *scale_inv,
                                int num_tensors, int L, uint32_t format_mask, int margin,
                                bool clear_amax, cudaStream_t st);

// One GEMM of a grouped launch: D[M][N] = A[M][K] . B[N][K]^T (FP8 codes of
// formats fa / fb), dequantised by a_scale_inv * b_scale_inv into BF16, with
// the output amax max-combined into *d_amax (cleared first when zero_amax).
struct GemmSpec {
    const uint8_t *A;
    int fa;
    const uint8_t *B;
    int fb;
    int64_t M, N, K;
    const float *a_scale_inv;
    const float *b_scale_inv;
    void *D;
    float *d_amax;
    bool zero_amax;
};

// Up to two independent GEMMs in one persistent launch; their tiles form one
// list (the first spec's tiles first), so one GEMM's last partial wave is
// filled with the other's tiles.
cudaError_t launch_gemm_group(const GemmSpec *specs, int n, int sm_count, cudaStream_t st,
                              const char **what);

// FP8 "TN" GEMM on tcgen05 with the dequant + amax epilogue.  With
// zero_amax the amax word is cleared first.  Returns cudaErrorInvalidValue
// (with *what set) when a TMA descriptor cannot be built.
cudaError_t launch_gemm_tn(const uint8_t *A, int fa, const uint8_t *B, int fb, int64_t M,
                           int64_t N, int64_t K, const float *a_scale_inv,
                           const float *b_scale_inv, void *D, float *d_amax, bool zero_amax,
                           int sm_count, cudaStream_t st, const char **what);

// One decoupled-precision Adam step (optim.cu): first moment E4M3 + scale,
// second moment FP16, master weights FP16 + scale; writes the model's BF16
// weights and amax[2] (new first moment, new weights), then the new scales.
struct AdamSpec {
    const void *grad;
    int64_t n;
    uint8_t *m1;
    float *m1_scale, *m1_scale_inv;
    uint16_t *m2, *w16;
    float *w_scale, *w_scale_inv;
    void *w_bf16;
    float *amax;
    float lr, b1, b2, eps, wd, bc1, bc2;
    int margin;
};
cudaError_t launch_adam_step(const AdamSpec &s, int sm_count, cudaStream_t st);

// Initial decoupled-precision Adam state of a BF16 weight tensor: zero
// moments, FP16 master weights under the just-in-time scale of w (fmax
// 65504), the four scales, and amax = {0, amax(w)}.
struct AdamInitSpec {
    const void *w;
    int64_t n;
    int margin;
    uint8_t *m1;
    float *m1_scale, *m1_scale_inv;
    uint16_t *m2, *w16;
    float *w_scale, *w_scale_inv;
    float *amax;
};
cudaError_t launch_adam_init(const AdamInitSpec &s, int sm_count, cudaStream_t st);

// Decode-and-sum of nranks FP8 parts [nranks][n] sharing one scale (optim.cu).
cudaError_t launch_dequant_sum(const uint8_t *parts, int nranks, int64_t n, int fmt,
                               const float *scale, void *out, int sm_count, cudaStream_t st);

// Diagnostic: while acc is not null, the first CTA of every GEMM launch adds
// its SM clock cycles to acc[0] and its nanoseconds to acc[1] (gemm.cu).
void set_clock_probe(unsigned long long *acc);

// Set the message fp8_last_error() returns on this host thread.
void set_last_error(const char *msg);

// Read and clear the cast kernels' device error flag (cast.cu).
cudaError_t read_and_clear_cast_error_flag(unsigned *flags);

// Read and clear the FP8 sum kernel's device error flag (optim.cu).
cudaError_t read_and_clear_sum_error_flag(unsigned *flags);

// Read and clear the device error flag the kernels set when a bounded wait
// gives up (synchronizes the device flag's stream).
cudaError_t read_and_clear_error_flag(unsigned *flags, cudaStream_t st);

}  // namespace fp8k
