/*
 * fp8amax.h -- C ABI of the GB300 (sm_103a) FP8 delayed-scaling linear layer.
 *
 * The operations follow three web pages on FP8 mixed-precision training:
 *  - "NVIDIA Transformer Engine and FP8 mixed precision: implementation guide"
 *    (ai-tool-zukan.com): section "What are Transformer Engine and FP8 mixed
 *    precision" (E4M3 = 4 exponent / 3 mantissa bits for the forward pass,
 *    E5M2 = 5 / 2 for the backward pass; dynamic scaling watches each
 *    tensor's range and adjusts its scale factor) and section "Dynamic
 *    scaling and the FP8 recipe" (DelayedScaling with margin, fp8_format,
 *    amax_history_len; Format.HYBRID = E4M3 forward / E5M2 backward; the
 *    amax history is part of the model state).
 *  - "FP8 quantization with NVIDIA TensorRT" (ai.warp-studio.com): explicit
 *    quantize / dequantize (Q/DQ) nodes and the Absolute-Max statistic.
 *  - "Mixed-precision training" wiki note (notes.yuuk.io): "Definition" table
 *    (E4M3 max 448, E5M2 max 57,344) and the bullets "extension to FP8"
 *    (only the GEMMs run in FP8) and "per-tensor scaling is the key"
 *    (delayed or just-in-time per-tensor scaling).
 *
 * Numerics (identical on every call):
 *  - amax(x) = max |x_i| over the tensor, NaN entries skipped, exact.
 *  - cast: v = fl32(x * scale) (one binary32 multiply), then round to the
 *    nearest FP8 value, ties to the even code; |v| above the largest finite
 *    value and +-inf saturate to +-448 (E4M3) / +-57344 (E5M2); NaN stays NaN;
 *    the sign of zero is kept.  E4M3 is the variant with no infinities whose
 *    only NaN code is S.1111.111 (largest finite 448); E5M2 is IEEE-style.
 *  - scale update: history <- [amax, history[0..L-2]]; m = max(history); if
 *    0 < m < inf then scale = fl32(fl32(fmax / m) * 2^-margin) (+inf clamped
 *    to FLT_MAX) and scale_inv = fl32(1 / scale); otherwise both unchanged.
 *  - GEMM: D[i][j] = bf16_rne(fl32(acc[i][j] * fl32(a_scale_inv * b_scale_inv)))
 *    with acc = sum_k A[i][k] * B[j][k] accumulated in fp32 by the tensor
 *    cores, and d_amax = max |D| over the emitted BF16 values.
 *
 * Conventions for every entry point:
 *  - Pointers named as DEVICE pointers must be device (or managed) memory of
 *    the current device; the caller allocates and owns every buffer.  The
 *    library allocates no device memory, never synchronizes the stream (except
 *    fp8_sync_status), and keeps no state beyond cached device properties,
 *    one device-side error flag, the diagnostic clock-probe pointer
 *    (fp8_set_clock_probe) and the fixed work array that
 *    fp8_linear_bwd_noalloc uses (described there).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  All work is enqueued on it, in order; scales are read on the
 *    device, so a training step needs no host round trip.
 *  - Tensors are dense row-major.  Row and column counts must be multiples of
 *    16 and tensor pointers 16-byte aligned (else FP8_ERR_ALIGN), so that
 *    every row of every FP8 and BF16 tensor starts on a 16-byte boundary.
 *    Pointers to fp32 scalars and to the fp8_meta buffers need 4-byte
 *    alignment only.
 *  - Arguments are checked on the host before anything is enqueued; on any
 *    status other than FP8_OK nothing was enqueued, and fp8_last_error()
 *    gives a message (thread-local).  Errors reported by the CUDA runtime at
 *    launch give FP8_ERR_CUDA.
 *  - Bounded waits: every spin-wait in a kernel gives up after about two
 *    seconds, sets a device error flag and returns; fp8_sync_status() reports
 *    it as FP8_ERR_TIMEOUT.
 */
#ifndef FP8AMAX_H
#define FP8AMAX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8AMAX_ABI_VERSION 4

typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_format;

typedef enum {
    FP8_OK = 0,
    FP8_ERR_ARG = 1,         /* bad size, NULL pointer, bad format / margin / history length */
    FP8_ERR_ALIGN = 2,       /* size not a multiple of 16 or a pointer misaligned */
    FP8_ERR_CUDA = 3,        /* the CUDA runtime reported an error */
    FP8_ERR_TIMEOUT = 4,     /* a kernel's bounded wait ran out (see fp8_sync_status) */
    FP8_ERR_UNSUPPORTED = 5  /* the current device is not an sm_103 GPU */
} fp8_status;

/* The five tensors of one linear layer whose scaling state is tracked. */
enum { FP8_SLOT_X = 0, FP8_SLOT_W = 1, FP8_SLOT_Y = 2, FP8_SLOT_DY = 3, FP8_SLOT_DX = 4,
       FP8_NUM_SLOTS = 5 };

/* Scaling state of one linear layer (the DelayedScaling state the
 * implementation guide says is saved with the model).  All DEVICE pointers,
 * caller-owned, fp32:
 *   history   [5][history_len]  row = slot; history[slot*L + 0] is the newest
 *   amax      [5]               this step's amax of each slot
 *   scale     [5]               multiplier applied before the FP8 cast (init 1)
 *   scale_inv [5]               1 / scale, applied in the GEMM epilogue (init 1)
 * A fresh state is history = 0, amax = 0, scale = scale_inv = 1. */
typedef struct {
    float *history;
    float *amax;
    float *scale;
    float *scale_inv;
    int32_t history_len;
} fp8_meta;

/* DelayedScaling recipe (implementation guide, "Dynamic scaling and the FP8
 * recipe"): margin (>= 0, default 0; larger = fewer overflows, more
 * underflow), amax_history_len (default 1024) and the format choice.
 * hybrid = 1: E4M3 for X, W, Y and E5M2 for dY, dX (Format.HYBRID);
 * hybrid = 0: E4M3 for all five.  The scale is updated every step.
 * scaling selects between the two per-tensor scalings the wiki note names
 * ("per-tensor scaling is the key": delayed or just-in-time):
 *   FP8_SCALING_DELAYED  the casts use the scales the previous step's
 *                        fp8_amax_scale_update derived from the history;
 *   FP8_SCALING_CURRENT  X, W and dY are cast with a scale derived from
 *                        their own amax in the same call (the formula with
 *                        a history of one), written to meta->scale /
 *                        scale_inv; the history update still runs. */
enum { FP8_SCALING_DELAYED = 0, FP8_SCALING_CURRENT = 1 };
typedef struct {
    int32_t margin;
    int32_t history_len;
    int32_t hybrid;
    int32_t scaling;
} fp8_recipe;

/* ABI version of the loaded library (FP8AMAX_ABI_VERSION). */
int32_t fp8_abi_version(void);

/* Message of the last non-OK status returned on this host thread. */
const char *fp8_last_error(void);

/* Synchronize `stream`, then report (and clear) the device error flag:
 * FP8_ERR_TIMEOUT if a kernel gave up a bounded wait since the last call,
 * FP8_ERR_CUDA if the stream reports an error, else FP8_OK. */
fp8_status fp8_sync_status(void *stream);

/* Diagnostic, not part of the method: launches one warp that waits with the
 * library's bounded wait on a barrier nothing ever signals, so the wait runs
 * out after limit_ns (1 .. 5e9) and the kernel records it in the device
 * error flag and returns -- the path every kernel takes when a wait runs out.
 * The next fp8_sync_status on the stream then returns FP8_ERR_TIMEOUT (and
 * clears the flag); the context stays usable. */
fp8_status fp8_selftest_wait_timeout(int64_t limit_ns, void *stream);

/* Diagnostic, not part of the method: a clock probe for measuring the SM
 * clock the GEMMs actually run at.  While acc is not NULL, the first CTA of
 * every GEMM launch (fp8_gemm_tn, fp8_gemm_tn_grouped and the GEMMs inside
 * the layer calls) adds the SM clock cycles (%clock64) and the nanoseconds
 * (%globaltimer) between its start and its end to acc[0] and acc[1] (atomic
 * adds); acc[0] / acc[1] is then the average SM clock during those launches
 * in GHz.  The kernels persist over all tiles, so that CTA lives as long as
 * the launch.  acc: DEVICE, 2 uint64, 8-byte aligned, caller-owned and
 * zeroed by the caller; NULL (the default) turns the probe off.  The
 * setting is process-wide and is read when a launch is enqueued (a CUDA
 * graph keeps the value it was captured with). */
fp8_status fp8_set_clock_probe(uint64_t *acc);

/* amax of a BF16 tensor (the implementation guide's range monitoring; the
 * TensorRT page's Absolute-Max statistic).
 *   x     DEVICE, n BF16 values (n >= 0, multiple of 16; n == 0 gives 0)
 *   amax  DEVICE, 1 float, overwritten with max |x_i| (NaN skipped). */
fp8_status fp8_amax(const void *x, int64_t n, float *amax, void *stream);

/* Fused scaled cast BF16 -> FP8 with transposed copy and amax (the Q node of
 * the TensorRT page; formats of the implementation guide / wiki table).
 *   x      DEVICE, [rows][cols] BF16
 *   scale  DEVICE, 1 float, read on the device
 *   fmt    FP8_E4M3 or FP8_E5M2
 *   out    DEVICE, [rows][cols] FP8 codes, or NULL
 *   out_t  DEVICE, [cols][rows] FP8 codes (the transpose of out), or NULL
 *   amax   DEVICE, 1 float overwritten with amax(x), or NULL
 * rows, cols >= 0 and multiples of 16.  At least one of out / out_t unless
 * the tensor is empty (then only the amax, 0, is written). */
fp8_status fp8_quantize_transpose(const void *x, int64_t rows, int64_t cols, const float *scale,
                                  int32_t fmt, uint8_t *out, uint8_t *out_t, float *amax,
                                  void *stream);

/* Scaled cast of an fp32 tensor to FP8 (the Q node of the TensorRT page on
 * fp32 values, such as the fp32 quantities that FP8-LM stores in FP8, wiki
 * note "extension to FP8"): q_i = satRNE_fmt(fl32(x_i * scale)) in element
 * order, with the same rounding, saturation and NaN rules as the BF16 cast.
 *   x      DEVICE, n fp32 values, 16-byte aligned (n >= 0, multiple of 16)
 *   scale  DEVICE, 1 float, read on the device
 *   fmt    FP8_E4M3 or FP8_E5M2
 *   out    DEVICE, n FP8 codes, 16-byte aligned (may be NULL when n == 0)
 *   amax   DEVICE, 1 float overwritten with max |x_i| (NaN skipped), or NULL */
fp8_status fp8_quantize_f32(const float *x, int64_t n, const float *scale, int32_t fmt,
                            uint8_t *out, float *amax, void *stream);

/* Just-in-time (current) scaling of one tensor (wiki note, "per-tensor
 * scaling is the key": the scale comes from the tensor itself): amax(x),
 * then scale = the recipe formula applied to that amax alone, then the fused
 * cast with that scale.  Two kernels, in stream order.
 *   x, rows, cols, fmt, out, out_t  as fp8_quantize_transpose
 *   margin     0 <= margin <= 64
 *   amax       DEVICE, 1 float, overwritten with amax(x)
 *   scale, scale_inv  DEVICE, 1 float each: replaced by the new scale and
 *              its inverse when 0 < amax < inf, left as they are otherwise
 *              (the cast then uses the given scale). */
fp8_status fp8_quantize_transpose_current(const void *x, int64_t rows, int64_t cols, int32_t fmt,
                                          int32_t margin, uint8_t *out, uint8_t *out_t,
                                          float *amax, float *scale, float *scale_inv,
                                          void *stream);

/* Delayed-scaling update of `num_tensors` independent scaling states (the
 * recipe section's margin and amax_history_len, with the scale formula in
 * the header comment).  All DEVICE:
 *   history    [num_tensors][history_len], shifted in place, [t][0] newest
 *   amax       [num_tensors], the value pushed into each history (read only)
 *   scale, scale_inv [num_tensors], updated in place
 * format_mask: bit t set = tensor t is E5M2 (fmax 57344), clear = E4M3 (448).
 * 1 <= num_tensors <= 32, 1 <= history_len <= 8192, 0 <= margin <= 64. */
fp8_status fp8_scale_update(float *history, const float *amax, float *scale, float *scale_inv,
                            int32_t num_tensors, int32_t history_len, uint32_t format_mask,
                            int32_t margin, void *stream);

/* The recipe's update of all five slots of one layer, run once per step
 * after fp8_linear_fwd and fp8_linear_bwd: fp8_scale_update over meta with
 * the recipe's formats (HYBRID: slots dY and dX are E5M2), after which the
 * five amax slots are cleared to 0 for the next step.
 * meta->history_len must equal recipe->history_len. */
fp8_status fp8_amax_scale_update(const fp8_meta *meta, const fp8_recipe *recipe, void *stream);

/* FP8 GEMM with both operands contiguous along K ("TN"), fp32 accumulation
 * in TMEM on the tcgen05 tensor cores, and the dequant epilogue (wiki note,
 * "extension to FP8"; the DQ node of the TensorRT page).
 *   A  DEVICE [M][K] FP8 codes of format fa;  B  DEVICE [N][K] of format fb
 *   a_scale_inv, b_scale_inv  DEVICE, 1 float each
 *   D  DEVICE [M][N] BF16 output
 *   d_amax  DEVICE, 1 float overwritten with max |D|, or NULL
 * M, N, K >= 16 and multiples of 16. */
fp8_status fp8_gemm_tn(const uint8_t *A, int32_t fa, const uint8_t *B, int32_t fb, int64_t M,
                       int64_t N, int64_t K, const float *a_scale_inv, const float *b_scale_inv,
                       void *D, float *d_amax, void *stream);

/* One GEMM of fp8_gemm_tn_grouped; fields as the arguments of fp8_gemm_tn. */
typedef struct {
    const uint8_t *A;
    int32_t fa;
    const uint8_t *B;
    int32_t fb;
    int64_t M, N, K;
    const float *a_scale_inv;
    const float *b_scale_inv;
    void *D;
    float *d_amax;
} fp8_gemm_desc;

/* One or two independent fp8_gemm_tn problems in a single persistent launch
 * (helper; the backward pass runs dgrad and wgrad this way): the tiles of
 * both form one list, so one GEMM's last partial wave is filled with the
 * other's tiles.  n is 1 or 2; each problem is checked as by fp8_gemm_tn,
 * and each d_amax (when not NULL) is overwritten with its own output amax. */
fp8_status fp8_gemm_tn_grouped(const fp8_gemm_desc *descs, int32_t n, void *stream);

/* One tensor of fp8_quantize_transpose_grouped; fields as the arguments of
 * fp8_quantize_transpose. */
typedef struct {
    const void *x;
    int64_t rows, cols;
    const float *scale;
    uint8_t *out;
    uint8_t *out_t;
    float *amax;
} fp8_cast_desc;

/* One or two fp8_quantize_transpose casts of the same format in a single
 * persistent launch (helper; the forward pass casts X and W this way).  Each
 * tensor is checked as by fp8_quantize_transpose; each amax (when not NULL)
 * is overwritten with its own tensor's amax. */
fp8_status fp8_quantize_transpose_grouped(const fp8_cast_desc *descs, int32_t n, int32_t fmt,
                                          void *stream);

/* LayerNorm fused with the scaled cast (te.LayerNorm in front of an FP8
 * linear; implementation guide, "Basic structure of FP8 training code"):
 *   mean[r] = sum_c x[r][c] / C,  var[r] = sum_c (x[r][c] - mean[r])^2 / C,
 *   rstd[r] = 1 / sqrt(var[r] + eps),
 *   y[r][c] = ((x[r][c] - mean[r]) * rstd[r]) * gamma[c] + beta[c]   (fp32),
 * then the cast of y exactly as fp8_quantize_transpose casts x (y is never
 * written out in BF16).  Rows of at most 4096 columns with out given: one
 * kernel computes the statistics and the row-major codes from one read of x,
 * and out_t (if given) is the byte transpose of those codes.  Otherwise two
 * kernels: row statistics, then LayerNorm + cast.  Both compute the same
 * statistics bit for bit.
 *   x      DEVICE [rows][cols] BF16;  gamma, beta  DEVICE [cols] BF16
 *   eps    >= 0;  scale  DEVICE, 1 float;  fmt, out, out_t as fp8_quantize_transpose
 *   amax   DEVICE, 1 float overwritten with max |y| (fp32 y, NaN skipped), or NULL
 *   mean, rstd  DEVICE [rows] fp32 outputs (kept for the LayerNorm backward)
 * rows, cols multiples of 16, cols >= 16.  Sums run in fp32 in a different
 * order from a sequential sum, so y matches an exact evaluation to about
 * 1e-6 relative, not bit for bit. */
fp8_status fp8_layernorm_quantize_transpose(const void *x, const void *gamma, const void *beta,
                                            int64_t rows, int64_t cols, float eps,
                                            const float *scale, int32_t fmt, uint8_t *out,
                                            uint8_t *out_t, float *amax, float *mean, float *rstd,
                                            void *stream);

/* LayerNorm row statistics alone (te.LayerNormLinear's LayerNorm; the same
 * page and section as fp8_layernorm_quantize_transpose): mean[r] and rstd[r]
 * exactly as that call computes them (bit for bit), which the LayerNorm
 * backward keeps, and, if amax is given, max |y| over y = LN(x) as defined
 * there: the amax that just-in-time scaling needs before any code is written.
 *   x      DEVICE [rows][cols] BF16
 *   gamma, beta  DEVICE [cols] BF16, read only when amax is given (else may be NULL)
 *   eps    >= 0
 *   mean, rstd  DEVICE [rows] fp32 outputs
 *   amax   DEVICE, 1 float overwritten with max |y| (fp32 y, NaN skipped; 0 for
 *          no rows), or NULL
 * rows, cols multiples of 16, cols >= 16; x, gamma, beta 16-byte aligned.
 * Rows of at most 4096 columns are held in registers (one HBM read of x);
 * wider rows are staged in shared memory or, past 8192 columns, read twice. */
fp8_status fp8_layernorm_stats(const void *x, const void *gamma, const void *beta, int64_t rows,
                               int64_t cols, float eps, float *mean, float *rstd, float *amax,
                               void *stream);

/* Forward of LayerNorm + FP8 linear (te.LayerNormLinear): Y = LN(X) W^T with
 * LN(X) cast to E4M3 as fp8_layernorm_quantize_transpose casts it (its amax
 * is slot X's; under delayed scaling X8t is the byte transpose of X8), W cast
 * as in fp8_linear_fwd, then fprop.  Arguments as fp8_linear_fwd plus gamma,
 * beta [K] (BF16), eps, and mean, rstd [M] (fp32 outputs).  X8 / X8t hold the
 * FP8 LayerNorm output, so fp8_linear_bwd follows unchanged. */
fp8_status fp8_layernorm_linear_fwd(const void *X, const void *gamma, const void *beta, float eps,
                                    const void *W, int64_t M, int64_t N, int64_t K,
                                    const fp8_meta *meta, const fp8_recipe *recipe, uint8_t *X8,
                                    uint8_t *X8t, uint8_t *W8, uint8_t *W8t, void *Y, float *mean,
                                    float *rstd, void *stream);

/* Forward of the FP8 linear layer Y = X W^T (te.Linear under fp8_autocast,
 * implementation guide "Basic structure of FP8 training code" and the
 * recipe section).  Uses this step's (delayed) scales of X and W, or under
 * FP8_SCALING_CURRENT derives them from X's and W's own amax first.
 *   X   DEVICE [M][K] BF16 input;   W  DEVICE [N][K] BF16 weight
 *   X8, X8t  DEVICE [M][K] and [K][M] FP8 (E4M3), written; X8t is kept for wgrad
 *   W8, W8t  DEVICE [N][K] and [K][N] FP8 (E4M3), written; W8t is kept for dgrad
 *   Y   DEVICE [M][N] BF16 output
 * Max-combines the amax of X, W and Y into meta->amax[X], [W], [Y]: the
 * slots hold the running max since the last fp8_amax_scale_update, which
 * clears them (a fresh meta has them at 0), so several forward calls before
 * one update (micro-batches) record the max over all of them.  Under
 * FP8_SCALING_CURRENT the X and W slots are overwritten with this call's
 * amax instead. */
fp8_status fp8_linear_fwd(const void *X, const void *W, int64_t M, int64_t N, int64_t K,
                          const fp8_meta *meta, const fp8_recipe *recipe, uint8_t *X8,
                          uint8_t *X8t, uint8_t *W8, uint8_t *W8t, void *Y, void *stream);

/* Backward of the FP8 linear layer: dX = dY W (dgrad), dW = dY^T X (wgrad),
 * with dY cast to E5M2 under HYBRID (E4M3 otherwise); under
 * FP8_SCALING_CURRENT dY's scale is derived from its own amax first.
 *   dY  DEVICE [M][N] BF16 output gradient
 *   X8t, W8t  DEVICE, the transposed copies written by fp8_linear_fwd
 *   dY8, dY8t DEVICE [M][N] and [N][M] FP8 work buffers, written
 *   dX  DEVICE [M][K] BF16;  dW  DEVICE [N][K] BF16
 * Max-combines the amax of dY and dX into meta->amax[dY], [dX] (as
 * fp8_linear_fwd does for its slots; under FP8_SCALING_CURRENT the dY slot is
 * overwritten with this call's amax). */
fp8_status fp8_linear_bwd(const void *dY, int64_t M, int64_t N, int64_t K, const fp8_meta *meta,
                          const fp8_recipe *recipe, const uint8_t *X8t, const uint8_t *W8t,
                          uint8_t *dY8, uint8_t *dY8t, void *dX, void *dW, void *stream);

/* Hyper-parameters of one Adam step (AdamW's decoupled weight decay).  The
 * bias corrections 1 - beta1^t and 1 - beta2^t are computed by the caller
 * for step t (>= 1) and passed as binary32. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    float bias_correction1, bias_correction2;
    int32_t margin;   /* for the state scales, 0..64 */
} fp8_adam_hyper;

/* One Adam step on optimizer states of decoupled precision (wiki note,
 * bullet "precision decoupling": first moment FP8, second moment FP16,
 * master weights FP16 with tensor scaling: 5 bytes of state per parameter;
 * the note's 6 also counts an FP8 gradient, which this path keeps BF16).  In
 * binary32, one rounding per operation, for every element (Adam's textbook
 * bias correction m / (1 - b1^t), v / (1 - b2^t); AdamW's decoupled decay):
 *   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g);
 *   u = (m / bc1) / (sqrt(v / bc2) + eps);  w = w - lr*(u + wd*w)
 * with m = E4M3 code * m1_scale_inv and w = FP16 code * w_scale_inv.  The new
 * states take just-in-time per-tensor scales: scale = (fmax / amax) /
 * 2^margin of the new values (fmax 448 for m, 65504 for w), kept when that
 * amax is 0 or not finite.  FP16 encodes round to nearest even and saturate
 * at +-65504.  Four kernels, in stream order.
 *   grad        DEVICE [n] BF16 gradient
 *   m1          DEVICE [n] E4M3 codes, updated in place
 *   m1_scale, m1_scale_inv   DEVICE 1 float each, updated
 *   m2          DEVICE [n] FP16 second moment, updated in place
 *   w16         DEVICE [n] FP16 master-weight codes, updated in place
 *   w_scale, w_scale_inv     DEVICE 1 float each, updated
 *   w_bf16      DEVICE [n] BF16 output: the weights for the next forward
 *   amax        DEVICE [2] output: amax of the new m and w (fp32)
 * n >= 0, a multiple of 16; arrays 16-byte aligned. */
fp8_status fp8_adam_step(const void *grad, int64_t n, uint8_t *m1, float *m1_scale,
                         float *m1_scale_inv, uint16_t *m2, uint16_t *w16, float *w_scale,
                         float *w_scale_inv, void *w_bf16, float *amax, const fp8_adam_hyper *hp,
                         void *stream);

/* Initial state for fp8_adam_step of one BF16 weight tensor (same bullet):
 * zero moments with first-moment scale and inverse 1, and the master weights
 * in FP16 under the just-in-time scale of w itself -- the recipe formula on
 * amax(w) alone with FP16's largest finite value:
 *   s_w = fl32(fl32(65504 / amax(w)) * 2^-margin)  (FLT_MAX if it overflows;
 *         1 when amax(w) is 0 or not finite),  w_scale_inv = fl32(1 / s_w),
 *   w16[i] = FP16 code of fl32(w[i] * s_w), nearest even, saturating.
 *   w       DEVICE [n] BF16 weights (read)
 *   margin  0..64
 *   m1 [n] E4M3 codes, m2 [n] FP16, w16 [n] FP16: DEVICE outputs
 *   m1_scale, m1_scale_inv, w_scale, w_scale_inv: DEVICE, 1 float each, written
 *   amax    DEVICE [2] output: {0, amax(w)}
 * n >= 0, a multiple of 16; arrays 16-byte aligned.  Three kernels (after a
 * one-word memset), in stream order. */
fp8_status fp8_adam_init(const void *w, int64_t n, int32_t margin, uint8_t *m1, float *m1_scale,
                         float *m1_scale_inv, uint16_t *m2, uint16_t *w16, float *w_scale,
                         float *w_scale_inv, float *amax, void *stream);

/* The summing half of an FP8 all-reduce with one shared scale (wiki note,
 * bullet "per-tensor scaling is the key": every rank casts with the one
 * scalar s'_g = min(s'_1, ..., s'_N), so the exchanged FP8 codes of all ranks
 * can be summed directly).  After this rank's shard of every rank's codes
 * has been exchanged:
 *   out[i] = bf16_rne( sum_r dec(parts[r][i]) * fl32(1 / scale) )
 * with the sum and the product exact, rounded once to BF16 (nearest, ties to
 * even; overflow to +-inf; gradual underflow, a nonzero result that rounds
 * to zero keeps its sign; an exact zero is +0).  Special codes follow IEEE
 * arithmetic: a NaN code, or +inf and -inf together, give NaN; one kind of
 * infinity gives that infinity times fl32(1 / scale) (NaN when that factor
 * is 0 or NaN).  The result does not depend on the order of the ranks.
 *   parts   DEVICE [nranks][n] FP8 codes of format fmt, 16-byte aligned
 *   scale   DEVICE, 1 float: the shared scale the parts were cast with
 *   out     DEVICE [n] BF16 output
 * 1 <= nranks <= 65536; n >= 0, a multiple of 16.  One kernel; it uses 96 KB
 * of shared memory per block and no global scratch memory. */
fp8_status fp8_dequant_sum(const uint8_t *parts, int32_t nranks, int64_t n, int32_t fmt,
                           const float *scale, void *out, void *stream);

/* fp8_linear_bwd for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a calling convenience, not part of the method.
 * It computes exactly what fp8_linear_bwd computes, but the two FP8 work
 * buffers (dY8, dY8t) are not passed in: they live in a fixed array in the
 * library's own device memory (64 MiB on every GPU that loads the library,
 * held until the process exits).  Callers that need it: a plugin handed only
 * its input and output tensors by a framework whose allocator owns the device
 * memory, or code that must not call cudaMalloc / cudaFree (cudaFree waits
 * for the whole device).
 *   Arguments as fp8_linear_bwd, without dY8 / dY8t.
 *   Limit: M * N <= 2^25 (33,554,432) elements; larger sizes return
 *   FP8_ERR_ARG ("exceeds the fixed work area") and nothing is enqueued.
 *   Other argument errors are those of fp8_linear_bwd.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address belongs to the device's primary
 *   context: after cudaDeviceReset on a device, do not call this function on
 *   that device again in the same process.
 *   All calls share the one array: calls that overlap on the GPU (on
 *   different streams, or from different threads without ordering) race on
 *   it; calls ordered on one stream do not.  Every call overwrites the part it
 *   uses before reading it, so it never depends on what a previous call left
 *   there. */
fp8_status fp8_linear_bwd_noalloc(const void *dY, int64_t M, int64_t N, int64_t K,
                                  const fp8_meta *meta, const fp8_recipe *recipe,
                                  const uint8_t *X8t, const uint8_t *W8t, void *dX, void *dW,
                                  void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8AMAX_H */
