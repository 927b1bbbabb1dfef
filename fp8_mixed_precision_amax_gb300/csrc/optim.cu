// optim.cu -- one Adam step on optimizer states of decoupled precision
// ("Mixed-precision training" wiki note, bullet "precision decoupling": the
// first moment in FP8, the second moment in FP16, master weights in FP16
// with tensor scaling -- 5 bytes of state per parameter instead of 12).
//
// Per element, in binary32 with one rounding per operation (Adam's bias
// correction in its textbook form, m / (1 - b1^t) and v / (1 - b2^t), and
// AdamW's decoupled weight decay):
//   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g)
//   u = (m / bc1) / (sqrt(v / bc2) + eps);  w = w - lr*(u + wd*w)
// m is decoded from E4M3 codes times the first moment's scale_inv, w from
// FP16 codes times the weights' scale_inv.  The new states get just-in-time
// per-tensor scales (fmax / amax of the new values, a history of one):
//   adam_amax_kernel    the amax of the new m and w (no stores);
//   adam_apply_kernel   recomputes, encodes with the new scales, stores m, v,
//                       w and the model's BF16 copy of w;
//   adam_scales_kernel  records the new scales after every block has decoded
//                       with the old ones.
// adam_init_kernel writes the initial state of a weight tensor: zero moments
// and the FP16 master weights under the just-in-time scale of the weights.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

namespace {

constexpr float kF16Max = 65504.0f;

__device__ __forceinline__ float f16_dec(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// Nearest FP16 value, ties to even, saturating at +-65504; NaN stays NaN.
__device__ __forceinline__ uint16_t f16_enc_sat(float v) {
    if (v != v) return 0x7e00;
    v = fminf(fmaxf(v, -kF16Max), kF16Max);
    return __half_as_ushort(__float2half_rn(v));
}

// Two E4M3 codes (low byte first) to two floats, exactly.
__device__ __forceinline__ void e4m3x2_dec(uint16_t c, float &lo, float &hi) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    lo = __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFF)));
    hi = __half2float(__ushort_as_half(static_cast<uint16_t>(h2 >> 16)));
}

struct AdamArgs {
    const uint16_t *grad;
    uint8_t *m1;
    float *m1_scale, *m1_scale_inv;
    uint16_t *m2, *w16;
    float *w_scale, *w_scale_inv;
    uint16_t *w_bf16;
    float *amax;              // [2]: new m, new w
    int64_t n;
    float lr, b1, b2, eps, wd, bc1, bc2;
    int margin;
};

struct Elem8 {
    float m[8], v[8], w[8];
};

// Loop-invariant operands, each duplicated into both lanes of an fp32 pair
// (the bias corrections are divisors, used one lane at a time).
struct AdamConst {
    uint64_t b1, omb1, b2, omb2, eps, lr, wd, msi, wsi;
    float bc1, bc2;
};

__device__ __forceinline__ AdamConst adam_const(const AdamArgs &a, float msi, float wsi) {
    AdamConst c;
    c.b1 = splat_f32x2(a.b1);
    c.omb1 = splat_f32x2(__fsub_rn(1.0f, a.b1));
    c.b2 = splat_f32x2(a.b2);
    c.omb2 = splat_f32x2(__fsub_rn(1.0f, a.b2));
    c.bc1 = a.bc1;
    c.bc2 = a.bc2;
    c.eps = splat_f32x2(a.eps);
    c.lr = splat_f32x2(a.lr);
    c.wd = splat_f32x2(a.wd);
    c.msi = splat_f32x2(msi);
    c.wsi = splat_f32x2(wsi);
    return c;
}

__device__ __forceinline__ uint64_t f16x2_to_f32x2(uint32_t h2) {
    return f32x2_pack(f16_dec(static_cast<uint16_t>(h2 & 0xFFFF)),
                      f16_dec(static_cast<uint16_t>(h2 >> 16)));
}

// The update of the 8 elements at [i, i + 8): the multiplies two lanes at a
// time, the adds and subtracts (which take products as operands), square
// roots and divides scalar, since ptxas would fuse a packed add of a packed
// product into an fma.  Every operation is one IEEE rounding, in the order
// above.
struct Raw8 {
    uint4 g4, v4, w4;
    uint2 m8;
};

__device__ __forceinline__ Raw8 adam_load8(const AdamArgs &a, int64_t i) {
    Raw8 r;
    r.g4 = *reinterpret_cast<const uint4 *>(a.grad + i);
    r.m8 = *reinterpret_cast<const uint2 *>(a.m1 + i);
    r.v4 = *reinterpret_cast<const uint4 *>(a.m2 + i);
    r.w4 = *reinterpret_cast<const uint4 *>(a.w16 + i);
    return r;
}

__device__ __forceinline__ void adam8(const Raw8 &raw, const AdamConst &k, Elem8 &e) {
    const uint4 g4 = raw.g4, v4 = raw.v4, w4 = raw.w4;
    const uint2 m8 = raw.m8;
    const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, vw[4] = {v4.x, v4.y, v4.z, v4.w},
                   ww[4] = {w4.x, w4.y, w4.z, w4.w}, mw[2] = {m8.x, m8.y};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float md0, md1;
        e4m3x2_dec(static_cast<uint16_t>(mw[j >> 1] >> (16 * (j & 1))), md0, md1);
        const uint64_t g = f32x2_from_bf16x2(gw[j]);
        const uint64_t m_old = f32x2_mul(f32x2_pack(md0, md1), k.msi);
        const uint64_t v_old = f16x2_to_f32x2(vw[j]);
        const uint64_t w_old = f32x2_mul(f16x2_to_f32x2(ww[j]), k.wsi);
        float a0, a1, b0, b1;
        // m = b1*m + (1-b1)*g
        f32x2_unpack(f32x2_mul(k.b1, m_old), a0, a1);
        f32x2_unpack(f32x2_mul(k.omb1, g), b0, b1);
        const float m0 = __fadd_rn(a0, b0), m1 = __fadd_rn(a1, b1);
        // v = b2*v + (1-b2)*(g*g)
        f32x2_unpack(f32x2_mul(k.b2, v_old), a0, a1);
        f32x2_unpack(f32x2_mul(k.omb2, f32x2_mul(g, g)), b0, b1);
        const float v0 = __fadd_rn(a0, b0), v1 = __fadd_rn(a1, b1);
        // u = (m / bc1) / (sqrt(v / bc2) + eps)
        float e0, e1;
        const float n0 = __fdiv_rn(m0, k.bc1), n1 = __fdiv_rn(m1, k.bc1);
        const float q0 = __fdiv_rn(v0, k.bc2), q1 = __fdiv_rn(v1, k.bc2);
        f32x2_unpack(k.eps, e0, e1);
        const float u0 = __fdiv_rn(n0, __fadd_rn(__fsqrt_rn(q0), e0));
        const float u1 = __fdiv_rn(n1, __fadd_rn(__fsqrt_rn(q1), e1));
        // w = w - lr * (u + wd*w)
        float w0, w1, c0, c1;
        f32x2_unpack(w_old, w0, w1);
        f32x2_unpack(f32x2_mul(k.wd, w_old), c0, c1);
        f32x2_unpack(f32x2_mul(k.lr, f32x2_pack(__fadd_rn(u0, c0), __fadd_rn(u1, c1))), c0, c1);
        e.m[2 * j] = m0;
        e.m[2 * j + 1] = m1;
        e.v[2 * j] = v0;
        e.v[2 * j + 1] = v1;
        e.w[2 * j] = __fsub_rn(w0, c0);
        e.w[2 * j + 1] = __fsub_rn(w1, c1);
    }
}

__global__ void __launch_bounds__(256) adam_amax_kernel(const AdamArgs a) {
    pdl_wait();
    pdl_trigger();
    const AdamConst k = adam_const(a, *a.m1_scale_inv, *a.w_scale_inv);
    float mm = 0.0f, mw = 0.0f;   // max |new m|, max |new w|; fmaxf skips NaN
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
    int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
    // two groups of 8 in flight per thread: this pass reads and computes only
    for (; i + stride < a.n; i += 2 * stride) {
        const Raw8 r0 = adam_load8(a, i), r1 = adam_load8(a, i + stride);
        Elem8 e;
        adam8(r0, k, e);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            mm = fmaxf(mm, fabsf(e.m[j]));
            mw = fmaxf(mw, fabsf(e.w[j]));
        }
        adam8(r1, k, e);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            mm = fmaxf(mm, fabsf(e.m[j]));
            mw = fmaxf(mw, fabsf(e.w[j]));
        }
    }
    if (i < a.n) {
        Elem8 e;
        adam8(adam_load8(a, i), k, e);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            mm = fmaxf(mm, fabsf(e.m[j]));
            mw = fmaxf(mw, fabsf(e.w[j]));
        }
    }
    uint32_t bm = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mm));
    uint32_t bw = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mw));
    if ((threadIdx.x & 31) == 0) {
        if (bm) atomicMax(reinterpret_cast<unsigned *>(a.amax), bm);
        if (bw) atomicMax(reinterpret_cast<unsigned *>(a.amax + 1), bw);
    }
}

__global__ void __launch_bounds__(256) adam_apply_kernel(const AdamArgs a) {
    pdl_wait();
    pdl_trigger();
    const AdamConst k = adam_const(a, *a.m1_scale_inv, *a.w_scale_inv);
    bool valid;
    const float sm = recipe_scale(a.amax[0], 448.0f, a.margin, *a.m1_scale, valid);
    const float sw = recipe_scale(a.amax[1], kF16Max, a.margin, *a.w_scale, valid);
    const uint64_t sm2 = splat_f32x2(sm), sw2 = splat_f32x2(sw);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < a.n;
         i += stride) {
        Elem8 e;
        adam8(adam_load8(a, i), k, e);
        uint32_t mq[2], vq[4], wq[4], bq[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float a0, a1, c0, c1;
            f32x2_unpack(f32x2_mul(f32x2_pack(e.m[2 * j], e.m[2 * j + 1]), sm2), a0, a1);
            const uint32_t c = cvt2_e4m3(a0, a1);
            if (j & 1)
                mq[j >> 1] |= c << 16;
            else
                mq[j >> 1] = c;
            vq[j] = f16_enc_sat(e.v[2 * j]) | (static_cast<uint32_t>(f16_enc_sat(e.v[2 * j + 1])) << 16);
            f32x2_unpack(f32x2_mul(f32x2_pack(e.w[2 * j], e.w[2 * j + 1]), sw2), c0, c1);
            wq[j] = f16_enc_sat(c0) | (static_cast<uint32_t>(f16_enc_sat(c1)) << 16);
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(e.w[2 * j], e.w[2 * j + 1]);
            bq[j] = *reinterpret_cast<const uint32_t *>(&b2);
        }
        *reinterpret_cast<uint2 *>(a.m1 + i) = make_uint2(mq[0], mq[1]);
        *reinterpret_cast<uint4 *>(a.m2 + i) = make_uint4(vq[0], vq[1], vq[2], vq[3]);
        *reinterpret_cast<uint4 *>(a.w16 + i) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        *reinterpret_cast<uint4 *>(a.w_bf16 + i) = make_uint4(bq[0], bq[1], bq[2], bq[3]);
    }
}

__global__ void adam_scales_kernel(const AdamArgs a) {
    pdl_wait();
    pdl_trigger();
    bool valid;
    const float sm = recipe_scale(a.amax[0], 448.0f, a.margin, *a.m1_scale, valid);
    if (valid) {
        *a.m1_scale = sm;
        *a.m1_scale_inv = __fdiv_rn(1.0f, sm);
    }
    const float sw = recipe_scale(a.amax[1], kF16Max, a.margin, *a.w_scale, valid);
    if (valid) {
        *a.w_scale = sw;
        *a.w_scale_inv = __fdiv_rn(1.0f, sw);
    }
}

// ------------------------------------------------ FP8 all-reduce: the sum --
//
// out[i] = the exact sum_r dec(q[r][i]) times fl32(1 / scale), rounded once to
// BF16 (nearest, ties to even; overflow to inf; gradual underflow; an exact
// zero is +0).  The parts of all ranks share one scale (the minimum of the
// ranks' own scales), so their codes can be decoded and summed directly.
//
// No table and no FP64.  Each thread owns 16 consecutive elements and reads
// 16 codes of a rank with one 16-byte load.  The codes are decoded exactly
// by the hardware FP8 -> FP16 conversion (two codes per instruction) and
// widened to fp32, and summed in fp32 where every partial sum is an exact
// integer multiple of a power of two below 2^24 units:
//   E4M3  values are multiples of 2^-9 of magnitude <= 448 (< 2^18 units),
//         so one accumulator holds the exact sum of 64 ranks;
//   E5M2  values span 2^-16 .. 57344, so each value v is split exactly into
//         hi = v rounded to a multiple of 2^-2 ((v + 1.5 * 2^21) - 1.5 * 2^21:
//         the sum lands in [2^21, 2^22), whose spacing is 2^-2) and
//         lo = v - hi (a multiple of 2^-16, |lo| <= 2^-3); 64 ranks of hi
//         stay below 2^24 units of 2^-2 and of lo below 2^24 units of 2^-16.
// After every 64 ranks the fp32 sums move into an int64 count of quanta
// (2^-9 for E4M3, 2^-16 for E5M2).  fl32(1 / scale) is sig * 2^es with a
// 24-bit integer sig, so the exact result is |sum| * sig * 2^(es - q): one
// 64-bit product for up to 256 ranks (|sum| < 2^40), a 128-bit one beyond.
// It is rounded to BF16's 8 significant bits (or to its subnormal quantum
// 2^-133) by one integer round-to-nearest-even and the BF16 bits are
// assembled directly.  Infinity and NaN codes are found four codes at a time
// and follow IEEE arithmetic (a NaN code, or +inf with -inf, give NaN; one
// infinity gives that infinity times the factor); they leave the fp32 sums
// meaningless, which the flags then override.

constexpr uint32_t kBf16Nan = 0x7FC0u, kBf16Inf = 0x7F80u;

// The factor fl32(1 / scale) as sig * 2^es (sig < 2^24; 0 for a zero factor)
// with its sign and non-finite classes.
struct DqFactor {
    uint64_t sig;
    int es;
    uint32_t sign;      // 0x8000 when negative
    bool is_nan, is_inf;
};

__device__ __forceinline__ DqFactor dq_factor(float sinv) {
    const uint32_t b = __float_as_uint(sinv);
    const uint32_t e = (b >> 23) & 0xFFu, m = b & 0x7FFFFFu;
    DqFactor f;
    f.sign = (b >> 16) & 0x8000u;
    f.is_nan = e == 0xFFu && m != 0u;
    f.is_inf = e == 0xFFu && m == 0u;
    f.sig = e == 0u ? m : (m | 0x800000u);
    f.es = e == 0u ? -149 : static_cast<int>(e) - 150;
    return f;
}

// BF16 bits of M' * 2^u after rounding the exact (hi:lo) * 2^E at the
// quantum 2^u: u = (its leading bit) - 7, or BF16's subnormal quantum 2^-133.
__device__ __forceinline__ uint32_t bf16_assemble(uint64_t hi, uint64_t lo, int E) {
    const int nb = hi ? 128 - __clzll(static_cast<long long>(hi))
                      : 64 - __clzll(static_cast<long long>(lo));
    int u = nb - 1 + E - 7;               // quantum of an 8-significant-bit result
    if (u < -133) u = -133;               // BF16's subnormal quantum
    const int shift = u - E;
    uint64_t M;
    if (shift <= 0) {
        M = lo << (-shift);               // exact (then fewer than 9 bits)
    } else {
        uint64_t rest, half;
        if (shift < 64) {
            M = (lo >> shift) | (hi ? (hi << (64 - shift)) : 0u);
            rest = lo & ((uint64_t(1) << shift) - 1u);
            half = uint64_t(1) << (shift - 1);
        } else {                          // shift == 64 (a 72-bit product)
            M = hi;
            rest = lo;
            half = uint64_t(1) << 63;
        }
        if (rest > half || (rest == half && (M & 1u))) ++M;   // M may become 2^8
    }
    // biased exponent u + 134 over a 7-bit mantissa M - 128; a carry to
    // M = 256 moves into the exponent, and the subnormal case (u = -133)
    // reduces to bits = M
    uint32_t bits = static_cast<uint32_t>((u + 134) * 128 + static_cast<int>(M) - 128);
    if (u + 134 >= 255 || bits >= kBf16Inf) bits = kBf16Inf;
    return bits;
}

// BF16 bits of acc * 2^QEXP * factor, exactly rounded (finite factor).
// WIDE: |acc| may reach 2^48 (more than 256 ranks), so the product takes
// two 64-bit words; otherwise |acc| < 2^40 and it fits one.
template <int FMT, bool WIDE>
__device__ __forceinline__ uint32_t bf16_of_scaled_sum(int64_t acc, const DqFactor &f) {
    constexpr int QEXP = FMT == 0 ? -9 : -16;
    if (acc == 0 || f.sig == 0) return 0u;
    const uint32_t sign = ((acc < 0) ? 0x8000u : 0u) ^ f.sign;
    const uint64_t a = static_cast<uint64_t>(acc < 0 ? -acc : acc);
    const uint64_t lo = a * f.sig, hi = WIDE ? __umul64hi(a, f.sig) : 0u;
    return bf16_assemble(hi, lo, f.es + QEXP) | sign;
}

template <int FMT, bool WIDE>
__device__ __forceinline__ uint32_t dq_finish(int64_t acc, uint32_t fe, const DqFactor &f) {
    if (fe == 0u) {
        if (f.is_nan) return kBf16Nan;
        if (f.is_inf)   // a finite sum times an infinite factor: 0 * inf is NaN
            return acc == 0 ? kBf16Nan : (kBf16Inf | (((acc < 0) ? 0x8000u : 0u) ^ f.sign));
        return bf16_of_scaled_sum<FMT, WIDE>(acc, f);
    }
    if ((fe & 1u) || fe == 6u) return kBf16Nan;        // a NaN code, or +inf with -inf
    if (f.is_nan || f.sig == 0) return kBf16Nan;       // inf * NaN, inf * 0
    return kBf16Inf | (((fe & 4u) ? 0x8000u : 0u) ^ f.sign);
}

__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Two FP8 codes (low byte first) -> their exact values as a packed fp32 pair.
template <int FMT>
__device__ __forceinline__ uint64_t fp8x2_to_f32x2(uint32_t c2) {
    uint32_t h2;
    if constexpr (FMT == 0)
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(c2)));
    else
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(c2)));
    return f32x2_pack(__half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu))),
                      __half2float(__ushort_as_half(static_cast<uint16_t>(h2 >> 16))));
}

// Flags of one word of four codes: 3 bits per code (NaN, +inf, -inf) at bit
// 3 * (base + b).
template <int FMT>
__device__ __forceinline__ void dq_special_flags(uint32_t w, int base, uint64_t &flags) {
    constexpr uint32_t smask = FMT == 0 ? 0x7F7F7F7Fu : 0x7C7C7C7Cu;   // bits that mark a special
    if (!__vcmpeq4(w & smask, smask)) return;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t cb = (w >> (8 * b)) & 0xFFu;
        if ((cb & (smask & 0xFFu)) != (smask & 0xFFu)) continue;
        uint64_t fl;
        if (FMT == 0 || (cb & 3u) != 0u)
            fl = 1u;                       // NaN
        else
            fl = (cb & 0x80u) ? 4u : 2u;   // -inf : +inf
        flags |= fl << (3 * (base + b));
    }
}

constexpr int kDqElems = 16;        // elements per thread per pass (one 16-byte load per rank)
constexpr int kDqFlushRanks = 64;   // ranks whose fp32 sums stay exact

// The exact fp32 sums of ranks [r_begin, r_end) of this thread's 16
// elements, as packed pairs (elements 2p, 2p + 1); E5M2 keeps the hi and lo
// parts apart.  Special codes are recorded in flags.
template <int FMT, int NA>
__device__ __forceinline__ void dq_sum_ranks(const uint8_t *__restrict__ q, int64_t n, int64_t i,
                                             int r_begin, int r_end,
                                             uint64_t (&s)[NA][kDqElems / 2], uint64_t &flags) {
    const uint64_t C2 = splat_f32x2(3145728.0f);   // 1.5 * 2^21
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
        for (int p = 0; p < kDqElems / 2; ++p) s[a][p] = 0u;
    // four ranks' codes in flight at a time (every partial sum is exact, so
    // the order in which ranks are added does not matter)
    for (int r0 = r_begin; r0 < r_end; r0 += 4) {
        uint4 c[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            c[u] = r0 + u < r_end ? *reinterpret_cast<const uint4 *>(
                                        q + static_cast<int64_t>(r0 + u) * n + i)
                                  : make_uint4(0u, 0u, 0u, 0u);   // code 0 adds +0
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t cw[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                dq_special_flags<FMT>(cw[h], 4 * h, flags);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const uint64_t v = fp8x2_to_f32x2<FMT>(cw[h] >> (16 * k));
                    const int p = 2 * h + k;
                    if constexpr (FMT == 0) {
                        s[0][p] = f32x2_add(s[0][p], v);
                    } else {
                        const uint64_t hi = f32x2_sub(f32x2_add(v, C2), C2);
                        s[0][p] = f32x2_add(s[0][p], hi);
                        s[NA - 1][p] = f32x2_add(s[NA - 1][p], f32x2_sub(v, hi));
                    }
                }
            }
        }
    }
}

// Element e's exact fp32 sums as an integer count of quanta (2^-9 / 2^-16).
template <int FMT, int NA>
__device__ __forceinline__ long long dq_quanta(const uint64_t (&s)[NA][kDqElems / 2], int e) {
    float a0, a1;
    f32x2_unpack(s[0][e >> 1], a0, a1);
    const float a = (e & 1) ? a1 : a0;
    if constexpr (FMT == 0) {
        return __float2ll_rn(a * 512.0f);
    } else {
        float b0, b1;
        f32x2_unpack(s[NA - 1][e >> 1], b0, b1);
        const float b = (e & 1) ? b1 : b0;
        return (__float2ll_rn(a * 4.0f) << 14) + __float2ll_rn(b * 65536.0f);
    }
}

// MODE 0: at most 64 ranks (one pass of fp32 sums, 64-bit product);
// MODE 1: at most 256 ranks (int64 sums every 64 ranks, 64-bit product);
// MODE 2: more (128-bit product).
template <int FMT, int MODE>
__global__ void __launch_bounds__(256) dequant_sum_kernel(const uint8_t *__restrict__ q,
                                                          int nranks, int64_t n,
                                                          const float *__restrict__ scale,
                                                          uint16_t *__restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const DqFactor fac = dq_factor(__fdiv_rn(1.0f, *scale));
    constexpr int NA = FMT == 0 ? 1 : 2;           // fp32 sums per element (E5M2: hi, lo)
    constexpr bool WIDE = MODE == 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * kDqElems;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * kDqElems;
         i < n; i += stride) {
        uint64_t flags = 0;
        long long acc[kDqElems];
        uint64_t s[NA][kDqElems / 2];
        if constexpr (MODE == 0) {
            dq_sum_ranks<FMT, NA>(q, n, i, 0, nranks, s, flags);
#pragma unroll
            for (int e = 0; e < kDqElems; ++e) acc[e] = dq_quanta<FMT, NA>(s, e);
        } else {
#pragma unroll
            for (int e = 0; e < kDqElems; ++e) acc[e] = 0;
            for (int f0 = 0; f0 < nranks; f0 += kDqFlushRanks) {
                dq_sum_ranks<FMT, NA>(q, n, i, f0, min(nranks, f0 + kDqFlushRanks), s, flags);
#pragma unroll
                for (int e = 0; e < kDqElems; ++e) acc[e] += dq_quanta<FMT, NA>(s, e);
            }
        }
        uint32_t o[kDqElems / 2];
#pragma unroll
        for (int j = 0; j < kDqElems / 2; ++j)
            o[j] = dq_finish<FMT, WIDE>(acc[2 * j], static_cast<uint32_t>(flags >> (6 * j)) & 7u,
                                        fac) |
                   (dq_finish<FMT, WIDE>(acc[2 * j + 1],
                                         static_cast<uint32_t>(flags >> (6 * j + 3)) & 7u, fac)
                    << 16);
        uint4 *dst = reinterpret_cast<uint4 *>(out + i);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// Initial state of a weight tensor w (BF16): m1 = 0, m2 = 0, w16 =
// enc_f16(fl32(w * s_w)) with s_w the recipe formula on amax(w) and FP16's
// largest finite value (1 when that amax is 0 or not finite); block 0 also
// writes the four scales.  amax[1] holds amax(w) from the amax kernel.
__global__ void __launch_bounds__(256) adam_init_kernel(const uint16_t *__restrict__ w,
                                                        int64_t n, int margin, uint8_t *m1,
                                                        float *m1_scale, float *m1_scale_inv,
                                                        uint16_t *m2, uint16_t *w16,
                                                        float *w_scale, float *w_scale_inv,
                                                        const float *amax) {
    pdl_wait();
    pdl_trigger();
    bool valid;
    const float sw = recipe_scale(amax[1], kF16Max, margin, 1.0f, valid);
    const uint64_t sw2 = splat_f32x2(sw);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *m1_scale = 1.0f;
        *m1_scale_inv = 1.0f;
        *w_scale = sw;
        *w_scale_inv = __fdiv_rn(1.0f, sw);
    }
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < n;
         i += stride) {
        const uint4 x4 = *reinterpret_cast<const uint4 *>(w + i);
        const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w};
        uint32_t wq[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float c0, c1;
            f32x2_unpack(f32x2_mul(f32x2_from_bf16x2(xw[j]), sw2), c0, c1);
            wq[j] = f16_enc_sat(c0) | (static_cast<uint32_t>(f16_enc_sat(c1)) << 16);
        }
        *reinterpret_cast<uint2 *>(m1 + i) = make_uint2(0u, 0u);
        *reinterpret_cast<uint4 *>(m2 + i) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(w16 + i) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
    }
}

}  // namespace

cudaError_t launch_dequant_sum(const uint8_t *parts, int nranks, int64_t n, int fmt,
                               const float *scale, void *out, int sm_count, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (n / kDqElems + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    auto *o = static_cast<uint16_t *>(out);
    const dim3 g(static_cast<unsigned>(blocks)), b(threads);
    // up to 64 ranks the fp32 sums are exact in one pass; up to 256 the
    // exact count of quanta stays below 2^40 (E5M2: 256 * 57344 * 2^16), so
    // its product with a 24-bit significand fits 64 bits
    const int mode = nranks <= kDqFlushRanks ? 0 : (nranks <= 256 ? 1 : 2);
    if (fmt == 0) {
        if (mode == 0) return launch_pdl(dequant_sum_kernel<0, 0>, g, b, 0, st, parts, nranks, n, scale, o);
        if (mode == 1) return launch_pdl(dequant_sum_kernel<0, 1>, g, b, 0, st, parts, nranks, n, scale, o);
        return launch_pdl(dequant_sum_kernel<0, 2>, g, b, 0, st, parts, nranks, n, scale, o);
    }
    if (mode == 0) return launch_pdl(dequant_sum_kernel<1, 0>, g, b, 0, st, parts, nranks, n, scale, o);
    if (mode == 1) return launch_pdl(dequant_sum_kernel<1, 1>, g, b, 0, st, parts, nranks, n, scale, o);
    return launch_pdl(dequant_sum_kernel<1, 2>, g, b, 0, st, parts, nranks, n, scale, o);
}

cudaError_t launch_adam_init(const AdamInitSpec &s, int sm_count, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(s.amax, 0, sizeof(float), st);   // the first moment's amax
    if (e != cudaSuccess) return e;
    if ((e = launch_amax(s.w, s.n, s.amax + 1, sm_count, st)) != cudaSuccess) return e;
    const int threads = 256;
    int64_t blocks = (s.n / 8 + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(adam_init_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st,
                      static_cast<const uint16_t *>(s.w), s.n, s.margin, s.m1, s.m1_scale,
                      s.m1_scale_inv, s.m2, s.w16, s.w_scale, s.w_scale_inv,
                      static_cast<const float *>(s.amax));
}

cudaError_t launch_adam_step(const AdamSpec &s, int sm_count, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(s.amax, 0, 2 * sizeof(float), st);
    if (e != cudaSuccess) return e;
    AdamArgs a{static_cast<const uint16_t *>(s.grad), s.m1, s.m1_scale, s.m1_scale_inv, s.m2,
               s.w16, s.w_scale, s.w_scale_inv, static_cast<uint16_t *>(s.w_bf16), s.amax, s.n,
               s.lr, s.b1, s.b2, s.eps, s.wd, s.bc1, s.bc2, s.margin};
    if (s.n > 0) {
        const int threads = 256;
        int64_t blocks = (s.n / 8 + threads - 1) / threads;
        const int64_t cap = static_cast<int64_t>(sm_count) * 8;
        if (blocks > cap) blocks = cap;
        const dim3 g(static_cast<unsigned>(blocks)), b(threads);
        if ((e = launch_pdl(adam_amax_kernel, g, b, 0, st, a)) != cudaSuccess) return e;
        if ((e = launch_pdl(adam_apply_kernel, g, b, 0, st, a)) != cudaSuccess) return e;
    }
    return launch_pdl(adam_scales_kernel, dim3(1), dim3(1), 0, st, a);
}

}  // namespace fp8k
