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
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

namespace {

constexpr float kF16Max = 65504.0f;

__device__ __forceinline__ float f16_dec(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// Two values to their nearest FP16 values, ties to even, saturating at
// +-65504 (lo in the low half): one packed saturating conversion.  It rounds
// first and then saturates, which gives the same codes as clamping first: a
// value that rounds past 65504 is at least 65520 and saturates to 65504.  Its
// NaN result is the canonical FP16 NaN, so a NaN input is set to 0x7e00, the
// library's FP16 NaN code.
__device__ __forceinline__ uint32_t f16x2_enc_sat(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    if (lo != lo || hi != hi) {
        if (lo != lo) r = (r & 0xFFFF0000u) | 0x7e00u;
        if (hi != hi) r = (r & 0x0000FFFFu) | 0x7e000000u;
    }
    return r;
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

// Loop-invariant operands, each duplicated into both lanes of an fp32 pair;
// the bias corrections as divisors known in advance.
struct AdamConst {
    uint64_t b1, omb1, b2, omb2, eps, lr, wd, msi, wsi;
    DivConst bc1, bc2;
};

__device__ __forceinline__ AdamConst adam_const(const AdamArgs &a, float msi, float wsi) {
    AdamConst c;
    c.b1 = splat_f32x2(a.b1);
    c.omb1 = splat_f32x2(__fsub_rn(1.0f, a.b1));
    c.b2 = splat_f32x2(a.b2);
    c.omb2 = splat_f32x2(__fsub_rn(1.0f, a.b2));
    c.bc1 = div_const(a.bc1);
    c.bc2 = div_const(a.bc2);
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

// m = b1*m + (1-b1)*g for one pair: m decoded from its two E4M3 codes times
// the first moment's scale_inv, g the pair's gradient widened to fp32.
__device__ __forceinline__ void adam_m_pair(uint16_t mcodes, uint64_t g, const AdamConst &k,
                                            float &m0, float &m1) {
    float md0, md1, a0, a1, b0, b1;
    e4m3x2_dec(mcodes, md0, md1);
    const uint64_t m_old = f32x2_mul(f32x2_pack(md0, md1), k.msi);
    f32x2_unpack(f32x2_mul(k.b1, m_old), a0, a1);
    f32x2_unpack(f32x2_mul(k.omb1, g), b0, b1);
    m0 = __fadd_rn(a0, b0);
    m1 = __fadd_rn(a1, b1);
}

__device__ __forceinline__ void adam8(const Raw8 &raw, const AdamConst &k, Elem8 &e) {
    const uint4 g4 = raw.g4, v4 = raw.v4, w4 = raw.w4;
    const uint2 m8 = raw.m8;
    const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, vw[4] = {v4.x, v4.y, v4.z, v4.w},
                   ww[4] = {w4.x, w4.y, w4.z, w4.w}, mw[2] = {m8.x, m8.y};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t g = f32x2_from_bf16x2(gw[j]);
        const uint64_t v_old = f16x2_to_f32x2(vw[j]);
        const uint64_t w_old = f32x2_mul(f16x2_to_f32x2(ww[j]), k.wsi);
        float a0, a1, b0, b1, m0, m1;
        // m = b1*m + (1-b1)*g
        adam_m_pair(static_cast<uint16_t>(mw[j >> 1] >> (16 * (j & 1))), g, k, m0, m1);
        // v = b2*v + (1-b2)*(g*g)
        f32x2_unpack(f32x2_mul(k.b2, v_old), a0, a1);
        f32x2_unpack(f32x2_mul(k.omb2, f32x2_mul(g, g)), b0, b1);
        const float v0 = __fadd_rn(a0, b0), v1 = __fadd_rn(a1, b1);
        // u = (m / bc1) / (sqrt(v / bc2) + eps); the bias corrections are
        // divisors known in advance, each quotient correctly rounded
        float e0, e1, n0, n1, q0, q1;
        div_by_const2(m0, m1, k.bc1, n0, n1);
        div_by_const2(v0, v1, k.bc2, q0, q1);
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
            vq[j] = f16x2_enc_sat(e.v[2 * j], e.v[2 * j + 1]);
            f32x2_unpack(f32x2_mul(f32x2_pack(e.w[2 * j], e.w[2 * j + 1]), sw2), c0, c1);
            wq[j] = f16x2_enc_sat(c0, c1);
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
// Layout: persistent blocks of 8 consumer warps and 1 producer warp walk
// chunks of 4096 elements.  The producer stages each rank's 4 KB of codes of
// a chunk into shared memory with untiled bulk copies, 8 ranks per stage, in
// a ring of 3 stages, so HBM stays busy while the consumers compute; every
// consumer thread owns 16 consecutive elements of the chunk.  Waits are
// bounded.
//
// Arithmetic: no table, no FP64 and no conversion to or from fp32 (GB300
// runs those on its narrow FP64 / conversion pipe).  Codes become exact
// FP16 values two at a time (an E5M2 code is the top byte of its FP16
// pattern; E4M3 takes cvt.rn.f16x2.e4m3x2), and PTX mixed-precision adds
// (add.rn.f32.f16) put them into fp32 accumulators whose partial sums stay
// exact integer multiples below 2^24 units: E4M3 in one accumulator; E5M2
// in one accumulator too when each of a thread's codes is zero or at least
// 2^-3 (those are multiples of 2^-5, and 8 of them stay below 2^24 such
// units), else split exactly in packed FP16 into a 2^-2 grid part and the
// remainder (DqSums).  The fp32 sums become int64 counts of quanta (2^-9 for E4M3,
// 2^-16 for E5M2) by the exact "magic number" conversion (adding 1.5 * 2^23
// units puts the integer in the low mantissa bits), after every stage of 8
// ranks when there are more than 8.  fl32(1 / scale) is sig * 2^es with a
// 24-bit integer sig.  Each element is rounded once, by the first of three
// tiers that applies: (1) up to 8 ranks, a = fl32(sum) and p = fl32(a * sinv)
// rounded to BF16, unless p's exact error (a exact) or a rounding test (a
// inexact) says that may differ (dq_tier1_ok); (2) a result in BF16's normal
// range: the exact 64-bit product |sum| * sig, normalised, its top 8 bits
// rounded to nearest even with a sticky bit; (3) the general integer path (subnormal and
// overflowing results, special codes, non-finite factors; a 128-bit product
// beyond 256 ranks).  Special codes decode to FP16 infinities and NaN, so up
// to 8 ranks an element's fp32 sum is not finite exactly when it holds one,
// and only such an element reads its codes again; beyond 8 ranks they are
// detected with three integer operations per four codes and a thread that
// saw one re-reads its codes.  Either way they follow IEEE arithmetic (a NaN
// code, or +inf with -inf, give NaN; one infinity gives that infinity times
// the factor).

constexpr uint32_t kBf16Nan = 0x7FC0u, kBf16Inf = 0x7F80u;

// Set when the sum kernel gives up a bounded wait (read by fp8_sync_status).
__device__ unsigned g_sum_error_flags = 0;

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

// General rounding: BF16 bits of the exact (hi:lo) * 2^E (not zero), at the
// quantum 2^u with u = (its leading bit) - 7, or BF16's subnormal quantum
// 2^-133; overflow gives inf.
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

// BF16 bits of acc * 2^QEXP * factor for a finite factor, by the general
// rounding.  WIDE: |acc| may reach 2^48 (more than 256 ranks), so the
// product takes two 64-bit words; otherwise |acc| < 2^40 and it fits one.
template <int FMT, bool WIDE>
__device__ __forceinline__ uint32_t bf16_of_scaled_sum(int64_t acc, const DqFactor &f) {
    constexpr int QEXP = FMT == 0 ? -9 : -16;
    if (acc == 0 || f.sig == 0) return 0u;
    const uint32_t sign = ((acc < 0) ? 0x8000u : 0u) ^ f.sign;
    const uint64_t a = static_cast<uint64_t>(acc < 0 ? -acc : acc);
    const uint64_t lo = a * f.sig, hi = WIDE ? __umul64hi(a, f.sig) : 0u;
    return bf16_assemble(hi, lo, f.es + QEXP) | sign;
}

// The general path of one element: fe = its special flags (NaN 1, +inf 2,
// -inf 4), acc = its exact sum of the finite codes.
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

// The fast path for a finite, nonzero factor and |acc| < 2^40: BF16 bits of
// acc * 2^QEXP * factor when the result's leading bit lies in BF16's normal
// range (2^-126 .. 2^127; rounding may still overflow to inf); otherwise
// sets `slow`.
template <int FMT>
__device__ __forceinline__ uint32_t bf16_fast(int64_t acc, const DqFactor &f, bool &slow) {
    constexpr int QEXP = FMT == 0 ? -9 : -16;
    if (acc == 0) return 0u;
    const uint32_t sign = ((acc < 0) ? 0x8000u : 0u) ^ f.sign;
    const uint64_t P = static_cast<uint64_t>(acc < 0 ? -acc : acc) * f.sig;   // < 2^64
    const int lz = __clzll(static_cast<long long>(P));
    const int lead = 63 - lz + f.es + QEXP;            // P * 2^E in [2^lead, 2^(lead+1))
    if (lead < -126 || lead > 127) {
        slow = true;
        return 0u;
    }
    const uint64_t N = P << lz;                        // leading bit at bit 63
    const uint32_t hi = static_cast<uint32_t>(N >> 32);
    uint32_t M = hi >> 24;                             // the 8 significant bits kept
    const uint32_t rest = (hi & 0xFFFFFFu) | (static_cast<uint32_t>(N) != 0u ? 1u : 0u);
    M += (rest > 0x800000u || (rest == 0x800000u && (M & 1u))) ? 1u : 0u;
    uint32_t bits = static_cast<uint32_t>((lead + 127) * 128) + M - 128u;   // carry moves up
    if (bits >= kBf16Inf) bits = kBf16Inf;
    return bits | sign;
}

// Flags of one word of four codes: 3 bits per code (NaN, +inf, -inf) at bit
// 3 * (base + b).
template <int FMT>
__device__ __forceinline__ void dq_special_flags(uint32_t w, int base, uint64_t &flags) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t cb = (w >> (8 * b)) & 0xFFu;
        uint64_t fl = 0;
        if (FMT == 0) {
            if ((cb & 0x7Fu) == 0x7Fu) fl = 1u;                           // NaN
        } else if ((cb & 0x7Cu) == 0x7Cu) {
            fl = (cb & 3u) ? 1u : ((cb & 0x80u) ? 4u : 2u);              // NaN, -inf, +inf
        }
        flags |= fl << (3 * (base + b));
    }
}

// Bit 7 of a byte of the result is set where the code in that byte of w is
// special (E4M3: S.1111.111; E5M2: exponent 31); the additions carry into no
// other byte.
template <int FMT>
__device__ __forceinline__ uint32_t dq_special_bits(uint32_t w) {
    return FMT == 0 ? (w & 0x7F7F7F7Fu) + 0x01010101u : (w & 0x7C7C7C7Cu) + 0x04040404u;
}

// 1.5 * 2^k as a binary32 constant (normal k).
__host__ __device__ constexpr uint32_t magic_bits(int k) {
    return (static_cast<uint32_t>(k + 127) << 23) | 0x400000u;
}

// An fp32 value that is an integer multiple n of 2^U with |n| < 2^22, as n:
// adding 1.5 * 2^(23 + U) (exact: the sum keeps spacing 2^U) leaves n in the
// low mantissa bits.
template <int U>
__device__ __forceinline__ long long f32_units(float a) {
    const float m = __uint_as_float(magic_bits(U + 23));
    return static_cast<long long>(static_cast<int32_t>(__float_as_uint(__fadd_rn(a, m)) -
                                                       magic_bits(U + 23)));
}

constexpr int kDqElems = 16;                          // elements per consumer thread
constexpr int kDqConsumers = 256;                     // consumer threads per block
constexpr int kDqChunk = kDqConsumers * kDqElems;     // elements per chunk (4096)
constexpr int kDqGroup = 8;                           // ranks per stage
constexpr int kDqStages = 3;
constexpr size_t kDqSmem = 128 + static_cast<size_t>(kDqStages) * kDqGroup * kDqChunk +
                           2 * kDqStages * 8 + 16;

// fp32 += FP16 value, one instruction: the FP16 operand is widened exactly
// and the sum rounded once (PTX mixed-precision add).
__device__ __forceinline__ float add_f32_f16(float acc, uint16_t h) {
    asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(h));
    return acc;
}

// The fp32 sums of one thread's 16 elements.  Codes become exact FP16
// values two at a time (E5M2: the code is the top byte of its FP16 pattern,
// one byte permute per pair; E4M3: one cvt.rn.f16x2.e4m3x2 per pair) and
// are added into fp32 accumulators by mixed-precision adds.  E4M3 values
// are multiples of 2^-9 of magnitude <= 448 (< 2^18 units), so one
// accumulator holds the exact sum of 16 ranks.  E5M2 values span
// 2^-16 .. 57344, so each pair is split exactly in packed FP16: hi = v
// rounded to a multiple of 2^-2 ((v + 384) - 384: for |v| < 128 the sum lies
// in [256, 512), whose spacing is 2^-2; larger E5M2 values are multiples of
// 32 and pass unchanged) and lo = v - hi (a multiple of 2^-16, |lo| <=
// 2^-3); 16 ranks of each stay below 2^22 units.
template <int FMT>
struct DqSums {
    static constexpr int NA = FMT == 0 ? 1 : 2;
    float s[NA][kDqElems];
    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
            for (int e = 0; e < kDqElems; ++e) s[a][e] = 0.0f;
    }
    // add the 16 codes of one rank (one 16-byte vector)
    __device__ __forceinline__ void add(const uint4 c, uint32_t &special) {
        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            special |= dq_special_bits<FMT>(cw[h]);
#pragma unroll
            for (int k = 0; k < 4; k += 2) {
                const int e = 4 * h + k;
                uint32_t v2;   // FP16 values of codes k (low half) and k + 1
                if constexpr (FMT == 0) {
                    asm("cvt.rn.f16x2.e4m3x2 %0, %1;"
                        : "=r"(v2)
                        : "h"(static_cast<uint16_t>(cw[h] >> (8 * k))));
                    s[0][e] = add_f32_f16(s[0][e], static_cast<uint16_t>(v2));
                    s[0][e + 1] = add_f32_f16(s[0][e + 1], static_cast<uint16_t>(v2 >> 16));
                } else {
                    v2 = __byte_perm(cw[h], 0u, k == 0 ? 0x1404u : 0x3424u);
                    const __half2 v = *reinterpret_cast<const __half2 *>(&v2);
                    const __half2 c384 = __half2half2(__ushort_as_half(0x5E00u));   // 384
                    const __half2 hi = __hsub2(__hadd2(v, c384), c384);
                    const __half2 lo = __hsub2(v, hi);
                    s[0][e] = add_f32_f16(s[0][e], __half_as_ushort(__low2half(hi)));
                    s[0][e + 1] = add_f32_f16(s[0][e + 1], __half_as_ushort(__high2half(hi)));
                    s[1][e] = add_f32_f16(s[1][e], __half_as_ushort(__low2half(lo)));
                    s[1][e + 1] = add_f32_f16(s[1][e + 1], __half_as_ushort(__high2half(lo)));
                }
            }
        }
    }
    // Add the 16 codes of one rank unsplit: one accumulator per element.
    // E4M3 sums are always exact this way.  An E5M2 value of magnitude
    // >= 2^-3 is a multiple of 2^-5, and 8 of them (at most 8 * 57344 <
    // 2^19) stay below 2^24 such units, so their fp32 sum is exact too
    // (e5m2_small_bits marks the codes for which it may not be).
    __device__ __forceinline__ void add_direct(const uint4 c) {
        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
#pragma unroll
            for (int k = 0; k < 4; k += 2) {
                const int e = 4 * h + k;
                uint32_t v2;
                if constexpr (FMT == 0) {
                    asm("cvt.rn.f16x2.e4m3x2 %0, %1;"
                        : "=r"(v2)
                        : "h"(static_cast<uint16_t>(cw[h] >> (8 * k))));
                } else {
                    v2 = __byte_perm(cw[h], 0u, k == 0 ? 0x1404u : 0x3424u);
                }
                s[0][e] = add_f32_f16(s[0][e], static_cast<uint16_t>(v2));
                s[0][e + 1] = add_f32_f16(s[0][e + 1], static_cast<uint16_t>(v2 >> 16));
            }
        }
    }
    // element e's exact sum as an integer count of quanta (2^-9 / 2^-16)
    __device__ __forceinline__ long long quanta(int e) const {
        if constexpr (FMT == 0)
            return f32_units<-9>(s[0][e]);
        else
            return (f32_units<-2>(s[0][e]) << 14) + f32_units<-16>(s[NA - 1][e]);
    }
};

// Bit 7 of a byte of the result is set where the E5M2 code in that byte of
// the vector is nonzero and below 2^-3 in magnitude ((c & 0x7F) in 1 ..
// 0x2F); no carry leaves a byte.
__device__ __forceinline__ uint32_t e5m2_small_bits(const uint4 c) {
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    uint32_t small = 0;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const uint32_t x = cw[h] & 0x7F7F7F7Fu;
        small |= (x + 0x7F7F7F7Fu) & ~(x + 0x50505050u);
    }
    return small;
}

// The exact count of 2^-16 quanta of an unsplit E5M2 sum a (a multiple of
// 2^-5 below 2^19): a = h + l with h = a rounded to a multiple of 2^-2 (by
// adding and removing 1.5 * 2^21) and l = a - h, both exact.
__device__ __forceinline__ long long e5m2_direct_quanta(float a) {
    const float m = __uint_as_float(magic_bits(21));
    const float t = __fadd_rn(a, m);
    const long long hi = static_cast<int32_t>(__float_as_uint(t) - magic_bits(21));
    return (hi << 14) + f32_units<-16>(__fsub_rn(a, __fsub_rn(t, m)));
}

// Special flags (NaN 1, +inf 2, -inf 4) of element k of the ranks' codes
// (read from global memory; only for an element whose sum is not finite).
template <int FMT>
__device__ __forceinline__ uint32_t dq_element_flags(const uint8_t *q, int nranks, int64_t n,
                                                     int64_t k) {
    uint32_t fe = 0;
    for (int r = 0; r < nranks; ++r) {
        const uint32_t cb = q[static_cast<int64_t>(r) * n + k];
        if (FMT == 0) {
            if ((cb & 0x7Fu) == 0x7Fu) fe |= 1u;
        } else if ((cb & 0x7Cu) == 0x7Cu) {
            fe |= (cb & 3u) ? 1u : ((cb & 0x80u) ? 4u : 2u);
        }
    }
    return fe;
}

// Tier 1 of the 8-rank path for a finite nonzero factor: a = fl32(S) for the
// element's exact sum S, p = fl32(a * sinv) and e = fma(a, sinv, -p), its
// exact error (p at least 2^-100).  BF16 rounds at bit 16 of the binary32
// pattern; its midpoints have low 16 bits 0x8000, and every midpoint is a
// binary32 value.
//  * a exact (a == S): a * sinv = p + e, so rounding p to BF16 rounds
//    S * sinv correctly unless p is a midpoint while e != 0.
//  * a inexact (the split sums do not add exactly; a rounding test in the
//    manner of Ziv): |S - a| <= 2^-24 |a| gives |S * sinv - p| < 1.5 ulp(p),
//    so when p's low 16 bits differ from 0x8000 by at least 2, S * sinv lies
//    on p's side of every midpoint and BF16(S * sinv) is p rounded.  (The
//    window is not used for exact sums: a factor such as fl32(amax / 57344),
//    whose significand repeats the bits of 1/7, puts the products of short
//    sums next to midpoints far more often than chance.)
// Otherwise, and when p is below 2^-100 or not finite, the element takes the
// integer tiers.  A zero sum gives +0 when the factor is positive.
__device__ __forceinline__ bool dq_tier1_ok(float a, float p, float e, bool exact,
                                            bool pos_factor) {
    const float ap = fabsf(p);
    const uint32_t low = __float_as_uint(p) & 0xFFFFu;
    const bool declined = exact ? (low == 0x8000u && e != 0.0f) : (low - 0x7FFFu <= 2u);
    return (ap >= 0x1p-100f && ap <= 0x1.fffffep127f && !declined) || (a == 0.0f && pos_factor);
}

// One element of the 8-rank path after tier 1 declined some element of its
// thread: BF16 bits of its result when tier 1 does not stand for it (the
// integer tiers on its exact count of quanta), else 0xFFFFFFFF.  hs / ls:
// its fp32 sums (ls = 0 unless split; E4M3: hs alone).  Not inlined, so that
// the integer tiers take one copy of code rather than one per element: warps
// enter them often on codes spread over many binades, and sixteen inlined
// copies overflowed the instruction cache.
template <int FMT>
__device__ __noinline__ uint32_t dq_slow_element(float hs, float ls, bool split, bool general,
                                                 bool pos_factor, float sinv, DqFactor fac,
                                                 const uint8_t *q, int nranks, int64_t n,
                                                 int64_t k) {
    if (!general) {
        const float a = split ? __fadd_rn(hs, ls) : hs;
        const float p = __fmul_rn(a, sinv);
        if (dq_tier1_ok(a, p, __fmaf_rn(a, sinv, -p), !split || __fsub_rn(a, hs) == ls,
                        pos_factor))
            return 0xFFFFFFFFu;
    }
    const uint32_t fe = fabsf(hs) <= 0x1.fffffep127f ? 0u : dq_element_flags<FMT>(q, nranks, n, k);
    long long qa = 0;
    if (fe == 0u) {
        if constexpr (FMT == 0)
            qa = f32_units<-9>(hs);
        else
            qa = split ? (f32_units<-2>(hs) << 14) + f32_units<-16>(ls) : e5m2_direct_quanta(hs);
    }
    bool outside = general || fe != 0u;
    uint32_t b = 0;
    if (!outside) b = bf16_fast<FMT>(qa, fac, outside);
    if (outside) b = dq_finish<FMT, false>(qa, fe, fac);
    return b & 0xFFFFu;
}

// MODE 0: at most 8 ranks (one stage, no int64 sums during the walk);
// MODE 1: at most 256 ranks (int64 sums after every stage, 64-bit product);
// MODE 2: more (128-bit product on the general path).
template <int FMT, int MODE>
__global__ void __launch_bounds__(kDqConsumers + 32, 2)
    dequant_sum_kernel(const uint8_t *__restrict__ q, int nranks, int64_t n,
                       const float *__restrict__ scale, uint16_t *__restrict__ out) {
    extern __shared__ uint8_t dq_smem_raw[];
    uint8_t *buf = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dq_smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    uint64_t *bars = reinterpret_cast<uint64_t *>(buf + static_cast<size_t>(kDqStages) *
                                                            kDqGroup * kDqChunk);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kDqStages);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * kDqStages);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int st = 0; st < kDqStages; ++st) {
            mbar_init(full0 + 8 * st, 1);
            mbar_init(empty0 + 8 * st, kDqConsumers / 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    const int64_t nchunks = (n + kDqChunk - 1) / kDqChunk;
    const int groups = (nranks + kDqGroup - 1) / kDqGroup;

    if (tid >= kDqConsumers) {
        // ------------------------------------------------------- producer
        if (tid == kDqConsumers) {
            int issued[kDqStages] = {};
            int64_t j = 0;
            bool ok = true;
            for (int64_t c = blockIdx.x; ok && c < nchunks; c += gridDim.x) {
                const int64_t e0 = c * kDqChunk;
                const int64_t left = n - e0;
                const uint32_t bytes = static_cast<uint32_t>(left < kDqChunk ? left : kDqChunk);
                for (int gi = 0; gi < groups; ++gi, ++j) {
                    const int st = static_cast<int>(j % kDqStages);
                    if (j >= kDqStages &&
                        !mbar_wait(empty0 + 8 * st,
                                   static_cast<uint32_t>(((j / kDqStages) & 1) ^ 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int r0 = gi * kDqGroup, nr = min(kDqGroup, nranks - r0);
                    mbar_arrive_expect_tx(full0 + 8 * st, static_cast<uint32_t>(nr) * bytes);
                    for (int u = 0; u < nr; ++u)
                        bulk_load_1d(smem_u32(buf + (static_cast<size_t>(st) * kDqGroup + u) *
                                                        kDqChunk),
                                     q + static_cast<int64_t>(r0 + u) * n + e0, bytes,
                                     full0 + 8 * st);
                    ++issued[st];
                }
            }
            if (!ok) {
                atomicOr(&g_sum_error_flags, kErrWaitTimeout);
                *abort_flag = 1;
            }
            // every copy issued must land before the block may exit
            for (int st = 0; st < kDqStages; ++st)
                if (issued[st] > 0)
                    mbar_wait(full0 + 8 * st, static_cast<uint32_t>((issued[st] - 1) & 1), nullptr,
                              100000000ull);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int lane = tid & 31;
    const float sinv = __fdiv_rn(1.0f, *scale);
    const DqFactor fac = dq_factor(sinv);
    const bool general = fac.is_nan || fac.is_inf || fac.sig == 0 || MODE == 2;
    int64_t j = 0;
    if constexpr (MODE == 0) {
        // one stage holds every rank; a thread's codes are added unsplit
        // unless one of them is an E5M2 code below 2^-3, which needs the
        // hi/lo split; special codes make the sum non-finite, and only such
        // elements look at their codes again
        const bool pos_factor = sinv > 0.0f;
        const uint64_t sinv2 = splat_f32x2(sinv);
        for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++j) {
            const int64_t i = c * kDqChunk + static_cast<int64_t>(tid) * kDqElems;
            const bool in = i < n;
            const int st = static_cast<int>(j % kDqStages);
            const bool got = mbar_wait(full0 + 8 * st, static_cast<uint32_t>((j / kDqStages) & 1),
                                       abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) {
                    atomicOr(&g_sum_error_flags, kErrWaitTimeout);
                    *abort_flag = 1;
                }
                return;
            }
            // the ranks' codes are added unsplit, or split when an E5M2 code
            // below 2^-3 is among them
            DqSums<FMT> sums;
            sums.clear();
            bool split = false;
            if (in) {
                const uint8_t *src = buf + static_cast<size_t>(st) * kDqGroup * kDqChunk +
                                     static_cast<size_t>(tid) * kDqElems;
                // rank 0's codes first: with a code below 2^-3 among them
                // (codes spread over all binades) the thread splits at once
                const uint4 c0 = *reinterpret_cast<const uint4 *>(src);
                uint32_t small = 0;
                if constexpr (FMT == 1) small = e5m2_small_bits(c0);
                if ((small & 0x80808080u) == 0u) {
                    sums.add_direct(c0);
#pragma unroll
                    for (int u = 1; u < kDqGroup; ++u) {
                        if (u < nranks) {
                            const uint4 cv = *reinterpret_cast<const uint4 *>(
                                src + static_cast<size_t>(u) * kDqChunk);
                            if constexpr (FMT == 1) small |= e5m2_small_bits(cv);
                            sums.add_direct(cv);
                        }
                    }
                }
                if constexpr (FMT == 1) {
                    if ((small & 0x80808080u) != 0u) {
                        split = true;
                        sums.clear();
                        uint32_t unused = 0;
#pragma unroll
                        for (int u = 0; u < kDqGroup; ++u)
                            if (u < nranks)
                                sums.add(*reinterpret_cast<const uint4 *>(
                                             src + static_cast<size_t>(u) * kDqChunk),
                                         unused);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
            if (!in) continue;
            // tier 1 takes a = fl32 of the element's exact sum: the unsplit
            // sum itself (exact), or hs + ls rounded once, exact when
            // (hs + ls) - hs == ls (Fast2Sum when |hs| >= |ls|; otherwise
            // |hs| < |ls| <= 1 and the sum has at most 17 bits)
            uint32_t o[kDqElems / 2];
            bool odd = general;
            if (!odd && !split) {
#pragma unroll
                for (int e = 0; e < kDqElems; e += 2) {
                    const float a0 = sums.s[0][e], a1 = sums.s[0][e + 1];
                    const uint64_t a2 = f32x2_pack(a0, a1);
                    const uint64_t p2 = f32x2_mul(a2, sinv2);
                    const uint64_t e2 = f32x2_fma(a2, sinv2, p2 ^ 0x8000000080000000ull);
                    float p0, p1, e0, e1;
                    f32x2_unpack(p2, p0, p1);
                    f32x2_unpack(e2, e0, e1);
                    if (!dq_tier1_ok(a0, p0, e0, true, pos_factor) ||
                        !dq_tier1_ok(a1, p1, e1, true, pos_factor))
                        odd = true;
                    uint32_t h;
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(p1), "f"(p0));
                    o[e >> 1] = h;
                }
            } else if (!odd) {
#pragma unroll
                for (int e = 0; e < kDqElems; e += 2) {
                    float a[2];
                    bool exact[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float hs = sums.s[0][e + h], ls = sums.s[DqSums<FMT>::NA - 1][e + h];
                        a[h] = __fadd_rn(hs, ls);
                        exact[h] = __fsub_rn(a[h], hs) == ls;
                    }
                    const uint64_t a2 = f32x2_pack(a[0], a[1]);
                    const uint64_t p2 = f32x2_mul(a2, sinv2);
                    const uint64_t e2 = f32x2_fma(a2, sinv2, p2 ^ 0x8000000080000000ull);
                    float p0, p1, e0, e1;
                    f32x2_unpack(p2, p0, p1);
                    f32x2_unpack(e2, e0, e1);
                    if (!dq_tier1_ok(a[0], p0, e0, exact[0], pos_factor) ||
                        !dq_tier1_ok(a[1], p1, e1, exact[1], pos_factor))
                        odd = true;
                    uint32_t h;
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(p1), "f"(p0));
                    o[e >> 1] = h;
                }
            } else {
#pragma unroll
                for (int w = 0; w < kDqElems / 2; ++w) o[w] = 0u;
            }
            if (odd) {
                // the elements tier 1 declines: the exact count of quanta,
                // rounded by the 64-bit path or the general one
#pragma unroll
                for (int e = 0; e < kDqElems; ++e) {
                    const uint32_t b = dq_slow_element<FMT>(
                        sums.s[0][e], sums.s[DqSums<FMT>::NA - 1][e], split, general, pos_factor,
                        sinv, fac, q, nranks, n, i + e);
                    if (b == 0xFFFFFFFFu) continue;
                    const int w = e >> 1, sh = (e & 1) * 16;
                    o[w] = (o[w] & ~(0xFFFFu << sh)) | (b << sh);
                }
            }
            uint4 *dst = reinterpret_cast<uint4 *>(out + i);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
    } else {
        // more than 8 ranks: int64 sums of quanta after every stage of 8
        for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
            const int64_t i = c * kDqChunk + static_cast<int64_t>(tid) * kDqElems;
            const bool in = i < n;
            DqSums<FMT> sums;
            sums.clear();
            long long acc[kDqElems];
#pragma unroll
            for (int e = 0; e < kDqElems; ++e) acc[e] = 0;
            uint32_t special = 0;
            for (int gi = 0; gi < groups; ++gi, ++j) {
                const int st = static_cast<int>(j % kDqStages);
                const bool got = mbar_wait(full0 + 8 * st, static_cast<uint32_t>((j / kDqStages) & 1),
                                           abort_flag);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    if (lane == 0) {
                        atomicOr(&g_sum_error_flags, kErrWaitTimeout);
                        *abort_flag = 1;
                    }
                    return;
                }
                const int nr = min(kDqGroup, nranks - gi * kDqGroup);
                if (in) {
                    const uint8_t *src = buf + static_cast<size_t>(st) * kDqGroup * kDqChunk +
                                         static_cast<size_t>(tid) * kDqElems;
#pragma unroll
                    for (int u = 0; u < kDqGroup; ++u)
                        if (u < nr)
                            sums.add(*reinterpret_cast<const uint4 *>(src + static_cast<size_t>(u) *
                                                                                kDqChunk),
                                     special);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * st);
#pragma unroll
                for (int e = 0; e < kDqElems; ++e) acc[e] += sums.quanta(e);
                sums.clear();
            }
            if (!in) continue;
            // special codes (re-read from global memory; rare) for the general path
            uint64_t flags = 0;
            if ((special & 0x80808080u) != 0u) {
                for (int r = 0; r < nranks; ++r) {
                    const uint4 cv = *reinterpret_cast<const uint4 *>(q + static_cast<int64_t>(r) * n + i);
                    dq_special_flags<FMT>(cv.x, 0, flags);
                    dq_special_flags<FMT>(cv.y, 4, flags);
                    dq_special_flags<FMT>(cv.z, 8, flags);
                    dq_special_flags<FMT>(cv.w, 12, flags);
                }
            }
            // each element: the normalised 64-bit integer rounding (results in
            // BF16's normal range) or the general path (special codes,
            // non-finite factors, subnormal or overflowing results)
            uint32_t o[kDqElems / 2];
#pragma unroll
            for (int e = 0; e < kDqElems; ++e) {
                const uint32_t fe = static_cast<uint32_t>(flags >> (3 * e)) & 7u;
                bool outside = general || fe != 0u;
                uint32_t b = 0;
                if (!outside) b = bf16_fast<FMT>(acc[e], fac, outside);
                if (outside) b = dq_finish<FMT, MODE == 2>(acc[e], fe, fac);
                if (e & 1)
                    o[e >> 1] |= (b & 0xFFFFu) << 16;
                else
                    o[e >> 1] = b & 0xFFFFu;
            }
            uint4 *dst = reinterpret_cast<uint4 *>(out + i);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
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
            wq[j] = f16x2_enc_sat(c0, c1);
        }
        *reinterpret_cast<uint2 *>(m1 + i) = make_uint2(0u, 0u);
        *reinterpret_cast<uint4 *>(m2 + i) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(w16 + i) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
    }
}

}  // namespace

template <int FMT, int MODE>
cudaError_t launch_dq(int64_t grid, const uint8_t *parts, int nranks, int64_t n,
                      const float *scale, uint16_t *o, cudaStream_t st) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(dequant_sum_kernel<FMT, MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kDqSmem));
    });
    if (attr != cudaSuccess) return attr;
    return launch_pdl(dequant_sum_kernel<FMT, MODE>, dim3(static_cast<unsigned>(grid)),
                      dim3(kDqConsumers + 32), kDqSmem, st, parts, nranks, n, scale, o);
}

cudaError_t launch_dequant_sum(const uint8_t *parts, int nranks, int64_t n, int fmt,
                               const float *scale, void *out, int sm_count, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int64_t nchunks = (n + kDqChunk - 1) / kDqChunk;
    const int64_t cap = static_cast<int64_t>(sm_count) * 2;   // two blocks per SM
    const int64_t grid = nchunks < cap ? nchunks : cap;
    auto *o = static_cast<uint16_t *>(out);
    // up to 8 ranks one stage holds them all; up to 256 the exact count of
    // quanta stays below 2^40 (E5M2: 256 * 57344 * 2^16), so its product with
    // a 24-bit significand fits 64 bits
    const int mode = nranks <= kDqGroup ? 0 : (nranks <= 256 ? 1 : 2);
    if (fmt == 0) {
        if (mode == 0) return launch_dq<0, 0>(grid, parts, nranks, n, scale, o, st);
        if (mode == 1) return launch_dq<0, 1>(grid, parts, nranks, n, scale, o, st);
        return launch_dq<0, 2>(grid, parts, nranks, n, scale, o, st);
    }
    if (mode == 0) return launch_dq<1, 0>(grid, parts, nranks, n, scale, o, st);
    if (mode == 1) return launch_dq<1, 1>(grid, parts, nranks, n, scale, o, st);
    return launch_dq<1, 2>(grid, parts, nranks, n, scale, o, st);
}

cudaError_t read_and_clear_sum_error_flag(unsigned *flags) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_sum_error_flags, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_sum_error_flags, &zero, sizeof(unsigned));
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
