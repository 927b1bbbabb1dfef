// cast.cu -- the HBM-bound kernels of the FP8 delayed-scaling layer:
//  * amax of a BF16 tensor (range monitoring of dynamic scaling, "NVIDIA
//    Transformer Engine and FP8 mixed precision: implementation guide",
//    section "What are Transformer Engine and FP8 mixed precision"; the
//    Absolute-Max statistic of "FP8 quantization with NVIDIA TensorRT");
//  * the fused scaled cast BF16 -> FP8 (E4M3 / E5M2) with transposed copy and
//    amax (the Q node of the TensorRT page);
//  * the delayed-scaling history / scale update (DelayedScaling's margin and
//    amax_history_len, implementation guide section "Dynamic scaling and the
//    FP8 recipe");
//  * just-in-time scaling: the cast deriving its scale from the amax of the
//    same step ("Mixed-precision training" wiki note, bullet "per-tensor
//    scaling is the key");
//  * LayerNorm row statistics and the LayerNorm branch of the cast
//    (te.LayerNorm ahead of an FP8 linear, implementation guide section
//    "Basic structure of FP8 training code");
//  * the scaled cast of fp32 tensors (no transposed copy).
#include <cfloat>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

// Set when a cast kernel gives up a bounded wait (read by fp8_sync_status).
__device__ unsigned g_cast_error_flags = 0;

// ------------------------------------------------------------------- amax --

// Grid-stride max of |x| over 16-byte vectors (8 BF16), 4 vectors in flight
// per thread, packed BF16 abs / max (NaN skipped), one atomicMax per block.
// STREAM: evict-first loads, for a tensor larger than L2; a tensor that fits
// is read with plain loads and stays in L2 for the cast that follows (the
// just-in-time cast of a 67 MB tensor: 37.9 -> 35.8 us; evict-first loads
// are 2 % faster on a 537 MB one).
template <bool STREAM>
__device__ __forceinline__ uint4 amax_load(const uint4 *p) {
    if constexpr (STREAM)
        return __ldcs(p);
    else
        return *p;
}

template <bool STREAM>
__global__ void __launch_bounds__(512) amax_kernel(const uint4 *__restrict__ x, int64_t nvec,
                                                   unsigned *__restrict__ amax_bits) {
    pdl_wait();
    pdl_trigger();
    uint32_t m2 = 0;   // two BF16 magnitude maxima
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = amax_load<STREAM>(x + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            m2 = absmax_bf16x2(m2, v[u].x);
            m2 = absmax_bf16x2(m2, v[u].y);
            m2 = absmax_bf16x2(m2, v[u].z);
            m2 = absmax_bf16x2(m2, v[u].w);
        }
    }
    for (; i < nvec; i += stride) {
        uint4 v = amax_load<STREAM>(x + i);
        m2 = absmax_bf16x2(m2, v.x);
        m2 = absmax_bf16x2(m2, v.y);
        m2 = absmax_bf16x2(m2, v.z);
        m2 = absmax_bf16x2(m2, v.w);
    }
    uint32_t m = absmax_bf16x2_finish(m2);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ uint32_t warp_max[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_max[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < static_cast<int>(blockDim.x >> 5) ? warp_max[lane] : 0u;
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0 && m != 0) atomicMax(amax_bits, m << 16);
    }
}

// ------------------------------------------------------ fp32 scaled cast --

// q_i = satRNE(fl32(x_i * s)) of an fp32 tensor, element order kept, with
// amax(x) fused (NaN skipped, integer max on magnitude bits).  Grid-stride,
// eight values per thread and iteration: two 16-byte streaming loads and one
// 8-byte store.
template <int FMT>
__global__ void __launch_bounds__(256)
    quantize_f32_kernel(const float4 *__restrict__ x, int64_t n8, const float *__restrict__ scale,
                        uint2 *__restrict__ out, unsigned *__restrict__ amax_bits) {
    pdl_wait();
    pdl_trigger();
    const float s = *scale;
    uint32_t m = 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += stride) {
        const float4 a = __ldcs(x + 2 * i), b = __ldcs(x + 2 * i + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t u = __float_as_uint(v[j]) & 0x7FFFFFFFu;
            m = max(m, u > 0x7F800000u ? 0u : u);
        }
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = cvt2_fp8<FMT>(__fmul_rn(v[2 * j], s), __fmul_rn(v[2 * j + 1], s));
        __stcs(out + i, make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16)));
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ uint32_t warp_max[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_max[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < static_cast<int>(blockDim.x >> 5) ? warp_max[lane] : 0u;
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0 && m != 0 && amax_bits != nullptr) atomicMax(amax_bits, m);
    }
}

// ----------------------------------------------------- quantize_transpose --
//
// Persistent CTAs of 256 threads (two per SM) convert 128 x 128 tiles.  The
// BF16 input reaches shared memory through a 2-stage TMA ring, so the load of
// the next tile is in flight while the current one is converted:
//  phase 1  each thread takes 8 x 16 B of BF16 from the staged tile, scales,
//           converts to FP8, stores 8 B to the row-major output and the same
//           8 B into a tile of 32-bit words [128 rows][32 words] whose word
//           column is XOR-swizzled with the row's 16-row block, so that the
//           phase 2 reads are bank-conflict free;
//  phase 2  each thread owns 16 rows x 4 columns: it reads 16 words, turns
//           four 4 x 4 byte blocks around with byte permutes and writes four
//           16-byte runs of the transposed output; the 8 threads sharing a
//           column write one contiguous 128-byte line.
// The staged tile is released (and the TMA load of a later tile issued) as
// soon as phase 1 is done with it.  Consecutive tiles use alternate word
// tiles, so one barrier per tile suffices: a thread starting phase 1 of tile
// t+1 has passed the barrier after phase 1 of tile t, which every thread
// reached only after finishing phase 2 of tile t-1, the last reader of that
// word tile.  Waits are bounded.

constexpr int kQtTile = 128;
constexpr int kQtThreads = 256;
constexpr int kQtStages = 2;
constexpr int kQtStageBytes = kQtTile * kQtTile * 2;
constexpr size_t kQtSmem = 128 + kQtStages * kQtStageBytes + 2 * kQtTile * kQtTile + 64;

__device__ __forceinline__ int qt_swz(int row) { return ((row >> 4) & 7) << 2; }

// Transpose a 4 x 4 block of bytes held as 4 words (w[i] = row i, byte j =
// column j) into t[j] = column j (byte i = row i).
__device__ __forceinline__ void transpose4x4(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                             uint32_t &t0, uint32_t &t1, uint32_t &t2,
                                             uint32_t &t3) {
    const uint32_t a01 = __byte_perm(w0, w1, 0x5140);  // w0.b0 w1.b0 w0.b1 w1.b1
    const uint32_t b01 = __byte_perm(w0, w1, 0x7362);  // w0.b2 w1.b2 w0.b3 w1.b3
    const uint32_t a23 = __byte_perm(w2, w3, 0x5140);
    const uint32_t b23 = __byte_perm(w2, w3, 0x7362);
    t0 = __byte_perm(a01, a23, 0x5410);
    t1 = __byte_perm(a01, a23, 0x7632);
    t2 = __byte_perm(b01, b23, 0x5410);
    t3 = __byte_perm(b01, b23, 0x7632);
}

// One tensor of a cast launch (a launch may carry two tensors of the same
// format, e.g. X and W of the forward pass, whose tiles form one list).
struct CastTensor {
    int64_t rows, cols, tiles_c, tile_begin;
    float *scale;            // read; in just-in-time mode also written
    float *scale_inv;        // written in just-in-time mode
    const float *amax_in;    // just-in-time mode: this tensor's amax
    uint8_t *out, *out_t;    // row-major and transposed FP8 outputs (either may be null)
    unsigned *amax_bits;     // fused amax output (max-combined), or null
    // LayerNorm in front of the cast (null = plain cast): per-row mean and
    // rstd (fp32), per-column gamma and beta (BF16).  The cast then takes
    // y = ((x - mean) * rstd) * gamma + beta, and the amax is of y.
    const float *ln_mean, *ln_rstd;
    const uint16_t *ln_gamma, *ln_beta;
};

struct CastArgs {
    CUtensorMap maps[2];
    CastTensor t[2];
    int num_tensors;
    int margin;
    int64_t num_tiles;
};

// CURRENT = just-in-time scaling: each tensor's scale is derived here from
// its amax (computed by amax_kernel just before) instead of being read as
// given; block 0 also writes it and its inverse back.
template <int FMT, bool CURRENT>
__global__ void __launch_bounds__(kQtThreads, 2)
    quantize_transpose_kernel(const __grid_constant__ CastArgs a) {
    extern __shared__ uint8_t qt_smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(qt_smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    uint8_t *stage_base = base;
    uint32_t *tile0 = reinterpret_cast<uint32_t *>(base + kQtStages * kQtStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(base + kQtStages * kQtStageBytes +
                                                  2 * kQtTile * kQtTile);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + kQtStages);

    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int st = 0; st < kQtStages; ++st) mbar_init(smem_u32(full + st), 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int i = 0; i < a.num_tensors; ++i)
            if (a.t[i].rows > 0 && a.t[i].cols > 0) prefetch_tmap(&a.maps[i]);
    }
    pdl_wait();
    pdl_trigger();
    float sc[2];
    uint32_t tmax[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        sc[i] = i < a.num_tensors ? *a.t[i].scale : 0.0f;
        if constexpr (CURRENT) {
            if (i < a.num_tensors) {
                bool valid;
                sc[i] = recipe_scale(*a.t[i].amax_in, FMT == 0 ? 448.0f : 57344.0f, a.margin,
                                     sc[i], valid);
                if (valid && blockIdx.x == 0 && tid == 0) {
                    *a.t[i].scale = sc[i];
                    *a.t[i].scale_inv = __fdiv_rn(1.0f, sc[i]);
                }
            }
        }
    }
    // thread 0's count of loads issued into / consumed from each stage
    int issued[kQtStages] = {}, consumed[kQtStages] = {};

    auto issue = [&](int st, int64_t t) {
        const int p = (a.num_tensors > 1 && t >= a.t[1].tile_begin) ? 1 : 0;
        const int64_t lt = t - a.t[p].tile_begin;
        ++issued[st];
        mbar_arrive_expect_tx(smem_u32(full + st), kQtStageBytes);
        tma_load_2d(smem_u32(stage_base + st * kQtStageBytes), &a.maps[p], smem_u32(full + st),
                    static_cast<int32_t>((lt % a.t[p].tiles_c) * kQtTile),
                    static_cast<int32_t>((lt / a.t[p].tiles_c) * kQtTile));
    };

    if (tid == 0) {
        for (int st = 0; st < kQtStages; ++st) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(st) * gridDim.x;
            if (t < a.num_tiles) issue(st, t);
        }
    }
    __syncthreads();

    int64_t it = 0;
    for (int64_t t = blockIdx.x; t < a.num_tiles; t += gridDim.x, ++it) {
        const int st = static_cast<int>(it % kQtStages);
        const uint32_t parity = static_cast<uint32_t>((it / kQtStages) & 1);
        const int p = (a.num_tensors > 1 && t >= a.t[1].tile_begin) ? 1 : 0;
        const CastTensor &T = a.t[p];
        const int64_t lt = t - T.tile_begin;
        const int64_t r0 = (lt / T.tiles_c) * kQtTile;
        const int64_t c0 = (lt % T.tiles_c) * kQtTile;
        const int64_t rows = T.rows, cols = T.cols;
        const float s = p ? sc[1] : sc[0];
        // LayerNorm parameters of this tile (independent of the staged x):
        // loaded before the wait so that their latency overlaps it
        const bool ln = T.ln_mean != nullptr;
        const int lvv = tid & 15;
        const int64_t lc = c0 + lvv * 8;
        uint4 lg4 = make_uint4(0, 0, 0, 0), lb4 = make_uint4(0, 0, 0, 0);
        float lmu[8], lrs[8];
        if (ln) {
            if (lc < cols) {
                lg4 = *reinterpret_cast<const uint4 *>(T.ln_gamma + lc);
                lb4 = *reinterpret_cast<const uint4 *>(T.ln_beta + lc);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t r = r0 + ((i * kQtThreads + tid) >> 4);
                lmu[i] = r < rows ? T.ln_mean[r] : 0.0f;
                lrs[i] = r < rows ? T.ln_rstd[r] : 0.0f;
            }
        }
        const bool ok = mbar_wait(smem_u32(full + st), parity, abort_flag);
        const uint16_t *xs = reinterpret_cast<const uint16_t *>(stage_base + st * kQtStageBytes);
        uint32_t *tile = tile0 + (it & 1) * (kQtTile * kQtTile / 4);   // word tile of this iteration
        if (ok) {
        if (tid == 0) ++consumed[st];

        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = i * kQtThreads + tid;
            v[i] = *reinterpret_cast<const uint4 *>(xs + (idx >> 4) * kQtTile + (idx & 15) * 8);
        }
        uint32_t m = 0;
        if (!ln) {
            // packed BF16 abs / max for the amax (NaN skipped), one packed
            // fp32 multiply per pair, two-lane FP8 converts: the conversion
            // is issue-bound enough that the instruction count matters
            const uint64_t s2 = splat_f32x2(s);
            uint32_t m2 = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int idx = i * kQtThreads + tid;
                const int rr = idx >> 4, vv = idx & 15;
                const int64_t r = r0 + rr, c = c0 + vv * 8;
                m2 = absmax_bf16x2(m2, v[i].x);
                m2 = absmax_bf16x2(m2, v[i].y);
                m2 = absmax_bf16x2(m2, v[i].z);
                m2 = absmax_bf16x2(m2, v[i].w);
                uint2 q;
                q.x = scale_fp8x2_bf16x2<FMT>(v[i].x, s2) | (scale_fp8x2_bf16x2<FMT>(v[i].y, s2) << 16);
                q.y = scale_fp8x2_bf16x2<FMT>(v[i].z, s2) | (scale_fp8x2_bf16x2<FMT>(v[i].w, s2) << 16);
                if (T.out != nullptr && r < rows && c < cols)
                    *reinterpret_cast<uint2 *>(T.out + r * cols + c) = q;
                *reinterpret_cast<uint2 *>(&tile[rr * 32 + ((vv * 2) ^ qt_swz(rr))]) = q;
            }
            m = absmax_bf16x2_finish(m2) << 16;   // BF16 magnitude bits -> fp32 bits
        } else {
            // LayerNorm first: y = ((x - mean) * rstd) * gamma + beta in fp32,
            // one rounding per operation in that order: the subtract and the
            // add of beta in the mixed-precision scalar forms (x and beta stay
            // BF16), the two multiplies two lanes at a time.
            // This thread's 8 columns are the same for all 8 of its vectors.
            const int vv = lvv;
            const int64_t c = lc;
            uint64_t gam2[4];
            const uint32_t bw[4] = {lb4.x, lb4.y, lb4.z, lb4.w};
            {
                const uint32_t gw[4] = {lg4.x, lg4.y, lg4.z, lg4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) gam2[j] = f32x2_from_bf16x2(gw[j]);
            }
            const uint64_t s2 = splat_f32x2(s);
            float ymax = 0.0f;   // max |y| over in-range elements; fmaxf skips NaN
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rr = (i * kQtThreads + tid) >> 4;
                const int64_t r = r0 + rr;
                const bool in = r < rows && c < cols;
                const float mu = in ? lmu[i] : 0.0f;
                const uint64_t rs2 = splat_f32x2(in ? lrs[i] : 0.0f);
                const uint32_t xw[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t qw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float p0, p1, q0, q1;
                    const float d0 = bf16lo_sub_f32(xw[j], mu), d1 = bf16hi_sub_f32(xw[j], mu);
                    f32x2_unpack(f32x2_mul(f32x2_mul(f32x2_pack(d0, d1), rs2), gam2[j]), p0, p1);
                    const float y0 = bf16lo_add_f32(bw[j], p0);
                    const float y1 = bf16hi_add_f32(bw[j], p1);
                    const uint64_t y2 = f32x2_pack(y0, y1);
                    if (in) ymax = fmaxf(ymax, fmaxf(fabsf(y0), fabsf(y1)));
                    f32x2_unpack(f32x2_mul(y2, s2), q0, q1);
                    qw[j] = cvt2_fp8<FMT>(q0, q1);
                }
                uint2 q;
                q.x = qw[0] | (qw[1] << 16);
                q.y = qw[2] | (qw[3] << 16);
                if (T.out != nullptr && in) *reinterpret_cast<uint2 *>(T.out + r * cols + c) = q;
                *reinterpret_cast<uint2 *>(&tile[rr * 32 + ((vv * 2) ^ qt_swz(rr))]) = q;
            }
            m = __float_as_uint(ymax);   // fp32 bits of a value >= 0
        }
        if (p)
            tmax[1] = max(tmax[1], m);
        else
            tmax[0] = max(tmax[0], m);
        }
        // stage st fully read and this word tile complete; a thread whose
        // wait gave up skipped phase 1 and makes every thread leave together
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(&g_cast_error_flags, kErrWaitTimeout);
                *abort_flag = 1;
            }
            break;
        }

        if (tid == 0) {
            const int64_t tn = t + static_cast<int64_t>(kQtStages) * gridDim.x;
            if (tn < a.num_tiles) issue(st, tn);
        }

        if (T.out_t != nullptr) {
            const int lane = tid & 31, warp = tid >> 5;
            const int rblk = lane & 7;              // 16-row block of the tile
            const int cw = warp * 4 + (lane >> 3);  // word column = 4 tile columns
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int rr = rblk * 16 + j;
                w[j] = tile[rr * 32 + (cw ^ qt_swz(rr))];
            }
            uint32_t o[4][4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
                transpose4x4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3], o[0][g], o[1][g],
                             o[2][g], o[3][g]);
            const int64_t r = r0 + rblk * 16;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int64_t c = c0 + cw * 4 + cc;
                if (r < rows && c < cols)
                    *reinterpret_cast<uint4 *>(T.out_t + c * rows + r) =
                        make_uint4(o[cc][0], o[cc][1], o[cc][2], o[cc][3]);
            }
        }
    }

    // Loads still in flight (only after an abandoned wait) must land before exit.
    if (tid == 0 && *abort_flag) {
        for (int st = 0; st < kQtStages; ++st)
            if (issued[st] > consumed[st])
                mbar_wait(smem_u32(full + st), static_cast<uint32_t>((issued[st] - 1) & 1),
                          nullptr, 100000000ull);
    }

    __shared__ uint32_t warp_max[2][kQtThreads / 32];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, tmax[i]);
        if ((tid & 31) == 0) warp_max[i][tid >> 5] = m;
    }
    __syncthreads();
    if (tid < 32) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint32_t m = tid < kQtThreads / 32 ? warp_max[i][tid] : 0u;
            m = __reduce_max_sync(0xFFFFFFFFu, m);
            if (tid == 0 && m != 0 && i < a.num_tensors && a.t[i].amax_bits != nullptr)
                atomicMax(a.t[i].amax_bits, m);   // fp32 bits of a value >= 0
        }
    }
}

// ------------------------------------------------------- FP8 transpose --
//
// out_t[c][r] = in[r][c] for a [rows][cols] array of bytes (FP8 codes), in
// 128 x 128 tiles, with the word tile and the second phase of
// quantize_transpose_kernel: each thread loads 8 x 8 bytes of the tile
// (16 threads cover a 128-byte row segment), stores them into the
// XOR-swizzled word tile, and after a barrier turns 4 x 4 byte blocks around
// and writes four 16-byte runs of the transposed output.  The LayerNorm cast
// uses it to transpose the row-major codes it has just written (still in L2)
// instead of reading x a second time.

__global__ void __launch_bounds__(kQtThreads) transpose_u8_kernel(const uint8_t *__restrict__ in,
                                                                 int64_t rows, int64_t cols,
                                                                 int64_t tiles_c, int64_t num_tiles,
                                                                 uint8_t *__restrict__ out_t) {
    __shared__ uint32_t tile[kQtTile * kQtTile / 4];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x;
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        const int64_t r0 = (t / tiles_c) * kQtTile, c0 = (t % tiles_c) * kQtTile;
        uint2 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = i * kQtThreads + tid;
            const int64_t r = r0 + (idx >> 4), c = c0 + (idx & 15) * 8;
            v[i] = r < rows && c < cols ? *reinterpret_cast<const uint2 *>(in + r * cols + c)
                                        : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = i * kQtThreads + tid;
            const int rr = idx >> 4, vv = idx & 15;
            *reinterpret_cast<uint2 *>(&tile[rr * 32 + ((vv * 2) ^ qt_swz(rr))]) = v[i];
        }
        __syncthreads();
        const int lane = tid & 31, warp = tid >> 5;
        const int rblk = lane & 7;              // 16-row block of the tile
        const int cw = warp * 4 + (lane >> 3);  // word column = 4 tile columns
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int rr = rblk * 16 + j;
            w[j] = tile[rr * 32 + (cw ^ qt_swz(rr))];
        }
        uint32_t o[4][4];
#pragma unroll
        for (int g = 0; g < 4; ++g)
            transpose4x4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3], o[0][g], o[1][g],
                         o[2][g], o[3][g]);
        const int64_t r = r0 + rblk * 16;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int64_t c = c0 + cw * 4 + cc;
            if (r < rows && c < cols)
                *reinterpret_cast<uint4 *>(out_t + c * rows + r) =
                    make_uint4(o[cc][0], o[cc][1], o[cc][2], o[cc][3]);
        }
        __syncthreads();   // the word tile is refilled by the next tile
    }
}

// ------------------------------------------------------ LayerNorm row stats --
//
// One warp per row (grid-stride over rows): mean = sum(x) / C, then
// var = sum((x - mean)^2) / C over a second read of the row (from L1 / L2),
// rstd = 1 / sqrt(var + eps), all in fp32 with correctly rounded operations;
// each squared deviation is accumulated with one fused multiply-add.
// With amax_bits, a third read computes y = ((x - mean) * rstd) * gamma + beta
// and max-combines max |y| (for just-in-time scaling of the LayerNorm output).

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    return v;
}

__global__ void __launch_bounds__(256) ln_stats_kernel(const uint16_t *__restrict__ x,
                                                       const uint16_t *__restrict__ gamma,
                                                       const uint16_t *__restrict__ beta,
                                                       int64_t rows, int64_t cols, float eps,
                                                       float *__restrict__ mean,
                                                       float *__restrict__ rstd,
                                                       unsigned *__restrict__ amax_bits) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t nvec = cols / 8;
    const float inv_c = __fdiv_rn(1.0f, static_cast<float>(cols));
    uint32_t m = 0;
    for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < rows;
         r += warps) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + r * cols);
        // four 16-byte loads in flight per lane, eight independent partial
        // sums per lane (one per element position of a 16-byte vector)
        float part[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int64_t i = lane; i < nvec; i += 128) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = i + 32 * u < nvec ? xr[i + 32 * u] : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    part[2 * j] = __fadd_rn(part[2 * j], bf16_lo(w[j]));
                    part[2 * j + 1] = __fadd_rn(part[2 * j + 1], bf16_hi(w[j]));
                }
            }
        }
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) sum = __fadd_rn(sum, part[j]);
        const float mu = __fmul_rn(warp_sum(sum), inv_c);
#pragma unroll
        for (int j = 0; j < 8; ++j) part[j] = 0.0f;
        for (int64_t i = lane; i < nvec; i += 128) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = i + 32 * u < nvec ? xr[i + 32 * u] : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (i + 32 * u >= nvec) break;
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float d0 = __fsub_rn(bf16_lo(w[j]), mu);
                    const float d1 = __fsub_rn(bf16_hi(w[j]), mu);
                    part[2 * j] = __fmaf_rn(d0, d0, part[2 * j]);
                    part[2 * j + 1] = __fmaf_rn(d1, d1, part[2 * j + 1]);
                }
            }
        }
        float sq = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) sq = __fadd_rn(sq, part[j]);
        const float var = __fmul_rn(warp_sum(sq), inv_c);
        const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
        if (lane == 0) {
            mean[r] = mu;
            rstd[r] = rs;
        }
        if (amax_bits != nullptr) {
            for (int64_t i = lane; i < nvec; i += 32) {
                const uint4 v = xr[i];
                const uint4 g4 = reinterpret_cast<const uint4 *>(gamma)[i];
                const uint4 b4 = reinterpret_cast<const uint4 *>(beta)[i];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g4.x, g4.y, g4.z, g4.w},
                               bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float y0 = __fadd_rn(
                        __fmul_rn(__fmul_rn(__fsub_rn(bf16_lo(w[j]), mu), rs), bf16_lo(gw[j])),
                        bf16_lo(bw[j]));
                    const float y1 = __fadd_rn(
                        __fmul_rn(__fmul_rn(__fsub_rn(bf16_hi(w[j]), mu), rs), bf16_hi(gw[j])),
                        bf16_hi(bw[j]));
                    const uint32_t a0 = __float_as_uint(y0) & 0x7FFFFFFFu;
                    const uint32_t a1 = __float_as_uint(y1) & 0x7FFFFFFFu;
                    m = max(m, a0 > 0x7F800000u ? 0u : a0);
                    m = max(m, a1 > 0x7F800000u ? 0u : a1);
                }
            }
        }
    }
    if (amax_bits != nullptr) {
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0 && m != 0) atomicMax(amax_bits, m);
    }
}

// The same statistics for rows of at most 8192 columns, each row staged in
// shared memory by an untiled bulk copy.  Each CTA owns a balanced
// contiguous range of rows, dealt to its warps in turn.  Every warp owns two
// row buffers: while it reduces one row its next row is already in flight,
// so the loads of all warps keep HBM busy through the reductions (a row read
// only into registers left the loads idle while each warp reduced).  The
// sum, the squared deviations and the optional amax(y) read the staged row;
// each lane visits its vectors in the same order as ln_stats_kernel, so the
// fp32 results are the same bit for bit.  Waits are bounded.
constexpr int kLnBufs = 2;

__global__ void __launch_bounds__(512) ln_stats_bulk_kernel(const uint16_t *__restrict__ x,
                                                            const uint16_t *__restrict__ gamma,
                                                            const uint16_t *__restrict__ beta,
                                                            int64_t rows, int64_t cols, float eps,
                                                            float *__restrict__ mean,
                                                            float *__restrict__ rstd,
                                                            unsigned *__restrict__ amax_bits) {
    extern __shared__ uint8_t ln_smem_raw[];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int nw = static_cast<int>(blockDim.x >> 5);
    const uint32_t row_bytes = static_cast<uint32_t>(cols) * 2u;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ln_smem_raw);            // [nw][kLnBufs]
    uint8_t *bufs = ln_smem_raw + 16 * nw * kLnBufs;                       // 128-byte aligned below
    bufs = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(bufs) + 127) &
                                       ~static_cast<uintptr_t>(127));
    uint8_t *mybuf = bufs + static_cast<size_t>(wib) * kLnBufs * row_bytes;
    const uint32_t bar0 = smem_u32(bars + wib * kLnBufs);
    if (lane == 0) {
        for (int b = 0; b < kLnBufs; ++b) mbar_init(bar0 + 8 * b, 1);
        fence_mbar_init();
    }
    __syncwarp();
    pdl_wait();
    pdl_trigger();
    // this CTA's rows: a balanced contiguous range, dealt to its warps in turn
    // (a grid-wide deal would give some SMs a whole extra round of rows)
    const int64_t rend = rows * (blockIdx.x + 1) / gridDim.x;
    const int64_t first = rows * blockIdx.x / gridDim.x + wib;
    const int64_t warps = nw;
    const int nvec = static_cast<int>(cols / 8);
    const float inv_c = __fdiv_rn(1.0f, static_cast<float>(cols));
    int issued[kLnBufs] = {}, consumed[kLnBufs] = {};   // lane 0's counts
    auto issue = [&](int b, int64_t r) {
        ++issued[b];
        mbar_arrive_expect_tx(bar0 + 8 * b, row_bytes);
        bulk_load_1d(smem_u32(mybuf + b * row_bytes), x + r * cols, row_bytes, bar0 + 8 * b);
    };
    if (lane == 0)
        for (int b = 0; b < kLnBufs; ++b)
            if (first + b * warps < rend) issue(b, first + b * warps);
    uint32_t m = 0;
    bool failed = false;
    int64_t j = 0;
    for (int64_t r = first; r < rend; r += warps, ++j) {
        const int b = static_cast<int>(j % kLnBufs);
        const uint32_t parity = static_cast<uint32_t>((j / kLnBufs) & 1);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar0 + 8 * b, parity, nullptr))) {
            failed = true;
            break;
        }
        if (lane == 0) ++consumed[b];
        const uint4 *xr = reinterpret_cast<const uint4 *>(mybuf + b * row_bytes);
        // the sum: eight partial sums per lane (one per element position of
        // a 16-byte vector), vectors lane, lane + 32, ...; each one IEEE add
        // of the widened BF16 (the mixed-precision form)
        float part[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        for (int i = lane; i < nvec; i += 32) {
            const uint4 v = xr[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                part[2 * q] = bf16lo_add_f32(w[q], part[2 * q]);
                part[2 * q + 1] = bf16hi_add_f32(w[q], part[2 * q + 1]);
            }
        }
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) sum = __fadd_rn(sum, part[q]);
        const float mu = __fmul_rn(warp_sum(sum), inv_c);
        // the squared deviations, each accumulated with one fused
        // multiply-add (d * d + part, rounded once)
#pragma unroll
        for (int q = 0; q < 8; ++q) part[q] = 0.0f;
        for (int i = lane; i < nvec; i += 32) {
            const uint4 v = xr[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float d0 = bf16lo_sub_f32(w[q], mu), d1 = bf16hi_sub_f32(w[q], mu);
                part[2 * q] = __fmaf_rn(d0, d0, part[2 * q]);
                part[2 * q + 1] = __fmaf_rn(d1, d1, part[2 * q + 1]);
            }
        }
        float sq = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) sq = __fadd_rn(sq, part[q]);
        const float var = __fmul_rn(warp_sum(sq), inv_c);
        const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
        if (lane == 0) {
            mean[r] = mu;
            rstd[r] = rs;
        }
        if (amax_bits != nullptr) {
            for (int i = lane; i < nvec; i += 32) {
                const uint4 v = xr[i];
                const uint4 g4 = reinterpret_cast<const uint4 *>(gamma)[i];
                const uint4 b4 = reinterpret_cast<const uint4 *>(beta)[i];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g4.x, g4.y, g4.z, g4.w},
                               bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float y0 = __fadd_rn(
                        __fmul_rn(__fmul_rn(__fsub_rn(bf16_lo(w[q]), mu), rs), bf16_lo(gw[q])),
                        bf16_lo(bw[q]));
                    const float y1 = __fadd_rn(
                        __fmul_rn(__fmul_rn(__fsub_rn(bf16_hi(w[q]), mu), rs), bf16_hi(gw[q])),
                        bf16_hi(bw[q]));
                    const uint32_t a0 = __float_as_uint(y0) & 0x7FFFFFFFu;
                    const uint32_t a1 = __float_as_uint(y1) & 0x7FFFFFFFu;
                    m = max(m, a0 > 0x7F800000u ? 0u : a0);
                    m = max(m, a1 > 0x7F800000u ? 0u : a1);
                }
            }
        }
        // every lane is done with this buffer: refill it with a later row
        __syncwarp();
        if (lane == 0 && r + kLnBufs * warps < rend) issue(b, r + kLnBufs * warps);
    }
    if (failed) {
        // a wait gave up: record it, and let this warp's copies still in
        // flight land (bounded) before the CTA may exit
        if (lane == 0) {
            atomicOr(&g_cast_error_flags, kErrWaitTimeout);
            for (int b = 0; b < kLnBufs; ++b)
                if (issued[b] > consumed[b])
                    mbar_wait(bar0 + 8 * b, static_cast<uint32_t>((issued[b] - 1) & 1), nullptr,
                              100000000ull);
        }
        __syncwarp();
    }
    if (amax_bits != nullptr) {
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0 && m != 0) atomicMax(amax_bits, m);
    }
}

// ------------------------------------ LayerNorm + row-major cast, one pass --
//
// Delayed scaling knows the scale before the cast, so the statistics, the
// normalisation and the row-major cast can share one read of x (rows of at
// most 4096 columns).  The same kernel computes the statistics alone (and
// max |y| for just-in-time scaling), for fp8_layernorm_stats and ahead of
// the two-kernel cast of such rows.  Each CTA owns a balanced, contiguous
// range of rows and has 16 warps; warp w takes rows w, w + 16, ... of the
// range.  Every warp owns one row buffer: it
// copies its row from the buffer into registers (16 vectors of 8 BF16 per
// lane at most), at once starts the untiled bulk copy of its next row into
// the same buffer, and works on the registers meanwhile.  From them it
// computes mean and rstd with the same operations in the same order as
// ln_stats_bulk_kernel (the results are identical bit for bit), then
// y = ((x - mean) * rstd) * gamma + beta and its cast exactly as the
// LayerNorm branch of quantize_transpose_kernel (gamma and beta staged in
// shared memory once per CTA), and writes the codes; a transposed copy, when
// wanted, is a byte transpose of those codes afterwards.  The two statistics
// passes, the subtract of the mean and the add of beta use the
// mixed-precision BF16 + fp32 forms, which round exactly as widening first
// does.  Waits are bounded.

constexpr int kLnfWarps = 16;
constexpr int kLnfThreads = kLnfWarps * 32;
constexpr int kLnfMaxCols = 4096;
constexpr int kLnfVecs = kLnfMaxCols / 256;         // 16-byte vectors per lane

// MODE kLnfStats: mean and rstd only; kLnfStatsAmax: and max |y|; kLnfCast:
// and the codes of y (out) with max |y|.
constexpr int kLnfStats = 0, kLnfStatsAmax = 1, kLnfCast = 2;

template <int FMT, int MODE>
__global__ void __launch_bounds__(kLnfThreads, 1)
    ln_cast_rows_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ gamma,
                        const uint16_t *__restrict__ beta, int64_t rows, int cols, float eps,
                        const float *__restrict__ scale, float *__restrict__ mean,
                        float *__restrict__ rstd, uint8_t *__restrict__ out,
                        unsigned *__restrict__ amax_bits) {
    extern __shared__ uint8_t lnf_smem_raw[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(lnf_smem_raw);   // one per warp
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + kLnfWarps);
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(bars + kLnfWarps + 1) + 127) & ~static_cast<uintptr_t>(127));
    const uint32_t row_bytes = static_cast<uint32_t>(cols) * 2u;
    uint16_t *gb_s = reinterpret_cast<uint16_t *>(ring + static_cast<size_t>(kLnfWarps) * row_bytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar = smem_u32(bars + warp);
    uint8_t *mybuf = ring + static_cast<size_t>(warp) * row_bytes;
    const int64_t rbeg = rows * blockIdx.x / gridDim.x;
    const int nrows = static_cast<int>(rows * (blockIdx.x + 1) / gridDim.x - rbeg);
    if (lane == 0) mbar_init(bar, 1);
    if (tid == 0) *abort_flag = 0;
    fence_mbar_init();
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    // this warp's first row in flight, then gamma and beta into shared memory
    int issued = 0, consumed = 0;   // lane 0's copies into this warp's buffer
    if (lane == 0 && warp < nrows) {
        mbar_arrive_expect_tx(bar, row_bytes);
        bulk_load_1d(smem_u32(mybuf), x + (rbeg + warp) * cols, row_bytes, bar);
        ++issued;
    }
    const int nvec = cols / 8;
    if constexpr (MODE != kLnfStats) {
        for (int i = tid; i < nvec; i += kLnfThreads) {
            reinterpret_cast<uint4 *>(gb_s)[i] = reinterpret_cast<const uint4 *>(gamma)[i];
            reinterpret_cast<uint4 *>(gb_s + cols)[i] = reinterpret_cast<const uint4 *>(beta)[i];
        }
    }
    __syncthreads();

    const float inv_c = __fdiv_rn(1.0f, static_cast<float>(cols));
    const uint64_t s2 = splat_f32x2(MODE == kLnfCast ? *scale : 1.0f);
    float ymax = 0.0f;   // max |y|; fmaxf skips NaN
    int use = 0;         // this warp's rows so far (the parity of its buffer)
    for (int j = warp; j < nrows; j += kLnfWarps, ++use) {
        const int64_t r = rbeg + j;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar, static_cast<uint32_t>(use & 1), abort_flag))) {
            if (lane == 0) {
                atomicOr(&g_cast_error_flags, kErrWaitTimeout);
                *abort_flag = 1;
            }
            break;
        }
        if (lane == 0) ++consumed;
        uint4 v[kLnfVecs];
        const uint4 *xr = reinterpret_cast<const uint4 *>(mybuf);
#pragma unroll
        for (int t = 0; t < kLnfVecs; ++t) {
            const int i = lane + 32 * t;
            v[t] = i < nvec ? xr[i] : make_uint4(0u, 0u, 0u, 0u);
        }
        // the row is in registers: the buffer takes this warp's next row
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && j + kLnfWarps < nrows) {
            mbar_arrive_expect_tx(bar, row_bytes);
            bulk_load_1d(smem_u32(mybuf), x + (r + kLnfWarps) * cols, row_bytes, bar);
            ++issued;
        }
        // the sum: eight partial sums per lane over vectors lane, lane + 32, ...
        // (partial 2q + h takes the half h of word q)
        float part[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int t = 0; t < kLnfVecs; ++t) {
            if (lane + 32 * t >= nvec) break;
            const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                part[2 * q] = bf16lo_add_f32(w[q], part[2 * q]);
                part[2 * q + 1] = bf16hi_add_f32(w[q], part[2 * q + 1]);
            }
        }
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) sum = __fadd_rn(sum, part[q]);
        const float mu = __fmul_rn(warp_sum(sum), inv_c);
        // the squared deviations, one fused multiply-add each
#pragma unroll
        for (int q = 0; q < 8; ++q) part[q] = 0.0f;
#pragma unroll
        for (int t = 0; t < kLnfVecs; ++t) {
            if (lane + 32 * t >= nvec) break;
            const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float d0 = bf16lo_sub_f32(w[q], mu), d1 = bf16hi_sub_f32(w[q], mu);
                part[2 * q] = __fmaf_rn(d0, d0, part[2 * q]);
                part[2 * q + 1] = __fmaf_rn(d1, d1, part[2 * q + 1]);
            }
        }
        float sq = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) sq = __fadd_rn(sq, part[q]);
        const float var = __fmul_rn(warp_sum(sq), inv_c);
        const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
        if (lane == 0) {
            mean[r] = mu;
            rstd[r] = rs;
        }
        if constexpr (MODE == kLnfStats) continue;
        // y and its codes: the subtract of the mean and the add of beta in
        // the mixed-precision scalar forms (x and beta stay BF16), both
        // multiplies two lanes at a time
        const uint64_t rs2 = splat_f32x2(rs);
#pragma unroll
        for (int t = 0; t < kLnfVecs; ++t) {
            const int i = lane + 32 * t;
            if (i >= nvec) break;
            const uint4 g4 = reinterpret_cast<const uint4 *>(gb_s)[i];
            const uint4 b4 = reinterpret_cast<const uint4 *>(gb_s + cols)[i];
            const uint32_t xw[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
            const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w}, bw[4] = {b4.x, b4.y, b4.z, b4.w};
            uint32_t qw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float p0, p1, c0, c1;
                const float d0 = bf16lo_sub_f32(xw[q], mu), d1 = bf16hi_sub_f32(xw[q], mu);
                f32x2_unpack(f32x2_mul(f32x2_mul(f32x2_pack(d0, d1), rs2),
                                       f32x2_from_bf16x2(gw[q])),
                             p0, p1);
                const float y0 = bf16lo_add_f32(bw[q], p0);
                const float y1 = bf16hi_add_f32(bw[q], p1);
                ymax = fmaxf(ymax, fmaxf(fabsf(y0), fabsf(y1)));
                if constexpr (MODE == kLnfCast) {
                    f32x2_unpack(f32x2_mul(f32x2_pack(y0, y1), s2), c0, c1);
                    qw[q] = cvt2_fp8<FMT>(c0, c1);
                }
            }
            if constexpr (MODE == kLnfCast)
                *reinterpret_cast<uint2 *>(out + r * cols + 8 * i) =
                    make_uint2(qw[0] | (qw[1] << 16), qw[2] | (qw[3] << 16));
        }
    }
    // a copy still in flight (only after a wait gave up) lands before exit
    if (lane == 0 && issued > consumed)
        mbar_wait(bar, static_cast<uint32_t>((issued - 1) & 1), nullptr, 100000000ull);
    // max |y| over the CTA
    __shared__ uint32_t warp_max[kLnfWarps];
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(ymax));
    if (lane == 0) warp_max[warp] = m;
    __syncthreads();
    if (tid < 32) {
        uint32_t mm = tid < kLnfWarps ? warp_max[tid] : 0u;
        mm = __reduce_max_sync(0xFFFFFFFFu, mm);
        if (tid == 0 && mm != 0 && amax_bits != nullptr) atomicMax(amax_bits, mm);
    }
}

// Warps per block and dynamic shared memory of ln_stats_bulk_kernel for
// rows of `cols` columns: two row buffers per warp in at most ~200 KB.
inline int ln_bulk_warps(int64_t cols) {
    const int64_t per_warp = kLnBufs * cols * 2;
    int64_t w = (200 * 1024) / per_warp;
    if (w > 16) w = 16;
    return static_cast<int>(w);
}
inline size_t ln_bulk_smem(int warps, int64_t cols) {
    return static_cast<size_t>(16 * warps * kLnBufs + 128) +
           static_cast<size_t>(warps) * kLnBufs * static_cast<size_t>(cols) * 2;
}

// Dynamic shared memory of ln_cast_rows_kernel: barriers, one row buffer per
// warp, gamma and beta (BF16).
inline size_t lnf_smem(int cols) {
    return static_cast<size_t>(8 * kLnfWarps + 8 + 128) +
           static_cast<size_t>(kLnfWarps) * 2 * static_cast<size_t>(cols) +
           2 * 2 * static_cast<size_t>(cols);
}

bool ln_cast_rows_fits(int64_t rows, int64_t cols) {
    return rows >= 0 && cols % 16 == 0 && cols >= 16 && cols <= kLnfMaxCols;
}

template <int FMT, int MODE>
static cudaError_t lnf_launch(int64_t rows, int cols, int sm_count, cudaStream_t st,
                              const void *x, const void *g, const void *b, float eps,
                              const float *scale, float *mean, float *rstd, uint8_t *out,
                              float *amax) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(ln_cast_rows_kernel<FMT, MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    });
    if (attr != cudaSuccess) return attr;
    int64_t grid = (rows + kLnfWarps - 1) / kLnfWarps;
    if (grid > sm_count) grid = sm_count;
    return launch_pdl(ln_cast_rows_kernel<FMT, MODE>, dim3(static_cast<unsigned>(grid)),
                      dim3(kLnfThreads), lnf_smem(cols), st,
                      reinterpret_cast<const uint16_t *>(x), reinterpret_cast<const uint16_t *>(g),
                      reinterpret_cast<const uint16_t *>(b), rows, cols, eps, scale, mean, rstd,
                      out, reinterpret_cast<unsigned *>(amax));
}

cudaError_t launch_ln_stats(const void *x, const void *gamma, const void *beta, int64_t rows,
                            int64_t cols, float eps, float *mean, float *rstd, float *amax,
                            int sm_count, cudaStream_t st) {
    if (amax != nullptr) {
        cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
        if (e != cudaSuccess) return e;
    }
    if (rows == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (rows + 7) / 8;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    const int64_t nvec = cols / 8;
    const dim3 grid(static_cast<unsigned>(blocks)), block(threads);
    const uint16_t *xb = reinterpret_cast<const uint16_t *>(x);
    const uint16_t *gb = reinterpret_cast<const uint16_t *>(gamma);
    const uint16_t *bb = reinterpret_cast<const uint16_t *>(beta);
    unsigned *ab = reinterpret_cast<unsigned *>(amax);
    // rows of up to 4096 columns: held in registers, one HBM read of x
    if (ln_cast_rows_fits(rows, cols)) {
        const int c = static_cast<int>(cols);
        return amax != nullptr
                   ? lnf_launch<0, kLnfStatsAmax>(rows, c, sm_count, st, x, gamma, beta, eps,
                                                   nullptr, mean, rstd, nullptr, amax)
                   : lnf_launch<0, kLnfStats>(rows, c, sm_count, st, x, gamma, beta, eps, nullptr,
                                              mean, rstd, nullptr, nullptr);
    }
    // rows of up to 8192 columns: staged in shared memory, one HBM read of x
    if (nvec <= 1024) {
        const int warps = ln_bulk_warps(cols);
        const size_t smem = ln_bulk_smem(warps, cols);
        // at most 200 KB of row buffers plus the barriers (ln_bulk_warps)
        static std::once_flag once;
        static cudaError_t attr_err = cudaSuccess;
        std::call_once(once, [] {
            attr_err = cudaFuncSetAttribute(ln_stats_bulk_kernel,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            210 * 1024);
        });
        if (attr_err != cudaSuccess) return attr_err;
        int64_t bgrid = (rows + warps - 1) / warps;
        if (bgrid > sm_count) bgrid = sm_count;
        return launch_pdl(ln_stats_bulk_kernel, dim3(static_cast<unsigned>(bgrid)),
                          dim3(32 * warps), smem, st, xb, gb, bb, rows, cols, eps, mean, rstd, ab);
    }
    return launch_pdl(ln_stats_kernel, grid, block, 0, st,
                      reinterpret_cast<const uint16_t *>(x), reinterpret_cast<const uint16_t *>(gamma),
                      reinterpret_cast<const uint16_t *>(beta), rows, cols, eps, mean, rstd,
                      reinterpret_cast<unsigned *>(amax));
}

cudaError_t launch_ln_cast_rows(const void *x, const void *gamma, const void *beta, int64_t rows,
                                int64_t cols, float eps, const float *scale, int fmt,
                                uint8_t *out, float *amax, bool zero_amax, float *mean,
                                float *rstd, int sm_count, cudaStream_t st) {
    if (!ln_cast_rows_fits(rows, cols) || out == nullptr) return cudaErrorInvalidValue;
    if (amax != nullptr && zero_amax) {
        cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
        if (e != cudaSuccess) return e;
    }
    if (rows == 0) return cudaSuccess;
    const int c = static_cast<int>(cols);
    return fmt == 0 ? lnf_launch<0, kLnfCast>(rows, c, sm_count, st, x, gamma, beta, eps, scale,
                                              mean, rstd, out, amax)
                    : lnf_launch<1, kLnfCast>(rows, c, sm_count, st, x, gamma, beta, eps, scale,
                                              mean, rstd, out, amax);
}

cudaError_t launch_transpose_u8(const uint8_t *in, int64_t rows, int64_t cols, uint8_t *out_t,
                                int sm_count, cudaStream_t st) {
    if (rows % 16 != 0 || cols % 16 != 0) return cudaErrorInvalidValue;
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int64_t tiles_c = (cols + kQtTile - 1) / kQtTile;
    const int64_t num_tiles = ((rows + kQtTile - 1) / kQtTile) * tiles_c;
    int64_t grid = static_cast<int64_t>(sm_count) * 8;
    if (grid > num_tiles) grid = num_tiles;
    return launch_pdl(transpose_u8_kernel, dim3(static_cast<unsigned>(grid)), dim3(kQtThreads), 0,
                      st, in, rows, cols, tiles_c, num_tiles, out_t);
}

// ----------------------------------------------------------- scale update --
//
// One CTA per tensor: shift the history by one (newest at [0]), take its max,
// and recompute scale = fl32(fl32(fmax / m) * 2^-margin) (clamped to FLT_MAX)
// and scale_inv = fl32(1 / scale) when 0 < m < inf; otherwise keep both.

constexpr int kUpdThreads = 256;

__global__ void __launch_bounds__(kUpdThreads) scale_update_kernel(
    float *__restrict__ history, float *__restrict__ amax, float *__restrict__ scale,
    float *__restrict__ scale_inv, int L, uint32_t format_mask, int margin, int clear_amax) {
    extern __shared__ float old_hist[];
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    float *h = history + static_cast<int64_t>(t) * L;
    for (int i = threadIdx.x; i < L; i += blockDim.x) old_hist[i] = h[i];
    __syncthreads();
    const float a = amax[t];
    float m = 0.0f;
    for (int i = threadIdx.x; i < L; i += blockDim.x) {
        const float nv = i == 0 ? a : old_hist[i - 1];
        h[i] = nv;
        m = fmaxf(m, nv);
    }
    __shared__ float warp_max[kUpdThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kUpdThreads / 32; ++w) m = fmaxf(m, warp_max[w]);
        m = fmaxf(m, warp_max[0]);
        const float fmax = ((format_mask >> t) & 1u) ? 57344.0f : 448.0f;
        bool valid;
        const float sc = recipe_scale(m, fmax, margin, scale[t], valid);
        if (valid) {
            scale[t] = sc;
            scale_inv[t] = __fdiv_rn(1.0f, sc);
        }
        // the amax has been pushed into the history: start the next step at 0
        if (clear_amax) amax[t] = 0.0f;
    }
}

// ---------------------------------------------------------------- launchers --

cudaError_t launch_amax(const void *x, int64_t n, float *amax, int sm_count, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
    if (e != cudaSuccess || n == 0) return e;
    const int64_t nvec = n / 8;
    const int threads = 512;
    int64_t blocks = (nvec + threads * 4 - 1) / (threads * 4);
    const int64_t cap = static_cast<int64_t>(sm_count) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const dim3 grid(static_cast<unsigned>(blocks)), block(threads);
    const auto *xv = reinterpret_cast<const uint4 *>(x);
    auto *ab = reinterpret_cast<unsigned *>(amax);
    // tensors up to 96 MB (of the 129 MB L2) are left in L2 for a following cast
    return n * 2 <= (96ll << 20) ? launch_pdl(amax_kernel<false>, grid, block, 0, st, xv, nvec, ab)
                                 : launch_pdl(amax_kernel<true>, grid, block, 0, st, xv, nvec, ab);
}

cudaError_t launch_quantize_f32(const float *x, int64_t n, const float *scale, int fmt,
                                uint8_t *out, float *amax, int sm_count, cudaStream_t st) {
    if (amax != nullptr) {
        cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
        if (e != cudaSuccess) return e;
    }
    if (n == 0) return cudaSuccess;
    const int64_t n8 = n / 8;
    const int threads = 256;
    int64_t blocks = (n8 + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    const dim3 grid(static_cast<unsigned>(blocks)), block(threads);
    const float4 *xv = reinterpret_cast<const float4 *>(x);
    uint2 *ov = reinterpret_cast<uint2 *>(out);
    unsigned *ab = reinterpret_cast<unsigned *>(amax);
    return fmt == 0 ? launch_pdl(quantize_f32_kernel<0>, grid, block, 0, st, xv, n8, scale, ov, ab)
                    : launch_pdl(quantize_f32_kernel<1>, grid, block, 0, st, xv, n8, scale, ov, ab);
}

template <int FMT, bool CURRENT>
static cudaError_t qt_launch(const CastArgs &args, int sm_count, cudaStream_t st) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(quantize_transpose_kernel<FMT, CURRENT>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kQtSmem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (args.num_tiles == 0) return cudaSuccess;
    int64_t blocks = static_cast<int64_t>(sm_count) * 2;
    if (blocks > args.num_tiles) blocks = args.num_tiles;
    return launch_pdl(quantize_transpose_kernel<FMT, CURRENT>, dim3(static_cast<unsigned>(blocks)),
                      dim3(kQtThreads), kQtSmem, st, args);
}

// Fill the launch arguments for up to two tensors; false if a TMA
// descriptor cannot be built.
static bool cast_args(CastArgs &args, const CastSpec *specs, int n, int margin) {
    args.num_tensors = n;
    args.margin = margin;
    int64_t tiles = 0;
    for (int i = 0; i < n; ++i) {
        const CastSpec &c = specs[i];
        CastTensor &t = args.t[i];
        t.rows = c.rows;
        t.cols = c.cols;
        t.tiles_c = (c.cols + kQtTile - 1) / kQtTile;
        t.tile_begin = tiles;
        t.scale = c.scale;
        t.scale_inv = c.scale_inv;
        t.amax_in = c.amax;
        t.out = c.out;
        t.out_t = c.out_t;
        t.amax_bits = reinterpret_cast<unsigned *>(c.amax);
        t.ln_mean = c.ln_mean;
        t.ln_rstd = c.ln_rstd;
        t.ln_gamma = reinterpret_cast<const uint16_t *>(c.ln_gamma);
        t.ln_beta = reinterpret_cast<const uint16_t *>(c.ln_beta);
        if (c.rows > 0 && c.cols > 0) {
            if (!encode_tmap_2d(&args.maps[i], c.x, true, c.cols, c.rows, kQtTile, kQtTile, false))
                return false;
            tiles += ((c.rows + kQtTile - 1) / kQtTile) * t.tiles_c;
        } else {
            args.maps[i] = CUtensorMap{};
        }
    }
    for (int i = n; i < 2; ++i) {
        args.t[i] = args.t[0];
        args.maps[i] = args.maps[0];
    }
    args.num_tiles = tiles;
    return true;
}

cudaError_t launch_cast_group(const CastSpec *specs, int n, int fmt, bool current, int margin,
                              int sm_count, cudaStream_t st) {
    if (n < 1 || n > 2) return cudaErrorInvalidValue;
    // the amax passes run last tensor first, so that the first tensor, whose
    // tiles the cast takes first, is the one left in L2
    for (int i = n - 1; i >= 0; --i) {
        if (current && specs[i].ln_mean != nullptr) {
            // the LayerNorm statistics kernel has already written amax(y)
        } else if (current) {
            cudaError_t e = launch_amax(specs[i].x, specs[i].rows * specs[i].cols, specs[i].amax,
                                        sm_count, st);
            if (e != cudaSuccess) return e;
        } else if (specs[i].amax != nullptr && specs[i].zero_amax) {
            cudaError_t e = cudaMemsetAsync(specs[i].amax, 0, sizeof(float), st);
            if (e != cudaSuccess) return e;
        }
    }
    CastArgs args;
    if (!cast_args(args, specs, n, margin)) return cudaErrorInvalidValue;
    if (current) {
        // the amax was computed by amax_kernel; the cast only derives the scale
        for (int i = 0; i < n; ++i) args.t[i].amax_bits = nullptr;
        return fmt == 0 ? qt_launch<0, true>(args, sm_count, st)
                        : qt_launch<1, true>(args, sm_count, st);
    }
    return fmt == 0 ? qt_launch<0, false>(args, sm_count, st)
                    : qt_launch<1, false>(args, sm_count, st);
}

cudaError_t launch_quantize_transpose(const void *x, int64_t rows, int64_t cols,
                                      const float *scale, int fmt, uint8_t *out, uint8_t *out_t,
                                      float *amax, bool zero_amax, int sm_count,
                                      cudaStream_t st) {
    CastSpec c{x, rows, cols, const_cast<float *>(scale), nullptr, out, out_t, amax, zero_amax,
               nullptr, nullptr, nullptr, nullptr};
    return launch_cast_group(&c, 1, fmt, false, 0, sm_count, st);
}

cudaError_t launch_quantize_transpose_current(const void *x, int64_t rows, int64_t cols, int fmt,
                                              int margin, uint8_t *out, uint8_t *out_t,
                                              float *amax, float *scale, float *scale_inv,
                                              int sm_count, cudaStream_t st) {
    CastSpec c{x, rows, cols, scale, scale_inv, out, out_t, amax, true,
               nullptr, nullptr, nullptr, nullptr};
    return launch_cast_group(&c, 1, fmt, true, margin, sm_count, st);
}

cudaError_t launch_scale_update(float *history, float *amax, float *scale, float *scale_inv,
                                int num_tensors, int L, uint32_t format_mask, int margin,
                                bool clear_amax, cudaStream_t st) {
    const size_t smem = static_cast<size_t>(L) * sizeof(float);
    if (smem > 48 * 1024) {
        static bool raised = false;
        if (!raised) {
            cudaError_t e = cudaFuncSetAttribute(
                scale_update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
            if (e != cudaSuccess) return e;
            raised = true;
        }
    }
    return launch_pdl(scale_update_kernel, dim3(num_tensors), dim3(kUpdThreads), smem, st, history,
                      amax, scale, scale_inv, L, format_mask, margin, clear_amax ? 1 : 0);
}

}  // namespace fp8k

namespace fp8k {

// Diagnostic: one warp waits, with the library's bounded wait, on an
// mbarrier that nothing ever signals, gives up after limit_ns and reports it
// through the error flag -- the path every kernel takes when a wait runs out.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, nullptr, limit_ns))
        atomicOr(&g_cast_error_flags, kErrWaitTimeout);
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t read_and_clear_cast_error_flag(unsigned *flags) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_cast_error_flags, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_cast_error_flags, &zero, sizeof(unsigned));
}

}  // namespace fp8k
