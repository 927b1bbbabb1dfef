// gemm.cu -- FP8 GEMM on the sm_103a tcgen05 tensor cores with the dequant
// epilogue of the FP8 linear layer (fprop, dgrad and wgrad all use it).
//
// What it computes ("Mixed-precision training" wiki note, bullet "extension
// to FP8": only the GEMMs run in FP8, accumulating in higher precision; the
// DQ node of "FP8 quantization with NVIDIA TensorRT"):
//   D[i][j] = bf16_rne(fl32(acc[i][j] * fl32(a_scale_inv * b_scale_inv))),
//   acc[i][j] = sum_k A[i][k] * B[j][k]   (fp32, in tensor memory),
//   d_amax = max |D| over the emitted BF16 values.
// A is [M][K] and B is [N][K], both contiguous along K ("TN").
//
// Design (one CTA per SM, persistent over output tiles of 128 x 256):
//   warp 0     TMA producer: 128-byte-swizzled K-slices of A (128 x 128 B)
//              and B (256 x 128 B) into a 4-stage shared-memory ring;
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators)
//              and issues tcgen05.mma (128 x 256 x 32 per instruction, four
//              per K-slice); tcgen05.commit frees ring stages and hands a
//              finished accumulator to the epilogue;
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter, scale, BF16
//              round, running amax, 16-byte stores; releases the accumulator
//              so the next tile's MMAs overlap this tile's epilogue.
// Tiles are visited in groups of 16 row-blocks so that concurrently running
// CTAs share A and B slices in L2.  Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

__device__ unsigned g_error_flags = 0;

namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4;
constexpr int A_STAGE = BM * BK, B_STAGE = BN * BK;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int GROUP_M = 16;
constexpr int NUM_BARS = 2 * STAGES + 4 + 1;  // full, empty, acc_full x2, acc_empty x2, drain
constexpr size_t SMEM_BYTES =
    1024 /*alignment slack*/ + STAGES * (A_STAGE + B_STAGE) + NUM_BARS * 8 + 16;

struct GemmParams {
    __nv_bfloat16 *D;
    unsigned *amax_bits;
    const float *a_scale_inv;
    const float *b_scale_inv;
    int64_t M, N;
    int tiles_m, tiles_n, num_kb;
    uint32_t idesc;
};

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int &mb, int &nb) {
    const int group = tile / (GROUP_M * tiles_n);
    const int first_m = group * GROUP_M;
    const int gm = min(tiles_m - first_m, GROUP_M);
    const int in = tile - group * GROUP_M * tiles_n;
    mb = first_m + in % gm;
    nb = in / gm;
}

__device__ __forceinline__ void raise_error(volatile int *abort_flag) {
    atomicOr(&g_error_flags, kErrWaitTimeout);
    *abort_flag = 1;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * B_STAGE);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t accf0 = smem_u32(bars + 2 * STAGES), acce0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 4);  // one arrival per epilogue warp
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = p.tiles_m * p.tiles_n;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                int mb, nb;
                tile_coords(tile, p.tiles_m, p.tiles_n, mb, nb);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
                        raise_error(abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_arrive_expect_tx(fb, A_STAGE + B_STAGE);
                    tma_load_2d(smem_u32(sA + stage * A_STAGE), &tmA, fb, kb * BK, mb * BM);
                    tma_load_2d(smem_u32(sB + stage * B_STAGE), &tmB, fb, kb * BK, nb * BN);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let the copies already issued land before the CTA exits.
                for (int i = 0; i < STAGES && issued > 0; ++i, --issued) {
                    stage = stage == 0 ? STAGES - 1 : stage - 1;
                    if (stage == STAGES - 1) phase ^= 1u;
                    mbar_wait(full0 + 8 * stage, phase, nullptr, 100000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, any = false;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                if (!mbar_wait(acce0 + 8 * acc, acc_phase ^ 1u, abort_flag)) {
                    raise_error(abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) {
                        raise_error(abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * A_STAGE);
                    const uint32_t b0 = smem_u32(sB + stage * B_STAGE);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_f8f6f4(d_tmem, smem_desc_sw128(a0 + 32 * k),
                                   smem_desc_sw128(b0 + 32 * k), p.idesc, (kb | k) != 0);
                    mma_commit(empty0 + 8 * stage);
                    any = true;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(accf0 + 8 * acc);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok && any) {
                // Wait (bounded) for the MMAs in flight before TMEM is freed.
                mma_commit(drain_bar);
                mbar_wait(drain_bar, 0, nullptr, 100000000ull);
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const float sab = __fmul_rn(*p.a_scale_inv, *p.b_scale_inv);
        uint32_t tmax = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, p.tiles_m, p.tiles_n, mb, nb);
            const bool got = mbar_wait(accf0 + 8 * acc, acc_phase, abort_flag);
            // the lanes leave the wait one by one; tcgen05.ld needs the whole warp
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) raise_error(abort_flag);
                break;
            }
            tc_fence_after();
            const int64_t row = static_cast<int64_t>(mb) * BM + q * 32 + lane;
            const bool row_in = row < p.M;
            __nv_bfloat16 *drow = p.D + row * p.N;
            const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_load_32cols(t_lane + c * 32, r);
                const int64_t col0 = static_cast<int64_t>(nb) * BN + c * 32;
                uint32_t packed[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float y0 = __fmul_rn(__uint_as_float(r[2 * j]), sab);
                    const float y1 = __fmul_rn(__uint_as_float(r[2 * j + 1]), sab);
                    const __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
                    packed[j] = *reinterpret_cast<const uint32_t *>(&h);
                }
                if (row_in) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        if (col0 + 8 * v < p.N) {
                            tmax = amax_bits2(tmax, packed[4 * v]);
                            tmax = amax_bits2(tmax, packed[4 * v + 1]);
                            tmax = amax_bits2(tmax, packed[4 * v + 2]);
                            tmax = amax_bits2(tmax, packed[4 * v + 3]);
                            *reinterpret_cast<uint4 *>(drow + col0 + 8 * v) =
                                make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                           packed[4 * v + 3]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce0 + 8 * acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (p.amax_bits != nullptr) {
            tmax = __reduce_max_sync(0xFFFFFFFFu, tmax);
            if (lane == 0 && tmax != 0) atomicMax(p.amax_bits, tmax << 16);
        }
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// --------------------------------------------------------------- host side --

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encode_kmajor_fp8(CUtensorMap *map, const uint8_t *base, int64_t rows, int64_t K,
                       uint32_t box_rows) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode == nullptr) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm_tn(const uint8_t *A, int fa, const uint8_t *B, int fb, int64_t M,
                           int64_t N, int64_t K, const float *a_scale_inv,
                           const float *b_scale_inv, void *D, float *d_amax, bool zero_amax,
                           int sm_count, cudaStream_t st, const char **what) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(gemm_tn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(SMEM_BYTES));
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (d_amax != nullptr && zero_amax) {
        cudaError_t e = cudaMemsetAsync(d_amax, 0, sizeof(float), st);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap ta, tb;
    if (!encode_kmajor_fp8(&ta, A, M, K, BM) || !encode_kmajor_fp8(&tb, B, N, K, BN)) {
        if (what) *what = "cuTensorMapEncodeTiled failed for an operand";
        return cudaErrorInvalidValue;
    }
    GemmParams p;
    p.D = reinterpret_cast<__nv_bfloat16 *>(D);
    p.amax_bits = reinterpret_cast<unsigned *>(d_amax);
    p.a_scale_inv = a_scale_inv;
    p.b_scale_inv = b_scale_inv;
    p.M = M;
    p.N = N;
    p.tiles_m = static_cast<int>((M + BM - 1) / BM);
    p.tiles_n = static_cast<int>((N + BN - 1) / BN);
    p.num_kb = static_cast<int>((K + BK - 1) / BK);
    p.idesc = idesc_f8(static_cast<uint32_t>(fa), static_cast<uint32_t>(fb), BM, BN);
    const int num_tiles = p.tiles_m * p.tiles_n;
    const int grid = num_tiles < sm_count ? num_tiles : sm_count;
    gemm_tn_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(ta, tb, p);
    return cudaGetLastError();
}

cudaError_t read_and_clear_error_flag(unsigned *flags, cudaStream_t st) {
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(flags, g_error_flags, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_error_flags, &zero, sizeof(unsigned));
}

}  // namespace fp8k
