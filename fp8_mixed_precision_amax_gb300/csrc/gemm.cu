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
// Design (one CTA per SM, persistent over output tiles):
//   warp 0     TMA producer: 128-byte-swizzled 128-deep K-slices of A and B
//              into a shared-memory ring;
//   warp 1     allocates 512 TMEM columns (two 256-column fp32 accumulators)
//              and issues tcgen05.mma (four per K-slice); tcgen05.commit
//              frees ring stages and hands a finished accumulator on;
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter, scale and
//              round with packed fp32x2 / bf16x2 instructions (the epilogue
//              shares issue slots with the single-thread producer and MMA
//              loops, so its instruction count shows in the MMA rate),
//              running amax; each 32-row x 64-column chunk goes to a
//              128-byte-swizzled staging buffer (two per warp) and out with
//              one TMA store, so the output leaves in whole lines.  The
//              accumulator is released as soon as the tile's last tcgen05.ld
//              has landed, so the next tile's MMAs overlap this epilogue.
// Above 128 rows, two CTAs on two SMs (a cluster) share each 256 x 256 tile
// (tcgen05 cta_group::2): each loads its own 128 A rows and 128 of the 256 B
// rows, and the even CTA issues M = 256 MMAs that read both CTAs' shared
// memory and write both CTAs' tensor memory.  No TMA multicast is used.
// One launch may carry two independent GEMMs (the backward pass's dgrad and
// wgrad): their tiles form one list, so the last, partly filled wave of one
// is filled with tiles of the other.  Tiles are visited in groups of
// row-blocks chosen per problem so that the smaller operand stays in L2.
// Every wait is bounded.
#include <cuda_bf16.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

__device__ unsigned g_error_flags = 0;

// Diagnostic clock probe (fp8_set_clock_probe): a device pointer that every
// GEMM launch passes to its kernel while it is set.
std::atomic<unsigned long long *> g_clock_probe{nullptr};

void set_clock_probe(unsigned long long *acc) { g_clock_probe.store(acc); }

namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int GROUP_M = 16;                 // row-blocks per raster group when neither operand
constexpr int GROUP_M_SMALL = 8;            // fits: GROUP_M when A is the smaller, else GROUP_M_SMALL
constexpr int64_t RESIDENT_BYTES = 48 << 20;   // an operand this small is kept in L2
constexpr int MAX_PROBLEMS = 2;
constexpr int EPI_COLS = 64;                      // output columns per TMA store (128 B of BF16)
constexpr int EPI_BUF = 32 * EPI_COLS * 2;        // one warp's staging buffer: 32 rows x 128 B
constexpr int EPI_BYTES = 4 * 2 * EPI_BUF;        // four epilogue warps, two buffers each

template <bool PAIR>
struct Cfg {
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;    // B rows loaded per CTA
    static constexpr int STAGES = PAIR ? 6 : 4;
    static constexpr int A_STAGE = BM * BK;
    static constexpr int B_STAGE = B_ROWS * BK;
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;    // output rows per (pair) tile
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;  // full, empty, acc_full x2, acc_empty x2, drain
    static constexpr size_t SMEM =
        1024 + STAGES * (A_STAGE + B_STAGE) + EPI_BYTES + NUM_BARS * 8 + 16;
    static constexpr uint32_t STAGE_TX = (PAIR ? 2 : 1) * (A_STAGE + B_STAGE);
    static constexpr uint32_t EPI_ARRIVALS = PAIR ? 8 : 4;  // epilogue warps per tile
};

struct GemmProblem {
    __nv_bfloat16 *D;
    unsigned *amax_bits;
    const float *a_scale_inv;
    const float *b_scale_inv;
    int64_t M, N;
    int tiles_m, tiles_n, num_kb;
    int group_m;      // row-blocks per raster group (see make_args)
    int tile_begin;   // first index of this problem's tiles in the launch's tile list
    uint32_t idesc;
};

struct GemmArgs {
    CUtensorMap maps[2 * MAX_PROBLEMS];   // A0, B0, A1, B1
    CUtensorMap dmaps[MAX_PROBLEMS];      // D0, D1 (BF16, 64 x 32 boxes, 128-byte swizzle)
    GemmProblem prob[MAX_PROBLEMS];
    int num_problems;
    int num_tiles;
    unsigned long long *clock_probe;      // diagnostic: {SM cycles, ns} of CTA 0, or null
};

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m,
                                            int &mb, int &nb) {
    const int group = tile / (group_m * tiles_n);
    const int first_m = group * group_m;
    const int gm = min(tiles_m - first_m, group_m);
    const int in = tile - group * group_m * tiles_n;
    mb = first_m + in % gm;
    nb = in / gm;
}

// Problem and (row-block, column-block) of a tile of the launch's list.
__device__ __forceinline__ int locate(const GemmArgs &a, int tile, int &mb, int &nb) {
    const int p = (a.num_problems > 1 && tile >= a.prob[1].tile_begin) ? 1 : 0;
    tile_coords(tile - a.prob[p].tile_begin, a.prob[p].tiles_m, a.prob[p].tiles_n,
                a.prob[p].group_m, mb, nb);
    return p;
}

__device__ __forceinline__ void raise_error(volatile int *abort_flag) {
    atomicOr(&g_error_flags, kErrWaitTimeout);
    *abort_flag = 1;
}

template <bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_tn_kernel(const __grid_constant__ GemmArgs a) {
    using C = Cfg<PAIR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + C::STAGES * C::A_STAGE;
    uint8_t *sD = sB + C::STAGES * C::B_STAGE;   // epilogue staging, 1024-byte aligned
    uint64_t *bars = reinterpret_cast<uint64_t *>(sD + EPI_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;   // 0 = the CTA that issues MMAs
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int num_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + C::STAGES);
    const uint32_t accf0 = smem_u32(bars + 2 * C::STAGES);
    const uint32_t acce0 = smem_u32(bars + 2 * C::STAGES + 2);
    const uint32_t drain_bar = smem_u32(bars + 2 * C::STAGES + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, C::EPI_ARRIVALS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int i = 0; i < 2 * a.num_problems; ++i) prefetch_tmap(&a.maps[i]);
        for (int i = 0; i < a.num_problems; ++i) prefetch_tmap(&a.dmaps[i]);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    __syncthreads();
    if constexpr (PAIR) {
        __syncwarp();
        cluster_sync();   // both CTAs' barriers exist before any remote signal
    }
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the prologue above touched only this CTA's own memory
    pdl_wait();
    pdl_trigger();
    uint64_t probe_clk = 0, probe_ns = 0;
    if (a.clock_probe != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
        probe_clk = clock64();
        probe_ns = globaltimer_ns();
    }

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int tile = unit; ok && tile < a.num_tiles; tile += num_units) {
                int mb, nb;
                const int pi = locate(a, tile, mb, nb);
                const CUtensorMap *tmA = &a.maps[2 * pi];
                const CUtensorMap *tmB = &a.maps[2 * pi + 1];
                const int32_t arow = mb * C::TILE_M + static_cast<int32_t>(rank) * BM;
                const int32_t brow = nb * BN + static_cast<int32_t>(rank) * C::B_ROWS;
                const int num_kb = a.prob[pi].num_kb;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
                        raise_error(abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    const uint32_t dA = smem_u32(sA + stage * C::A_STAGE);
                    const uint32_t dB = smem_u32(sB + stage * C::B_STAGE);
                    if constexpr (PAIR) {
                        // both halves complete on the even CTA's barrier
                        const uint32_t fb0 = mapa_shared(fb, 0);
                        if (rank == 0) mbar_arrive_expect_tx(fb, C::STAGE_TX);
                        tma_load_2d_pair(dA, tmA, fb0, kb * BK, arow);
                        tma_load_2d_pair(dB, tmB, fb0, kb * BK, brow);
                    } else {
                        mbar_arrive_expect_tx(fb, C::STAGE_TX);
                        tma_load_2d(dA, tmA, fb, kb * BK, arow);
                        tma_load_2d(dB, tmB, fb, kb * BK, brow);
                    }
                    ++issued;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (ok) {
                // Every stage's last release must have arrived before the CTA exits
                // (in a pair it is signalled from the other SM).
                for (int i = 0; i < C::STAGES; ++i) {
                    mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            } else if (!PAIR || rank == 0) {
                // Let the copies already issued land before the CTA exits.
                for (int i = 0; i < C::STAGES && issued > 0; ++i, --issued) {
                    stage = stage == 0 ? C::STAGES - 1 : stage - 1;
                    if (stage == C::STAGES - 1) phase ^= 1u;
                    mbar_wait(full0 + 8 * stage, phase, nullptr, 100000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && rank == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, any = false;
            for (int tile = unit; ok && tile < a.num_tiles; tile += num_units) {
                int mb, nb;
                const int pi = locate(a, tile, mb, nb);
                const int num_kb = a.prob[pi].num_kb;
                const uint32_t idesc = a.prob[pi].idesc;
                if (!mbar_wait(acce0 + 8 * acc, acc_phase ^ 1u, abort_flag)) {
                    raise_error(abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) {
                        raise_error(abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * C::A_STAGE);
                    const uint32_t b0 = smem_u32(sB + stage * C::B_STAGE);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k) {
                        const uint64_t ad = smem_desc_sw128(a0 + 32 * k);
                        const uint64_t bd = smem_desc_sw128(b0 + 32 * k);
                        if constexpr (PAIR)
                            mma_f8f6f4_pair(d_tmem, ad, bd, idesc, (kb | k) != 0);
                        else
                            mma_f8f6f4(d_tmem, ad, bd, idesc, (kb | k) != 0);
                    }
                    if constexpr (PAIR)
                        mma_commit_pair(empty0 + 8 * stage, 0x3);
                    else
                        mma_commit(empty0 + 8 * stage);
                    any = true;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (PAIR)
                    mma_commit_pair(accf0 + 8 * acc, 0x3);
                else
                    mma_commit(accf0 + 8 * acc);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok && any) {
                // Wait (bounded) for the MMAs in flight before TMEM is freed.
                if constexpr (PAIR)
                    mma_commit_pair(drain_bar, 0x1);
                else
                    mma_commit(drain_bar);
                mbar_wait(drain_bar, 0, nullptr, 100000000ull);
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        float sab[MAX_PROBLEMS];
        uint32_t tmax[MAX_PROBLEMS];
#pragma unroll
        for (int i = 0; i < MAX_PROBLEMS; ++i) {
            sab[i] = i < a.num_problems ? __fmul_rn(*a.prob[i].a_scale_inv, *a.prob[i].b_scale_inv)
                                        : 0.0f;
            tmax[i] = 0;
        }
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t epi_chunk = 0;   // chunks staged so far (selects the staging buffer)
        for (int tile = unit; tile < a.num_tiles; tile += num_units) {
            int mb, nb;
            const int pi = locate(a, tile, mb, nb);
            const GemmProblem &P = a.prob[pi];
            const bool got = mbar_wait(accf0 + 8 * acc, acc_phase, abort_flag);
            // the lanes leave the wait one by one; tcgen05.ld needs the whole warp
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) raise_error(abort_flag);
                break;
            }
            tc_fence_after();
            const uint64_t s2 = splat_f32x2(pi ? sab[1] : sab[0]);
            uint32_t m2 = 0;   // two BF16 magnitude maxima
            const int64_t row0 = static_cast<int64_t>(mb) * C::TILE_M + rank * BM + q * 32;
            const bool row_in = row0 + lane < P.M;
            const CUtensorMap *tmD = &a.dmaps[pi];
            const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN / EPI_COLS; ++c) {
                uint32_t r[2][32];
                tmem_load_32cols(t_lane + c * EPI_COLS, r[0]);
                tmem_load_32cols(t_lane + c * EPI_COLS + 32, r[1]);
                if (c == BN / EPI_COLS - 1) {
                    // the whole accumulator is in registers: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR)
                            mbar_arrive_cluster(mapa_shared(acce0 + 8 * acc, 0));
                        else
                            mbar_arrive(acce0 + 8 * acc);
                    }
                }
                const int64_t col0 = static_cast<int64_t>(nb) * BN + c * EPI_COLS;
                uint32_t packed[32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        packed[16 * h + j] = scale_bf16x2(r[h][2 * j], r[h][2 * j + 1], s2);
                }
                if (row_in) {
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        if (col0 + 8 * v < P.N) {
                            m2 = absmax_bf16x2(m2, packed[4 * v]);
                            m2 = absmax_bf16x2(m2, packed[4 * v + 1]);
                            m2 = absmax_bf16x2(m2, packed[4 * v + 2]);
                            m2 = absmax_bf16x2(m2, packed[4 * v + 3]);
                        }
                    }
                }
                // this buffer's previous store (two chunks back) has read it
                if (lane == 0) bulk_wait_group_read<1>();
                __syncwarp();
                // row `lane` of the 32 x 128 B box; 16-byte chunk j sits at
                // j ^ (row mod 8), the 128-byte swizzle the tensor map names
                const uint32_t sbuf = smem_u32(sD + (q * 2 + (epi_chunk & 1)) * EPI_BUF);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4), packed[4 * j],
                                 packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (row0 < P.M && col0 < P.N)   // boxes wholly outside D are skipped
                        tma_store_2d(tmD, sbuf, static_cast<int32_t>(col0),
                                     static_cast<int32_t>(row0));
                    bulk_commit_group();
                }
                ++epi_chunk;
            }
            const uint32_t m = absmax_bf16x2_finish(m2);   // BF16 magnitude bits
            if (pi)
                tmax[1] = max(tmax[1], m);
            else
                tmax[0] = max(tmax[0], m);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // every store has left shared memory and reached global memory
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
#pragma unroll
        for (int i = 0; i < MAX_PROBLEMS; ++i) {
            if (i < a.num_problems && a.prob[i].amax_bits != nullptr) {
                const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, tmax[i]);
                if (lane == 0 && m != 0) atomicMax(a.prob[i].amax_bits, m << 16);
            }
        }
    }

    __syncthreads();
    if constexpr (PAIR) {
        __syncwarp();
        cluster_sync();   // the other SM is done with this CTA's memory
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (a.clock_probe != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
        atomicAdd(a.clock_probe, static_cast<unsigned long long>(clock64() - probe_clk));
        atomicAdd(a.clock_probe + 1, static_cast<unsigned long long>(globaltimer_ns() - probe_ns));
    }
}

// --------------------------------------------------------------- host side --

template <bool PAIR>
cudaError_t set_smem_attr() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(gemm_tn_kernel<PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(Cfg<PAIR>::SMEM));
    });
    return err;
}

// attr must have room for two attributes: the cluster shape and, with pdl,
// programmatic stream serialization.
cudaLaunchConfig_t pair_config(int grid, cudaLaunchAttribute *attr, cudaStream_t st, bool pdl) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg<true>::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cfg;
}

// Number of CTA pairs that can be resident at once (clusters of two need two
// SMs of the same GPC), cached per process.
int pair_slots(int sm_count) {
    static std::once_flag once;
    static int slots = 0;
    std::call_once(once, [sm_count] {
        if (set_smem_attr<true>() != cudaSuccess) return;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = pair_config(sm_count & ~1, attr, nullptr, false);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_tn_kernel<true>, &cfg) != cudaSuccess || n < 1)
            n = 0;
        slots = n;
    });
    return slots;
}

}  // namespace

cudaError_t launch_gemm_group(const GemmSpec *specs, int n, int sm_count, cudaStream_t st,
                              const char **what) {
    if (n < 1 || n > MAX_PROBLEMS) return cudaErrorInvalidValue;
    // CTA pairs when every problem is taller than one 128-row tile and the GPU
    // can hold them; single CTAs otherwise.
    bool tall = true;
    for (int i = 0; i < n; ++i) tall = tall && specs[i].M > BM;
    const int slots = tall ? pair_slots(sm_count) : 0;
    const bool pair = slots > 0;
    const int tile_m = pair ? 2 * BM : BM;
    const uint32_t b_rows = pair ? BN / 2 : BN;
    GemmArgs a;
    a.num_problems = n;
    a.clock_probe = g_clock_probe.load(std::memory_order_relaxed);
    int tiles = 0;
    for (int i = 0; i < n; ++i) {
        const GemmSpec &g = specs[i];
        if (g.d_amax != nullptr && g.zero_amax) {
            cudaError_t e = cudaMemsetAsync(g.d_amax, 0, sizeof(float), st);
            if (e != cudaSuccess) return e;
        }
        if (!encode_tmap_2d(&a.maps[2 * i], g.A, false, g.K, g.M, BK, BM, true) ||
            !encode_tmap_2d(&a.maps[2 * i + 1], g.B, false, g.K, g.N, BK, b_rows, true)) {
            if (what) *what = "cuTensorMapEncodeTiled failed for an operand";
            return cudaErrorInvalidValue;
        }
        if (!encode_tmap_2d(&a.dmaps[i], g.D, true, g.N, g.M, EPI_COLS, 32, true)) {
            if (what) *what = "cuTensorMapEncodeTiled failed for the output";
            return cudaErrorInvalidValue;
        }
        GemmProblem &p = a.prob[i];
        p.D = reinterpret_cast<__nv_bfloat16 *>(g.D);
        p.amax_bits = reinterpret_cast<unsigned *>(g.d_amax);
        p.a_scale_inv = g.a_scale_inv;
        p.b_scale_inv = g.b_scale_inv;
        p.M = g.M;
        p.N = g.N;
        p.tiles_m = static_cast<int>((g.M + tile_m - 1) / tile_m);
        p.tiles_n = static_cast<int>((g.N + BN - 1) / BN);
        p.num_kb = static_cast<int>((g.K + BK - 1) / BK);
        // Raster: tiles are walked down groups of group_m row-blocks.  When
        // one operand is small enough to stay in L2, walk so that it does
        // and the other streams through once: all row-blocks at a time when
        // A is the smaller (A resident), two row-blocks when B is (B
        // resident).  When neither fits: groups of GROUP_M row-blocks when
        // A is the smaller, so that the larger B is walked fewer times, and
        // of GROUP_M_SMALL otherwise, which keeps more of B in L2 from one
        // group's waves to the next.  (70B-shaped layer, DRAM bytes per
        // launch: fprop 1.10 GB with 16 against 1.47 GB with 8; the grouped
        // backward 3.85 GB with 8 and 8 against 4.51 GB with 16 and 16.)
        const int64_t a_bytes = g.M * g.K, b_bytes = g.N * g.K;
        if (a_bytes <= b_bytes && a_bytes <= RESIDENT_BYTES)
            p.group_m = p.tiles_m;
        else if (b_bytes < a_bytes && b_bytes <= RESIDENT_BYTES)
            p.group_m = 2;
        else
            p.group_m = a_bytes < b_bytes ? GROUP_M : GROUP_M_SMALL;
        p.tile_begin = tiles;
        p.idesc = idesc_f8(static_cast<uint32_t>(g.fa), static_cast<uint32_t>(g.fb),
                           static_cast<uint32_t>(tile_m), BN);
        tiles += p.tiles_m * p.tiles_n;
    }
    for (int i = n; i < MAX_PROBLEMS; ++i) {
        a.prob[i] = a.prob[0];
        a.maps[2 * i] = a.maps[0];
        a.maps[2 * i + 1] = a.maps[1];
        a.dmaps[i] = a.dmaps[0];
    }
    a.num_tiles = tiles;
    if (pair) {
        cudaError_t e = set_smem_attr<true>();
        if (e != cudaSuccess) return e;
        const int units = tiles < slots ? tiles : slots;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = pair_config(2 * units, attr, st, true);
        return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<true>, a);
    }
    cudaError_t e = set_smem_attr<false>();
    if (e != cudaSuccess) return e;
    const int grid = tiles < sm_count ? tiles : sm_count;
    return launch_pdl(gemm_tn_kernel<false>, dim3(grid), dim3(NUM_THREADS), Cfg<false>::SMEM, st,
                      a);
}

cudaError_t launch_gemm_tn(const uint8_t *A, int fa, const uint8_t *B, int fb, int64_t M,
                           int64_t N, int64_t K, const float *a_scale_inv,
                           const float *b_scale_inv, void *D, float *d_amax, bool zero_amax,
                           int sm_count, cudaStream_t st, const char **what) {
    GemmSpec g{A, fa, B, fb, M, N, K, a_scale_inv, b_scale_inv, D, d_amax, zero_amax};
    return launch_gemm_group(&g, 1, sm_count, st, what);
}

cudaError_t read_and_clear_error_flag(unsigned *flags, cudaStream_t st) {
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(flags, g_error_flags, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_error_flags, &zero, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    unsigned cast_flags = 0, sum_flags = 0;
    e = read_and_clear_cast_error_flag(&cast_flags);
    *flags |= cast_flags;
    if (e != cudaSuccess) return e;
    e = read_and_clear_sum_error_flag(&sum_flags);
    *flags |= sum_flags;
    return e;
}

}  // namespace fp8k
