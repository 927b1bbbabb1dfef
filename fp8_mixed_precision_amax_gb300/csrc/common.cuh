// common.cuh -- small inline-PTX helpers shared by the sm_103a kernels:
// mbarriers with bounded waits, TMA tile loads, tcgen05 (TMEM allocation,
// FP8 MMA, commit, TMEM loads) and the FP8 / BF16 conversions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "these kernels target sm_103a (tcgen05, TMA); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace fp8k {

// Bound on every spin-wait in a kernel (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Error bits a kernel may set in the library's device error flag.
constexpr unsigned kErrWaitTimeout = 1u;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------- programmatic dependent launch --
// Every kernel is launched so that it may start while the previous kernel in
// the stream is finishing (its launch and prologue overlap that tail).  Each
// kernel calls pdl_wait() before its first global-memory access: it returns
// once the previous kernel has completed and its writes are visible (at once
// when there is no such dependency).  pdl_trigger() then lets the next kernel
// be scheduled as soon as resources free up.

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch a kernel with the programmatic-stream-serialization attribute.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up (returns
// false) after kWaitLimitNs, or as soon as *abort_flag becomes non-zero.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile int *abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (abort_flag != nullptr && *abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

// -------------------------------------------------------------------- TMA --

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled TMA load of one box into shared memory; completion is signalled
// as transaction bytes on `bar`.  x is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// Untiled bulk copy of `bytes` contiguous bytes from global memory into this
// CTA's shared memory, completing as transaction bytes on `bar`.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void *src, uint32_t bytes,
                                             uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// TMA store of a box from this CTA's shared memory (bulk-group completion,
// tracked per issuing thread), and the waits on those groups.
__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t src, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// at most N of this thread's most recent bulk groups still reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// at most N of this thread's most recent bulk groups not yet complete
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
// generic-proxy writes to shared memory become visible to the async proxy (TMA)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05 --

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T, one 128 x N x 32 FP8 MMA issued by one thread.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row swizzle atoms of 1024
// bytes (stride byte offset), descriptor version 1, layout "128B swizzle".
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(16u >> 4) << 16;             // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;           // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                   // version
    d |= static_cast<uint64_t>(2u) << 61;                   // swizzle: 128 bytes
    return d;
}

// Instruction descriptor of kind::f8f6f4: fp32 accumulator, A / B formats
// (0 = E4M3, 1 = E5M2), both K-major, no negation, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f8(uint32_t fa, uint32_t fb, uint32_t m, uint32_t n) {
    return (1u << 4) | (fa << 7) | (fb << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

#define FP8K_R32(r)                                                                              \
    "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),       \
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), \
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),          \
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),          \
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])

// Load 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape,
// 32 repetitions) and wait for them.  The registers are tied through the wait
// so no use can be scheduled before it.
__device__ __forceinline__ void tmem_load_32cols(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : FP8K_R32(r)
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" : FP8K_R32(r) : : "memory");
}

// ------------------------------------------- CTA pairs (cta_group::2) --
// A cluster of two CTAs on two SMs computes one 256-row tile: each CTA
// TMA-loads its own operand halves into its own shared memory (no
// multicast), and the even CTA issues MMAs that read both CTAs' shared
// memory and write both CTAs' tensor memory.

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

// Address in the cluster's shared window of the variable at `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of any CTA of the cluster (address from mapa_shared).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *tmap, uint32_t bar_cluster,
                                                 int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D (both CTAs' tensor memory) (+)= A (256 rows, 128 per CTA) * B^T (N
// columns, half per CTA), issued by one thread of the even CTA.
__device__ __forceinline__ void mma_f8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at the same shared-memory offset in every CTA of
// `cta_mask` when all tcgen05 operations issued so far by this thread are done.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// ------------------------------------------------------------ conversions --

// Two binary32 values to two FP8 codes with round-to-nearest-even and
// saturation to the largest finite value (NaN stays NaN); `lo` lands in the
// low byte.
__device__ __forceinline__ uint32_t cvt2_e4m3(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t cvt2_e5m2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int FMT>
__device__ __forceinline__ uint32_t cvt2_fp8(float lo, float hi) {
    if constexpr (FMT == 0)
        return cvt2_e4m3(lo, hi);
    else
        return cvt2_e5m2(lo, hi);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed fp32 pairs (lo in the low word of a 64-bit register) and IEEE
// round-to-nearest arithmetic on both lanes at once: each lane is rounded
// exactly as the scalar operation would be.  One caution: ptxas contracts a
// packed multiply whose result feeds a packed add or subtract into one fused
// multiply-add, even with .rn and -fmad=false (and it folds an explicit fma
// with a -0 addend back into that pattern).  Where a product is added, the
// add is therefore done with the scalar __fadd_rn / __fsub_rn, which are
// never contracted.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    uint64_t v;
    asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
    return v;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// the two BF16 values of w (lo in the low half), widened to fp32
__device__ __forceinline__ uint64_t f32x2_from_bf16x2(uint32_t w) {
    uint64_t v;
    asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(w << 16), "r"(w & 0xFFFF0000u));
    return v;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// a * b + c per lane with one rounding (an explicit fused multiply-add)
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t splat_f32x2(float s) { return f32x2_pack(s, s); }

// Division by a divisor known in advance, correctly rounded (to nearest,
// ties to even), two lanes at a time.  With y = RN(1/b) (itself an IEEE
// division, once), q0 = RN(a*y) is within 1.5 ulp of a/b; one correction
// q1 = RN(q0 + RN(a - b*q0)*y) makes it faithful, and a second one is exact
// by Markstein's theorem (y within half an ulp of 1/b and q1 within one ulp
// of a/b give RN(q1 + (a - b*q1)*y) = RN(a/b), the remainder a - b*q1 being
// exact in an fma).  The theorem needs no overflow or underflow on the way,
// which holds for 2^-20 <= b <= 1 and 2^-100 <= |a| <= 2^100; other a
// (zeros, whose sign the corrections would lose, NaN, infinities, the
// extremes) and other b take __fdiv_rn.
struct DivConst {
    uint64_t y2, nb2;   // {y, y} and {-b, -b}
    float b;
    bool fast;          // 2^-20 <= b <= 1
};
__device__ __forceinline__ DivConst div_const(float b) {
    DivConst d;
    d.b = b;
    d.fast = b >= 0x1p-20f && b <= 1.0f;
    d.y2 = splat_f32x2(__fdiv_rn(1.0f, b));
    d.nb2 = splat_f32x2(-b);
    return d;
}
__device__ __forceinline__ bool div_const_in_range(float a) {
    const float aa = fabsf(a);
    return aa >= 0x1p-100f && aa <= 0x1p100f;   // false for NaN
}
static __device__ __noinline__ float div_const_slow(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ void div_by_const2(float a0, float a1, const DivConst &d, float &q0,
                                              float &q1) {
    const uint64_t a2 = f32x2_pack(a0, a1);
    uint64_t q = f32x2_mul(a2, d.y2);
    q = f32x2_fma(f32x2_fma(d.nb2, q, a2), d.y2, q);
    q = f32x2_fma(f32x2_fma(d.nb2, q, a2), d.y2, q);
    f32x2_unpack(q, q0, q1);
    const bool ok0 = d.fast && div_const_in_range(a0), ok1 = d.fast && div_const_in_range(a1);
    if (!(ok0 && ok1)) {
        if (!ok0) q0 = div_const_slow(a0, d.b);
        if (!ok1) q1 = div_const_slow(a1, d.b);
    }
}

// Mixed-precision scalar forms: the low or high BF16 of w, widened to fp32
// exactly, added to or less c with one rounding (the same result as widening
// first, without the register pairing of the packed forms).
__device__ __forceinline__ float bf16lo_add_f32(uint32_t w, float c) {
    float d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, lo, %2;\n\t}"
        : "=f"(d) : "r"(w), "f"(c));
    return d;
}
__device__ __forceinline__ float bf16hi_add_f32(uint32_t w, float c) {
    float d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, hi, %2;\n\t}"
        : "=f"(d) : "r"(w), "f"(c));
    return d;
}
__device__ __forceinline__ float bf16lo_sub_f32(uint32_t w, float c) {
    float d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tsub.rn.f32.bf16 %0, lo, %2;\n\t}"
        : "=f"(d) : "r"(w), "f"(c));
    return d;
}
__device__ __forceinline__ float bf16hi_sub_f32(uint32_t w, float c) {
    float d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tsub.rn.f32.bf16 %0, hi, %2;\n\t}"
        : "=f"(d) : "r"(w), "f"(c));
    return d;
}

// Two fp32 values (bit patterns lo, hi) times s2 = {s, s}, rounded to BF16
// and packed (lo in the low half).
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t lo, uint32_t hi, uint64_t s2) {
    float a, b;
    f32x2_unpack(f32x2_mul(f32x2_pack(__uint_as_float(lo), __uint_as_float(hi)), s2), a, b);
    uint32_t h;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(b), "f"(a));
    return h;
}

// Running max of |x| over packed BF16 pairs in one instruction per pair:
// each lane of m2 holds the largest magnitude so far (its sign bit is the
// xor of signs and carries no meaning).  max.xorsign.abs.bf16x2 returns the
// other operand when one is NaN (checked on the GPU against abs + max over
// all 2^32 lane pairs), so NaN entries are skipped and infinities kept; m2
// starts at 0 and is never NaN.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t m2, uint32_t w) {
    asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(w));
    return m2;
}

// The larger magnitude of m2's two lanes, as BF16 magnitude bits.
__device__ __forceinline__ uint32_t absmax_bf16x2_finish(uint32_t m2) {
    return max(m2 & 0x7FFFu, (m2 >> 16) & 0x7FFFu);
}

// The two BF16 values of w (lo in the low half) widened to fp32, times
// s2 = {s, s}, and cast to FP8 (lo in the low byte of the result).
template <int FMT>
__device__ __forceinline__ uint32_t scale_fp8x2_bf16x2(uint32_t w, uint64_t s2) {
    float a, b;
    f32x2_unpack(f32x2_mul(f32x2_from_bf16x2(w), s2), a, b);
    return cvt2_fp8<FMT>(a, b);
}

// ------------------------------------------------------- the scale formula --
// scale = fl32(fl32(fmax / m) * 2^-margin), +inf clamped to FLT_MAX, when
// 0 < m < inf (m = the amax, or the max over the amax history); otherwise the
// previous scale is kept (valid = false).  0 <= margin <= 64.
__device__ __forceinline__ float recipe_scale(float m, float fmax, int margin, float prev,
                                              bool &valid) {
    valid = m > 0.0f && m <= 3.402823466e38f;
    if (!valid) return prev;
    const float q = __fdiv_rn(fmax, m);
    const float p2 = __uint_as_float(static_cast<uint32_t>(127 - margin) << 23);
    float sc = __fmul_rn(q, p2);
    if (sc > 3.402823466e38f) sc = 3.402823466e38f;
    return sc;
}

}  // namespace fp8k
