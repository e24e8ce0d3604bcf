// fa_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA, tcgen05 (TMEM + MMA).
//
// Every wait in the library goes through wait_bounded(): a bounded mbarrier poll that gives
// up after a time limit (or when another role of the CTA has already given up), so a kernel
// never spins forever on a shared GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace fa {

// ---------------------------------------------------------------------------------------
// Generic helpers
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Named barrier over `nthreads` threads (a multiple of 32) that also ANDs a predicate across
// them: every participant gets true only if all passed true.  Used by warp pairs that share
// TMEM lanes; both warps reach it the same number of times on every path, so a failure seen
// by one warp stops both at the same point.
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Bounded wait by every lane of a warp, with a warp-uniform result.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                          uint64_t timeout_ns);

// Records a timeout in the device status word (first error wins) and tells the other roles
// of the CTA to stop.
__device__ __forceinline__ void record_timeout(int* status, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(status, 0, 4);
}

// ---------------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for phase `parity` of `bar` to complete.  Returns false (without completing) when
// `timeout_ns` elapses or when *abort becomes non-zero (abort may be null: time limit only);
// the caller then stops its role.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             const volatile int* abort, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (abort != nullptr && *abort) return false;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                          uint64_t timeout_ns) {
    return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort, timeout_ns));
}

// ---------------------------------------------------------------------------------------
// TMA (tiled tensor copies global -> shared, completion counted on an mbarrier)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 4-D tiled copy: coordinates (x = element in the row, y = row, z = head, w = batch).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

// Plain (untiled) bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completion counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------------------------------
// Tensor memory
// ---------------------------------------------------------------------------------------
// Whole warp: allocates `ncols` TMEM columns (power of two, 32..512); base address -> *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Generic-proxy writes to shared memory (st.shared) made visible to the async proxy (tcgen05.mma
// operand reads, bulk copies) of this CTA; each writing thread executes it before it signals.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Four fp32 additions into global memory, one 16-byte-aligned vector reduction (no result).
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-wide: thread t reads lane (lane_base + t), 32 consecutive 32-bit columns, and waits.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Warp-wide: two 32-column loads (addresses ta, tb) in flight together, then one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, uint32_t (&a)[32],
                                            uint32_t (&b)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]),
          "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
        : "r"(ta), "r"(tb)
        : "memory");
}

// Warp-wide: thread t writes 32 consecutive 32-bit columns of lane (lane_base + t).
// The caller issues tmem_st_wait() before publishing the data to another thread.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Warp-wide: thread t writes 16 consecutive 32-bit columns of lane (lane_base + t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// Warp-wide: thread t reads 16 consecutive 32-bit columns of lane (lane_base + t), and waits.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Warp-wide: thread t writes 8 consecutive 32-bit columns of lane (lane_base + t).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// Column-count generic forms (N = 16 or 32; stores also 8) used by kernels whose per-warp
// slice width is a compile-time constant.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]) {
    static_assert(N == 16 || N == 32, "16 or 32 columns");
    if constexpr (N == 16) tmem_ld16(taddr, r);
    else tmem_ld32(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&r)[N]) {
    static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 columns");
    if constexpr (N == 8) tmem_st8(taddr, r);
    else if constexpr (N == 16) tmem_st16(taddr, r);
    else tmem_st32(taddr, r);
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// tcgen05.mma (kind::f16: bf16 or fp16 operands, fp32 accumulator in TMEM)
// ---------------------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle, operand contiguous along K:
// rows of 128 B, groups of 8 rows 1024 B apart.  `saddr` may be offset by 32-byte steps
// inside a 1024-byte-aligned swizzle atom to select the K slice.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1u << 16) |
           ((uint64_t)(1024u >> 4) << 32) | ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

// Shared-memory matrix descriptor, 128-byte swizzle, operand contiguous along M or N:
// 64 16-bit elements per 128-byte row, consecutive K rows 128 B apart, groups of 8 K rows
// 1024 B apart, and 64-element M/N chunks `chunk_bytes` apart.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr, uint32_t chunk_bytes) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((chunk_bytes >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024u >> 4) << 32) | ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

// The same matrix descriptor with its start address moved by `bytes` (a multiple of 16; the
// resulting address stays below 256 KiB, so only the 14-bit start field changes).
__device__ __forceinline__ uint64_t sdesc_advance(uint64_t desc, uint32_t bytes) {
    return desc + (uint64_t)(bytes >> 4);
}

// Instruction descriptor: fp32 accumulate, A/B both bf16 (or both fp16), dense.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N, bool a_mn_major,
                                                 bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction-descriptor bit that negates the A operand (D = -A*B (+ D)); negation of a
// 16-bit value is exact, so the product is the exact negative of the plain one.
constexpr uint32_t kIdescNegateA = 1u << 13;

// D[tmem] (+)= A * B for one K=16 slice: mma_ss_w reads A and B from shared memory (via their
// descriptors), mma_ts_w reads A from TMEM (8 columns: two 16-bit values per 32-bit column, one
// row per lane).  Warp-converged: every lane of the warp executes the call with the same
// (warp-uniform) arguments and one lane chosen by elect.sync issues the instruction; keeping
// the issuing warp converged lets the descriptors stay warp-uniform values.  mma_commit_w
// arrives once on `bar` when every tcgen05 operation issued so far by that lane is done.
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Warp-wide load of N = 32, 64 or 128 consecutive columns (loads issued in pairs, one wait
// per pair).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
    static_assert(N == 32 || N == 64 || N == 128, "32, 64 or 128 columns");
    if constexpr (N == 32) {
        tmem_ld32(taddr, r);
    } else {
#pragma unroll
        for (int h = 0; h < N / 64; ++h)
            tmem_ld32x2(taddr + 64 * h, taddr + 64 * h + 32,
                        reinterpret_cast<uint32_t(&)[32]>(r[64 * h]),
                        reinterpret_cast<uint32_t(&)[32]>(r[64 * h + 32]));
    }
}

// Four consecutive fp32 values from shared memory (16-byte aligned shared address).  Shared
// tiles are addressed through pointers the compiler may only know as generic (an integer
// alignment round trip); an explicit ld.shared keeps these reads on the shared path.
__device__ __forceinline__ float4 lds_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// 16 bytes to / from shared memory at a 16-byte aligned shared address.
__device__ __forceinline__ void sts_u32x4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 lds_u32x4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// ---------------------------------------------------------------------------------------
// Counter-based random numbers for dropout: Philox-4x32 with 10 rounds (Salmon, Moraes, Dror,
// Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011), from that definition: each
// round multiplies words 0 and 2 by fixed odd constants, and the high halves, xored with words 1
// and 3 and the key, become the new words 0 and 2 (the low halves words 3 and 1); the key
// advances by two Weyl constants between rounds.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              uint32_t k0, uint32_t k1, uint32_t (&out)[4]) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

// Dropout keep bits of four consecutive keys j4..j4+3 (j4 a multiple of 4) of query row i of
// head bh: bit c set iff word c of the Philox block at counter (j4/4, i, bh, 0) is at least the
// threshold floor(p * 2^32).
__device__ __forceinline__ uint32_t dropout_keep4(uint32_t j4, uint32_t i, uint32_t bh,
                                                  uint32_t seed_lo, uint32_t seed_hi,
                                                  uint32_t threshold) {
    uint32_t w[4];
    philox4x32_10(j4 >> 2, i, bh, 0u, seed_lo, seed_hi, w);
    return (w[0] >= threshold ? 1u : 0u) | (w[1] >= threshold ? 2u : 0u) |
           (w[2] >= threshold ? 4u : 0u) | (w[3] >= threshold ? 8u : 0u);
}

// ---------------------------------------------------------------------------------------
// Math helpers
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs: the sm_100-family f32x2 instructions do two IEEE fp32 operations for one
// issue slot (each lane is rounded exactly like its scalar counterpart).
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Three-input maximum (one instruction; same NaN rule as fmaxf: a NaN operand is ignored).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
    if constexpr (BF16) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
        return __bfloat1622float2(h);
    } else {
        __half2 h = *reinterpret_cast<__half2*>(&u);
        return __half22float2(h);
    }
}

}  // namespace fa

namespace fa {

// Scales N fp32 values (as raw bits) by `mul`, rounds them to the 16-bit type and writes
// them as N*2 contiguous bytes at `dst` (16-byte aligned) with 16-byte stores.
template <bool BF16, int N>
__device__ __forceinline__ void store_row16(uint8_t* dst, const uint32_t (&r)[N], float mul) {
    static_assert(N % 8 == 0, "whole 16-byte stores");
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v = 0; v < N / 8; ++v) {
        uint4 w;
        w.x = pack2<BF16>(__uint_as_float(r[v * 8 + 0]) * mul, __uint_as_float(r[v * 8 + 1]) * mul);
        w.y = pack2<BF16>(__uint_as_float(r[v * 8 + 2]) * mul, __uint_as_float(r[v * 8 + 3]) * mul);
        w.z = pack2<BF16>(__uint_as_float(r[v * 8 + 4]) * mul, __uint_as_float(r[v * 8 + 5]) * mul);
        w.w = pack2<BF16>(__uint_as_float(r[v * 8 + 6]) * mul, __uint_as_float(r[v * 8 + 7]) * mul);
        d[v] = w;
    }
}

// Reads NCOLS (a multiple of 16) fp32 columns of this thread's TMEM lane, scales them and
// stores them as 16-bit values at `dst`; skips the stores (not the warp-wide loads) when
// `valid` is false.
template <bool BF16, int NCOLS>
__device__ __forceinline__ void tmem_row_to_global(uint32_t taddr, uint8_t* dst, float mul,
                                                   bool valid) {
    static_assert(NCOLS % 16 == 0, "16-column granularity");
    if constexpr (NCOLS % 32 == 0) {
#pragma unroll
        for (int c = 0; c < NCOLS / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(taddr + c * 32, r);
            if (valid) store_row16<BF16, 32>(dst + c * 64, r, mul);
        }
    } else {
#pragma unroll
        for (int c = 0; c < NCOLS / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(taddr + c * 16, r);
            if (valid) store_row16<BF16, 16>(dst + c * 32, r, mul);
        }
    }
}

// The rows of a warp (lane = row, NCOLS fp32 TMEM columns from taddr, NCOLS a multiple of 64)
// times `mul`, as 16-bit values into rows 0 .. 31 at dst0 + r * row_bytes (rows at or past
// n_rows are not written).  A row per lane would make every 16-byte store of the
// warp touch 32 cache lines; instead each 64-column chunk goes through the warp's 4 KB buffer
// at shared address `stage` (row r at 128 r, its 16-byte units XORed by r % 8, so that the
// row-wise writes and the column-wise reads are free of bank conflicts) and leaves as 4 rows
// of 128 contiguous bytes per store instruction.
template <bool BF16, int NCOLS>
__device__ __forceinline__ void tmem_rows_to_global_staged(uint32_t taddr, uint32_t stage,
                                                           uint8_t* dst0, size_t row_bytes,
                                                           int n_rows, float mul, int lane) {
    static_assert(NCOLS % 64 == 0, "64-column chunks");
#pragma unroll
    for (int c = 0; c < NCOLS / 64; ++c) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {  // 32 columns at a time
            uint32_t r[32];
            tmem_ld32(taddr + 64 * c + 32 * hf, r);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int u = 4 * hf + v;
                uint4 w;
                w.x = pack2<BF16>(__uint_as_float(r[8 * v + 0]) * mul, __uint_as_float(r[8 * v + 1]) * mul);
                w.y = pack2<BF16>(__uint_as_float(r[8 * v + 2]) * mul, __uint_as_float(r[8 * v + 3]) * mul);
                w.z = pack2<BF16>(__uint_as_float(r[8 * v + 4]) * mul, __uint_as_float(r[8 * v + 5]) * mul);
                w.w = pack2<BF16>(__uint_as_float(r[8 * v + 6]) * mul, __uint_as_float(r[8 * v + 7]) * mul);
                sts_u32x4(stage + lane * 128 + ((u ^ (lane & 7)) << 4), w);
            }
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int rr = 4 * k + (lane >> 3), uu = lane & 7;
            const uint4 w = lds_u32x4(stage + rr * 128 + ((uu ^ (rr & 7)) << 4));
            if (rr < n_rows)
                *reinterpret_cast<uint4*>(dst0 + (size_t)rr * row_bytes + c * 128 + uu * 16) = w;
        }
        __syncwarp();
    }
}

// The same read-out for a whole warp with coalesced stores.  Lane l holds row l of the warp's
// 32 (its TMEM lane); its NCOLS columns (16, 32 or 64), scaled and rounded to 16 bits, are
// U = NCOLS/8 16-byte units bound for dst0 + l * row_bytes.  A store per lane would touch 32
// rows (32 cache lines) per instruction.  Instead the warp transposes the units in groups of U
// lanes (a butterfly of xor shuffles), after which lane g*U + i holds unit i of rows
// g*U .. g*U+U-1, and each of U store instructions writes U contiguous units of one row per
// group: 32/U rows per instruction.  Rows at or past n_rows are not written.
template <bool BF16, int NCOLS>
__device__ __forceinline__ void tmem_rows_to_global_xpose(uint32_t taddr, uint8_t* dst0,
                                                          size_t row_bytes, int n_rows,
                                                          float mul, int lane) {
    static_assert(NCOLS == 16 || NCOLS == 32 || NCOLS == 64, "16, 32 or 64 columns");
    constexpr int U = NCOLS / 8;  // 16-byte units per row slice
    uint32_t m[U][4];             // m[e]: unit e of this row (before), unit i of row g*U+e (after)
#pragma unroll
    for (int c = 0; c < NCOLS; c += 16) {
        uint32_t r[16];
        tmem_ld16(taddr + c, r);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            m[c / 8 + k / 4][k % 4] =
                pack2<BF16>(__uint_as_float(r[2 * k]) * mul, __uint_as_float(r[2 * k + 1]) * mul);
    }
    // Stage s swaps, between lanes l and l^s, the units whose index differs from the lane's in
    // bit s: afterwards unit e of lane l came from lane (l & ~(U-1)) + e, unit index l % U.
#pragma unroll
    for (int s = U / 2; s >= 1; s /= 2) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int e = 0; e < U; ++e) {
            if (e & s) continue;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t send = upper ? m[e][k] : m[e | s][k];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, s);
                if (upper)
                    m[e][k] = recv;
                else
                    m[e | s][k] = recv;
            }
        }
    }
    const int g = lane / U, i = lane % U;
#pragma unroll
    for (int e = 0; e < U; ++e) {
        const int r = g * U + e;
        if (r < n_rows)
            *reinterpret_cast<uint4*>(dst0 + (size_t)r * row_bytes + i * 16) =
                make_uint4(m[e][0], m[e][1], m[e][2], m[e][3]);
    }
}

// Multiplies NCOLS fp32 TMEM columns of this thread's lane by `mul` in place.
template <int NCOLS>
__device__ __forceinline__ void tmem_row_scale(uint32_t taddr, float mul) {
    static_assert(NCOLS % 16 == 0, "16-column granularity");
    if constexpr (NCOLS % 32 == 0) {
#pragma unroll
        for (int c = 0; c < NCOLS / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(taddr + c * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * mul);
            tmem_st32(taddr + c * 32, r);
        }
    } else {
#pragma unroll
        for (int c = 0; c < NCOLS / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(taddr + c * 16, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * mul);
            tmem_st16(taddr + c * 16, r);
        }
    }
}

}  // namespace fa
