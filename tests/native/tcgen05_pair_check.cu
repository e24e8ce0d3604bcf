// tcgen05_pair_check.cu -- checks the CTA-pair (cta_group::2) tensor-core mechanics that a
// 2-CTA attention kernel is built on, against a CPU product, on one GB300 (sm_103a):
//   * a cluster of two CTAs on two SMs, tensor memory allocated for the pair
//     (tcgen05.alloc.cta_group::2 by one warp of each CTA) at the same column in both;
//   * one tcgen05.mma.cta_group::2 issued by the even CTA computes D (256 x N) = A B^T with
//     A's rows 0-127 in the even CTA's shared memory and rows 128-255 in the odd CTA's (same
//     offset), and B's first N/2 rows in the even CTA, the other N/2 in the odd one;
//     each CTA's tensor memory receives its own 128 rows x all N columns;
//   * the TS form (A from tensor memory, each CTA holding its 128 rows);
//   * completion signalled to both CTAs' mbarriers with two plain commits (no multicast).
// Inputs are small integers, so every fp32 sum is exact and the check is bit for bit.  It also
// times 2048 back-to-back pair steps (M = 256, N = 128, K = 16) of each form: clock64 cycles
// per step, against 64 for a single-CTA M = 128 step.
// Every wait is bounded (2 s); the program prints one JSON object and exits non-zero on a
// mismatch or a timeout.
//
// Build and run:  nvcc -std=c++17 -gencode arch=compute_103a,code=sm_103a -O3 \
//                     tests/native/tcgen05_pair_check.cu -o tcgen05_pair_check && ./tcgen05_pair_check
#include <cuda_runtime.h>

#include <cstdio>
#include <vector>

#include "../../tiled_attention_08_gb300/csrc/fa_ptx.cuh"

using namespace fa;

namespace {

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int N = 128;           // B rows (keys), N / 2 per CTA
constexpr int K = 64;            // one 128-byte swizzle row of 16-bit values
constexpr int kSmem = 120 * 1024;  // more than half an SM: the two CTAs sit on two SMs
constexpr uint32_t kCols = 256;  // TMEM columns per CTA (D: 0..127, A of the TS form: 128..)

__host__ __device__ inline float a_val(int m, int k) { return (float)((m + 2 * k) % 5 - 2); }
__host__ __device__ inline float b_val(int n, int k) { return (float)((3 * n + k) % 7 - 3); }

__device__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ uint32_t ld_cluster_u32(uint32_t caddr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(caddr) : "memory");
    return v;
}
__device__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ void alloc_pair(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ void dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ void mma_pair_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ void mma_pair_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                            uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ void commit_pair(uint32_t bar_cluster_addr) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(
            bar_cluster_addr)
        : "memory");
}

// 16-bit value (m, k) of a K-major tile with 128-byte rows and the 128-byte swizzle.
__device__ void put(uint8_t* tile, int row, int k, float v) {
    const int off = row * 128 + ((((k >> 3) ^ (row & 7)) << 4)) + (k & 7) * 2;
    *reinterpret_cast<__nv_bfloat16*>(tile + off) = __float2bfloat16(v);
}

// ts = 0: D = A B^T with A from shared memory; ts = 1: A copied into tensor memory first.
// reps > 0: instead of one product, `reps` groups of 8 steps back to back, timed (cycles of the
// even CTA into *cycles).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    pair_kernel(int ts, int reps, float* out, int* status, long long* cycles) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                             ~uintptr_t(1023));
    uint8_t* a_tile = sm;                // 128 rows (this CTA's rows of A)
    uint8_t* b_tile = sm + 128 * 128;    // N / 2 rows (this CTA's rows of B)
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const uint32_t rank = cluster_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 128 * K; i += blockDim.x)
        put(a_tile, i / K, i % K, a_val((int)rank * 128 + i / K, i % K));
    for (int i = threadIdx.x; i < (N / 2) * K; i += blockDim.x)
        put(b_tile, i / K, i % K, b_val((int)rank * (N / 2) + i / K, i % K));
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    if (warp == 0) alloc_pair(&tbase, kCols);
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // both CTAs: operands written, barrier initialised, TMEM allocated
    tc_fence_after_sync();
    const uint32_t tm = tbase;
    const bool same = ld_cluster_u32(peer_addr(smem_u32(&tbase), rank ^ 1u)) == tm;
    if (same && ts) {  // A (this CTA's 128 rows x K) into TMEM columns 128.., two per column
        uint32_t w[32];
        const int row = warp * 32 + lane;
        for (int h = 0; h < K / 64; ++h) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                __nv_bfloat162 v;
                v.x = __float2bfloat16(a_val((int)rank * 128 + row, 64 * h + 2 * c));
                v.y = __float2bfloat16(a_val((int)rank * 128 + row, 64 * h + 2 * c + 1));
                w[c] = *reinterpret_cast<uint32_t*>(&v);
            }
            tmem_st32(tm + ((uint32_t)(warp * 32) << 16) + 128 + 32 * h, w);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncthreads();
        cluster_sync_all();  // both CTAs' A in TMEM before the even CTA issues
        tc_fence_after_sync();
    }
    long long t0 = 0;
    if (same && rank == 0 && warp == 0) {
        const uint32_t idesc = idesc_f16(true, 256, N, false, false);
        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(a_tile));
        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(b_tile));
        __syncwarp();
        t0 = clock64();
        const int groups = reps > 0 ? reps : 1;
        for (int g = 0; g < groups; ++g) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int k4 = kk & (K / 16 - 1);  // K / 16 = 4 distinct slices, repeated
                if (ts)
                    mma_pair_ts(tm, tm + 128 + k4 * 8, sdesc_advance(bd, k4 * 32), idesc,
                                (g | kk) ? 1u : 0u);
                else
                    mma_pair_ss(tm, sdesc_advance(ad, k4 * 32), sdesc_advance(bd, k4 * 32),
                                idesc, (g | kk) ? 1u : 0u);
                if (reps == 0 && kk == K / 16 - 1) break;  // the checked product: K = 64
            }
        }
        commit_pair(smem_u32(&bar));                  // this CTA
        commit_pair(peer_addr(smem_u32(&bar), 1u));   // the odd CTA
    }
    bool ok = same;
    if (same) {
        ok = wait_warp(&bar, 0, nullptr, kWaitNs);
        tc_fence_after_sync();
        if (rank == 0 && warp == 0 && lane == 0 && reps > 0) *cycles = clock64() - t0;
        if (ok && reps == 0) {
            const int row = warp * 32 + lane;
            for (int c = 0; c < N; c += 32) {
                uint32_t r[32];
                tmem_ld32(tm + ((uint32_t)(warp * 32) << 16) + c, r);
                for (int i = 0; i < 32; ++i)
                    out[((int)rank * 128 + row) * N + c + i] = __uint_as_float(r[i]);
            }
        }
    }
    if (!ok && lane == 0) atomicOr(status, same ? 2 : 1);
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // both CTAs done with the pair's TMEM
    if (warp == 0) {
        tc_fence_after_sync();
        dealloc_pair(tm, kCols);
    }
}

}  // namespace

int main() {
    float* d_out = nullptr;
    int* d_status = nullptr;
    long long* d_cycles = nullptr;
    if (cudaMalloc(&d_out, 256 * N * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&d_status, sizeof(int)) != cudaSuccess ||
        cudaMalloc(&d_cycles, sizeof(long long)) != cudaSuccess)
        return 1;
    if (cudaFuncSetAttribute(pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess)
        return 1;
    std::vector<float> ref(256 * N);
    for (int m = 0; m < 256; ++m)
        for (int n = 0; n < N; ++n) {
            float s = 0.f;
            for (int k = 0; k < K; ++k) s += a_val(m, k) * b_val(n, k);
            ref[m * N + n] = s;
        }
    bool all_ok = true;
    std::printf("{");
    for (int ts = 0; ts < 2; ++ts) {
        cudaMemset(d_out, 0xff, 256 * N * sizeof(float));
        cudaMemset(d_status, 0, sizeof(int));
        pair_kernel<<<2, 128, kSmem>>>(ts, 0, d_out, d_status, d_cycles);
        const cudaError_t e = cudaDeviceSynchronize();
        std::vector<float> h(256 * N);
        int status = -1;
        cudaMemcpy(h.data(), d_out, h.size() * sizeof(float), cudaMemcpyDeviceToHost);
        cudaMemcpy(&status, d_status, sizeof(int), cudaMemcpyDeviceToHost);
        int bad = 0;
        for (size_t i = 0; i < h.size(); ++i) bad += h[i] != ref[i];
        const bool ok = e == cudaSuccess && status == 0 && bad == 0;
        all_ok &= ok;
        std::printf("%s\"%s\": {\"cuda\": \"%s\", \"status\": %d, \"mismatches\": %d}", ts ? ", " : "",
                    ts ? "ts" : "ss", cudaGetErrorString(e), status, bad);
        if (e != cudaSuccess) break;
    }
    const int reps = 256;
    for (int ts = 0; ts < 2 && all_ok; ++ts) {
        cudaMemset(d_status, 0, sizeof(int));
        pair_kernel<<<2, 128, kSmem>>>(ts, reps, d_out, d_status, d_cycles);
        long long cyc = -1;
        int status = -1;
        const cudaError_t e = cudaDeviceSynchronize();
        cudaMemcpy(&cyc, d_cycles, sizeof(cyc), cudaMemcpyDeviceToHost);
        cudaMemcpy(&status, d_status, sizeof(int), cudaMemcpyDeviceToHost);
        all_ok &= e == cudaSuccess && status == 0;
        std::printf(", \"%s_pair_M256_N128_cycles_per_step\": %.1f", ts ? "ts" : "ss",
                    (double)cyc / (reps * 8.0));
    }
    std::printf(", \"ok\": %s}\n", all_ok ? "true" : "false");
    cudaFree(d_out);
    cudaFree(d_status);
    cudaFree(d_cycles);
    return all_ok ? 0 : 2;
}
