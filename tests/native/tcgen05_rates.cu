// tcgen05_rates.cu -- microbenchmarks of the per-SM rates the attention kernels are laid out
// around, on one GB300 (sm_103a): tcgen05.mma kind::f16 (bf16, M = 128, K = 16 per step) with
// both operands in shared memory (SS) or A in tensor memory (TS) at N = 64, 128, 256; the
// latency of one 8-step group issued to an idle pipe; the latency of a thread's mbarrier
// arrive as seen by a waiting warp; and the issue rates of the elementwise instructions the
// softmax uses (ex2.approx, fma.rn.f32x2, cvt to bf16x2).
//
// One CTA per SM (the dynamic shared-memory request leaves room for one), every SM measuring
// its own clock64 cycles; the median over SMs is printed.  Shared-memory operands are zeros
// and the TS A operand is whatever the tensor memory holds: the rates do not depend on the
// values.  Every wait is bounded (2 s); a CTA that gives up reports it and the program exits
// non-zero.  Output: one JSON object on stdout.
//
// Build and run:  nvcc -std=c++17 -gencode arch=compute_103a,code=sm_103a -O3 \
//                     tests/native/tcgen05_rates.cu -o tcgen05_rates && ./tcgen05_rates
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <vector>

#include "../../tiled_attention_08_gb300/csrc/fa_ptx.cuh"

using namespace fa;

namespace {

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kSmemRequest = 160 * 1024;   // > half of an SM: one CTA per SM
constexpr int kAChunk = 128 * 128;         // 128 rows x 128 B (64 K elements)
constexpr int kBChunk = 256 * 128;         // up to 256 rows x 128 B

struct Out {
    long long cycles;  // best repetition
    int ok;
};

__device__ uint8_t* aligned_smem(uint8_t* raw) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                      ~uintptr_t(1023));
}

// `reps` repetitions of `groups` groups of 8 MMA steps (K = 128) into one accumulator, each
// repetition timed from its first issue to the completion its commit signals.
template <bool TS>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int n, int groups, int reps, Out* out) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = aligned_smem(raw);
    uint8_t* a = sm;
    uint8_t* b = sm + 2 * kAChunk;
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (2 * kAChunk + 2 * kBChunk) / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(sm)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&tbase, 512);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // zeros visible to the MMA
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = tbase;
    if (warp == 0) {
        const uint32_t idesc = idesc_f16(true, 128, n, false, false);
        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(a));
        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(b));
        long long best = -1;
        bool ok = true;
        for (int r = 0; r < reps && ok; ++r) {
            __syncwarp();
            const long long t0 = clock64();
            for (int g = 0; g < groups; ++g) {
#pragma unroll
                for (int kc = 0; kc < 2; ++kc) {
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint32_t acc = (g | kc | s) ? 1u : 0u;
                        const uint64_t bs = sdesc_advance(bd, kc * kBChunk + s * 32);
                        if (TS)
                            mma_ts_w(tm, tm + 256 + (kc * 4 + s) * 8, bs, idesc, acc);
                        else
                            mma_ss_w(tm, sdesc_advance(ad, kc * kAChunk + s * 32), bs, idesc,
                                     acc);
                    }
                }
            }
            mma_commit_w(&bar);
            ok = wait_warp(&bar, (uint32_t)r & 1u, nullptr, kWaitNs);
            const long long t1 = clock64();
            if (r > 0 && (best < 0 || t1 - t0 < best)) best = t1 - t0;
        }
        if ((threadIdx.x & 31) == 0) out[blockIdx.x] = {best, ok ? 1 : 0};
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tm, 512);
    }
}

// Warp 1 waits on an mbarrier; warp 0 reads the clock and arrives.  The cycles from that
// clock read to warp 1's return from the wait, best of `reps`.
__global__ void __launch_bounds__(64, 1) arrive_latency_kernel(int reps, Out* out) {
    __shared__ uint64_t bar;
    __shared__ long long t_arrive;
    __shared__ int ready;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    long long best = -1;
    bool ok = true;
    for (int r = 0; r < reps && ok; ++r) {
        if (threadIdx.x == 0) ready = 0;
        __syncthreads();
        if (warp == 1) {
            if (lane == 0) atomicExch(&ready, 1);
            ok = wait_warp(&bar, (uint32_t)r & 1u, nullptr, kWaitNs);
            const long long t1 = clock64();
            __syncwarp();
            if (lane == 0 && ok) {
                const long long d = t1 - *(volatile long long*)&t_arrive;
                if (r > 0 && (best < 0 || d < best)) best = d;
            }
        } else if (lane == 0) {
            int spins = 0;
            while (atomicAdd(&ready, 0) == 0 && ++spins < (1 << 24)) {
            }
            for (int i = 0; i < 200; ++i) __nanosleep(10);  // the waiter is polling by now
            t_arrive = clock64();
            __threadfence_block();
            mbar_arrive(&bar);  // the waiter gives up after its own time limit otherwise
        }
        ok = __syncthreads_and(ok);
    }
    if (threadIdx.x == 32) out[blockIdx.x] = {best, ok ? 1 : 0};
}

// Issue rates of the softmax's elementwise instructions: 16 warps (4 per SMSP), 8 independent
// chains per thread.  Cycles for `iters` iterations.
template <int OP>
__global__ void __launch_bounds__(512, 1) alu_rate_kernel(int iters, float seed, Out* out,
                                                          float* sink) {
    float x[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = seed * (float)(threadIdx.x + c);
    uint64_t y[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) y[c] = f2_make(x[c], -x[c]);
    const uint64_t half2 = f2_make(0.5f, 0.5f), quarter2 = f2_make(0.25f, 0.25f);
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // one instruction per chain step; values stay bounded
            if (OP == 0) x[c] = ex2_approx(-x[c]);
            if (OP == 1) y[c] = f2_fma(y[c], half2, quarter2);
            if (OP == 2) x[c] = __uint_as_float(pack2<true>(x[c], x[c]));
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    float acc = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float lo, hi;
        f2_split(y[c], lo, hi);
        acc += x[c] + lo + hi;
    }
    if (acc == 12345.678f) sink[threadIdx.x] = acc;  // keeps the chains live
    if (threadIdx.x == 0) out[blockIdx.x] = {t1 - t0, 1};
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
}

bool check(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return true;
    std::fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return false;
}

// Median over SMs of the cycles each CTA reported; -1 when any CTA gave up.
double median_cycles(Out* d, int n) {
    std::vector<Out> h(n);
    if (!check(cudaMemcpy(h.data(), d, n * sizeof(Out), cudaMemcpyDeviceToHost), "copy"))
        return -1.0;
    std::vector<long long> c;
    for (const Out& o : h) {
        if (!o.ok || o.cycles < 0) return -1.0;
        c.push_back(o.cycles);
    }
    std::sort(c.begin(), c.end());
    return (double)c[c.size() / 2];
}

}  // namespace

int main() {
    const int n_sm = sm_count();
    Out* d_out = nullptr;
    float* d_sink = nullptr;
    if (!check(cudaMalloc(&d_out, n_sm * sizeof(Out)), "malloc") ||
        !check(cudaMalloc(&d_sink, 512 * sizeof(float)), "malloc"))
        return 1;
    if (!check(cudaFuncSetAttribute(mma_rate_kernel<false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemRequest),
               "attr") ||
        !check(cudaFuncSetAttribute(mma_rate_kernel<true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemRequest),
               "attr"))
        return 1;
    bool all_ok = true;
    std::printf("{\"sms\": %d", n_sm);
    const int groups = 256, reps = 4;
    for (int ts = 0; ts < 2; ++ts) {
        for (int n : {64, 128, 256}) {
            cudaMemset(d_out, 0xff, n_sm * sizeof(Out));
            if (ts)
                mma_rate_kernel<true><<<n_sm, 128, kSmemRequest>>>(n, groups, reps, d_out);
            else
                mma_rate_kernel<false><<<n_sm, 128, kSmemRequest>>>(n, groups, reps, d_out);
            if (!check(cudaDeviceSynchronize(), "mma_rate_kernel")) return 1;
            const double cyc = median_cycles(d_out, n_sm);
            all_ok &= cyc > 0;
            const double per_step = cyc / (groups * 8.0);
            // FLOP per step: 2 * M * N * K = 2 * 128 * n * 16
            std::printf(", \"%s_N%d_cycles_per_step\": %.1f, \"%s_N%d_flop_per_clk\": %.0f",
                        ts ? "ts" : "ss", n, per_step, ts ? "ts" : "ss", n,
                        2.0 * 128 * n * 16 / per_step);
        }
    }
    // one 8-step group (K = 128, N = 128, SS) issued to an idle pipe: issue to completion seen
    cudaMemset(d_out, 0xff, n_sm * sizeof(Out));
    mma_rate_kernel<false><<<n_sm, 128, kSmemRequest>>>(128, 1, 16, d_out);
    if (!check(cudaDeviceSynchronize(), "group latency")) return 1;
    const double lat = median_cycles(d_out, n_sm);
    all_ok &= lat > 0;
    std::printf(", \"ss_N128_group8_latency_cycles\": %.0f", lat);
    cudaMemset(d_out, 0xff, n_sm * sizeof(Out));
    arrive_latency_kernel<<<n_sm, 64>>>(16, d_out);
    if (!check(cudaDeviceSynchronize(), "arrive latency")) return 1;
    const double arr = median_cycles(d_out, n_sm);
    all_ok &= arr > 0;
    std::printf(", \"mbarrier_arrive_to_waiter_cycles\": %.0f", arr);
    const int iters = 4096;
    const char* names[3] = {"ex2_approx", "fma_f32x2", "cvt_bf16x2"};
    for (int op = 0; op < 3; ++op) {
        cudaMemset(d_out, 0xff, n_sm * sizeof(Out));
        if (op == 0) alu_rate_kernel<0><<<n_sm, 512>>>(iters, 1e-3f, d_out, d_sink);
        if (op == 1) alu_rate_kernel<1><<<n_sm, 512>>>(iters, 1e-3f, d_out, d_sink);
        if (op == 2) alu_rate_kernel<2><<<n_sm, 512>>>(iters, 1e-3f, d_out, d_sink);
        if (!check(cudaDeviceSynchronize(), "alu_rate_kernel")) return 1;
        const double cyc = median_cycles(d_out, n_sm);
        all_ok &= cyc > 0;
        // warp instructions per cycle per SMSP: 16 warps x iters x 8 over 4 SMSPs
        const double per_smsp = 16.0 * iters * 8 / 4.0 / cyc;
        std::printf(", \"%s_warp_instr_per_clk_per_smsp\": %.3f", names[op], per_smsp);
    }
    std::printf(", \"ok\": %s}\n", all_ok ? "true" : "false");
    cudaFree(d_out);
    cudaFree(d_sink);
    return all_ok ? 0 : 2;
}
