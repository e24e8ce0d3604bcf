// fa_bwd_pre.cu -- backward preprocess: Delta_i = sum_d dO_id * O_id and LSE_i * log2(e).
//
// The backward recomputes P from the saved log-sum-exp instead of storing it ("FlashAttention
// data-flow optimisation: MI50 memory and bandwidth bottlenecks", section 2.2, third layer).
// dS = P o (dP - Delta) needs one scalar per query row, Delta_i = rowsum(P o dP), which equals
// rowsum(dO o O) because O = P V; this kernel computes it from O and dO in one streaming pass.
// Both per-row vectors go to a workspace padded to a whole number of 128-row tiles (zeros past
// L), so the backward kernels can copy them tile by tile with aligned bulk copies.
//
// HBM-bound: every (row, D) element of O and dO is read once, with 16-byte loads; D/8 threads
// share a row and reduce with shuffles.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdPreParams p) {
    constexpr int G = D / 8;              // threads per row (8 elements each)
    constexpr int kRowsPerBlock = 256 / G;
    const int g = threadIdx.x % G;
    const long long total = (long long)p.BH * p.Lpad;
    const long long stride = (long long)gridDim.x * kRowsPerBlock;
    for (long long base = (long long)blockIdx.x * kRowsPerBlock; base < total; base += stride) {
        const long long row = base + threadIdx.x / G;  // uniform loop trip count per warp
        float acc = 0.0f;
        int bh = 0, i = 0;
        if (row < total) {
            bh = (int)(row / p.Lpad);
            i = (int)(row % p.Lpad);
            if (i < p.L) {
                const size_t off = ((size_t)bh * p.L + i) * D + g * 8;
                const uint4 a = *reinterpret_cast<const uint4*>(
                    reinterpret_cast<const uint8_t*>(p.o) + off * 2);
                const uint4 b = *reinterpret_cast<const uint4*>(
                    reinterpret_cast<const uint8_t*>(p.dout) + off * 2);
                const uint32_t av[4] = {a.x, a.y, a.z, a.w};
                const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 x = unpack2<BF16>(av[t]);
                    const float2 y = unpack2<BF16>(bv[t]);
                    acc = fmaf(x.x, y.x, acc);
                    acc = fmaf(x.y, y.y, acc);
                }
            }
        }
#pragma unroll
        for (int w = G / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w, G);
        if (g == 0 && row < total) {
            p.delta_pad[row] = acc;
            p.nlse2_pad[row] = (i < p.L) ? -(p.lse[(size_t)bh * p.L + i] * kLog2e) : 0.0f;
        }
    }
}

template <int D, bool BF16>
cudaError_t launch_t(const BwdPreParams& p, cudaStream_t s) {
    constexpr int kRowsPerBlock = 256 / (D / 8);
    const long long total = (long long)p.BH * p.Lpad;
    long long blocks = (total + kRowsPerBlock - 1) / kRowsPerBlock;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    fa_bwd_pre_kernel<D, BF16><<<(unsigned)blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t s) {
    if (p.D == 64) return p.bf16 ? launch_t<64, true>(p, s) : launch_t<64, false>(p, s);
    return p.bf16 ? launch_t<128, true>(p, s) : launch_t<128, false>(p, s);
}

}  // namespace fa
