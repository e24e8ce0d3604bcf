// fa_bwd_pre.cu -- backward preprocess: Delta_i = sum_d dO_id * O_id and LSE_i * log2(e).
//
// The backward recomputes P from the saved log-sum-exp instead of storing it ("FlashAttention
// data-flow optimisation: MI50 memory and bandwidth bottlenecks", section 2.2, third layer).
// dS = P o (dP - Delta) needs one scalar per query row, Delta_i = rowsum(P o dP), which equals
// rowsum(dO o O) because O = P V; this kernel computes it from O and dO in one streaming pass.
// Both per-row vectors go to a workspace padded to a whole number of 128-row tiles (zeros past
// Lq), so the backward kernels can copy them tile by tile with aligned bulk copies.  Rows that
// see no key (the first Lq - Lk queries under the causal mask when Lq > Lk) get dQ = 0 here;
// the dQ pass skips query tiles in which no row sees a key.  When dQ is reduced into an fp32
// accumulator by the dK/dV pass instead, this kernel zeroes the accumulator's rows (all Lqpad
// of them) as it goes, and it zeroes the work counters of the persistent passes that follow.
//
// HBM-bound: every (row, D) element of O and dO is read once, with 16-byte loads; D/8 threads
// share a row and reduce with shuffles.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Block (x, y) covers 128-row tile x of heads y, y + gridDim.y, ...: the head's base addresses
// are worked out once per block, so a row costs one multiply-add per operand, and the block's
// threads walk the tile in passes of 256/G rows, one row per thread per pass.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdPreParams p) {
    constexpr int G = D / 8;                   // threads per row (8 elements each)
    constexpr int kRowsPerPass = 256 / G;
    const int g = threadIdx.x % G;
    const int i0 = blockIdx.x * kTileRows + threadIdx.x / G;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < kSchedCounters) p.sched[threadIdx.x] = 0;
    for (int bh = blockIdx.y; bh < p.BH; bh += gridDim.y) {
        const uint8_t* o_head =
            reinterpret_cast<const uint8_t*>(p.o) + row_offset(p.so, bh, p.H, 0) + g * 16;
        const uint8_t* d_head =
            reinterpret_cast<const uint8_t*>(p.dout) + row_offset(p.sdo, bh, p.H, 0) + g * 16;
        uint8_t* q_head = reinterpret_cast<uint8_t*>(p.dq) + row_offset(p.sdq, bh, p.H, 0) + g * 16;
        float* acc_head = p.dq_acc ? p.dq_acc + (size_t)bh * p.Lqpad * D + g * 8 : nullptr;
        const size_t o_step = (size_t)p.so.l * 2u, d_step = (size_t)p.sdo.l * 2u;
#pragma unroll 2
        for (int pass = 0; pass < kTileRows / kRowsPerPass; ++pass) {
            const int i = i0 + pass * kRowsPerPass;
            if (acc_head) {  // i < Lqpad always: the grid covers the padded tiles
                float4* z = reinterpret_cast<float4*>(acc_head + (size_t)i * D);
                z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float acc = 0.0f;
            if (i < p.Lq) {
                const uint4 a = *reinterpret_cast<const uint4*>(o_head + (size_t)i * o_step);
                const uint4 b = *reinterpret_cast<const uint4*>(d_head + (size_t)i * d_step);
                if (i < p.first_seen_row)
                    *reinterpret_cast<uint4*>(q_head + (size_t)i * (size_t)p.sdq.l * 2u) =
                        make_uint4(0u, 0u, 0u, 0u);
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
#pragma unroll
            for (int w = G / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w, G);
            if (g == 0) {
                const size_t row = (size_t)bh * p.Lqpad + i;
                p.delta_pad[row] = acc;
                p.nlse2_pad[row] = (i < p.Lq) ? -(p.lse[(size_t)bh * p.Lq + i] * kLog2e) : 0.0f;
            }
        }
    }
}

template <int D, bool BF16>
cudaError_t launch_t(const BwdPreParams& p, cudaStream_t s) {
    const unsigned tiles = (unsigned)(p.Lqpad / kTileRows);
    const unsigned heads = p.BH < 65535 ? (unsigned)p.BH : 65535u;
    return launch_kernel(fa_bwd_pre_kernel<D, BF16>, dim3(tiles, heads), dim3(256), 0, s, p);
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t s) {
    if (p.D == 64) return p.bf16 ? launch_t<64, true>(p, s) : launch_t<64, false>(p, s);
    return p.bf16 ? launch_t<128, true>(p, s) : launch_t<128, false>(p, s);
}

}  // namespace fa
