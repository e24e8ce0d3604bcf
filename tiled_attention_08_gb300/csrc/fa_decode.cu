// fa_decode.cu -- one decode step over a paged key/value cache (sm_103a).
//
// Serving ("FlashAttention principles and engineering practice", section 4.2: vLLM with
// PagedAttention, block_size 16, continuous batching): each sequence b adds one token, whose
// query row q[b, h] attends to all seq_lens[b] cached tokens of its head.  The cache is paged:
// token t of sequence b lives in physical page block_tables[b][t / 16] at slot t % 16.  The
// result is the plain definition with one query row: O = softmax(scale * q K^T) V and
// LSE = log sum exp(scale * q K^T); a sequence with no cached token gets O = 0, LSE = -inf.
//
// GB300 design.  One query row against a stream of keys is a matrix-vector product: 2 FLOPs per
// byte of K and V read, far below the tensor cores' ridge, so the step is bound by HBM and the
// kernel does the arithmetic on the FMA pipes.  Cache layout [num_pages, H, 16, D]: the 16 tokens
// of one head in one page are one contiguous chunk (4 KB at D = 128), fetched by a single bulk
// copy into a shared-memory ring.  CTA = one (sequence, head, split): a producer warp issues the
// copies (validating every page index first), four compute warps take 4 tokens of each page
// each and keep their own online softmax (running max, running sum and a D/32-element slice of
// the output per lane, in the log2 domain), and at the end the four partial results are merged
// in shared memory.  When there are too few (sequence, head) pairs to fill the GPU, the page
// range is split across CTAs and a small combine kernel merges the splits' (O, LSE).
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct DecCfg {
    static constexpr int kChunk = kPageTokens * D * 2;    // bytes of one head's page
    static constexpr int kStages = (D == 128) ? 6 : 8;    // ring depth (pages in flight)
    static constexpr int kComputeWarps = 4;
    static constexpr int kTokPerWarp = kPageTokens / kComputeWarps;
    static constexpr int kThreads = (kComputeWarps + 1) * 32;
    static constexpr int kPer = D / 32;                   // D elements per lane
    static constexpr int kSmemBytes = kStages * 2 * kChunk;
};

// kPer 16-bit values at `src` (kPer * 2 bytes, aligned) as fp32.
template <bool BF16, int N>
__device__ __forceinline__ void load_row16(const uint8_t* src, float (&out)[N]) {
    static_assert(N == 2 || N == 4, "2 or 4 elements per lane");
    if constexpr (N == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        const float2 a = unpack2<BF16>(u.x), b = unpack2<BF16>(u.y);
        out[0] = a.x;
        out[1] = a.y;
        out[2] = b.x;
        out[3] = b.y;
    } else {
        const float2 a = unpack2<BF16>(*reinterpret_cast<const uint32_t*>(src));
        out[0] = a.x;
        out[1] = a.y;
    }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(DecCfg<D>::kThreads) fa_decode_kernel(const DecodeParams p) {
    using C = DecCfg<D>;
    extern __shared__ __align__(128) uint8_t ring[];  // stage s: K page, then V page
    __shared__ uint64_t bar_full[C::kStages], bar_empty[C::kStages];
    __shared__ float red_m[C::kComputeWarps], red_l[C::kComputeWarps];
    __shared__ float red_o[C::kComputeWarps][D];
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The sequence's cached tokens (device data: checked here; a bad length counts as empty).
    int n = p.seq_lens[b];
    if (n < 0 || n > p.max_pages * kPageTokens) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, (int)kDevBadArg);
        n = 0;
    }
    const int n_pages = (n + kPageTokens - 1) / kPageTokens;
    const int pg0 = split * p.pages_per_split;
    const int pg1 = min(n_pages, pg0 + p.pages_per_split);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], C::kComputeWarps);
        }
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == C::kComputeWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int pg = pg0; pg < pg1; ++pg) {
                const int i = pg - pg0, st = i % C::kStages;
                if (i >= C::kStages &&
                    !wait_bounded(&bar_empty[st], ((uint32_t)(i / C::kStages) & 1u) ^ 1u, abort_v,
                                  p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const int phys = p.block_tables[(size_t)b * p.max_pages + pg];
                if (phys < 0 || phys >= p.num_pages) {  // never copy from outside the cache
                    atomicCAS(p.status, 0, (int)kDevBadArg);
                    *abort_v = 1;
                    break;
                }
                const size_t off = ((size_t)phys * p.H + h) * (size_t)C::kChunk;
                mbar_arrive_expect_tx(&bar_full[st], 2 * C::kChunk);
                bulk_load(ring + (2 * st) * C::kChunk,
                          reinterpret_cast<const uint8_t*>(p.k_cache) + off, C::kChunk,
                          &bar_full[st]);
                bulk_load(ring + (2 * st + 1) * C::kChunk,
                          reinterpret_cast<const uint8_t*>(p.v_cache) + off, C::kChunk,
                          &bar_full[st]);
                issued = i + 1;
            }
            if (!ok) record_timeout(p.status, abort_v);
            // Drain: no copy may still be landing when the CTA exits.
            for (int i = issued - 1; i >= 0 && i >= issued - C::kStages; --i)
                wait_bounded(&bar_full[i % C::kStages], (uint32_t)(i / C::kStages) & 1u, nullptr,
                             p.timeout_ns);
        }
    } else {
        // ------------------------------ compute warps ------------------------------
        // This lane's slice of q, scaled into the log2 domain: s2 = (q . k) * scale * log2(e).
        float qv[C::kPer];
        load_row16<BF16, C::kPer>(reinterpret_cast<const uint8_t*>(p.q) +
                                      ((size_t)(b * p.H + h) * D + lane * C::kPer) * 2,
                                  qv);
#pragma unroll
        for (int e = 0; e < C::kPer; ++e) qv[e] *= p.scale_log2;
        float m = -INFINITY, l = 0.0f, o[C::kPer];
#pragma unroll
        for (int e = 0; e < C::kPer; ++e) o[e] = 0.0f;
        for (int pg = pg0; pg < pg1; ++pg) {
            const int i = pg - pg0, st = i % C::kStages;
            if (!wait_warp(&bar_full[st], (uint32_t)(i / C::kStages) & 1u, abort_v, p.timeout_ns))
                break;
            const uint8_t* kp = ring + (2 * st) * C::kChunk;
            const uint8_t* vp = kp + C::kChunk;
            float s[C::kTokPerWarp];
#pragma unroll
            for (int tt = 0; tt < C::kTokPerWarp; ++tt) {
                const int t = warp * C::kTokPerWarp + tt;
                float kv[C::kPer];
                load_row16<BF16, C::kPer>(kp + (t * D + lane * C::kPer) * 2, kv);
                float d = 0.0f;
#pragma unroll
                for (int e = 0; e < C::kPer; ++e) d = fmaf(qv[e], kv[e], d);
                s[tt] = d;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int tt = 0; tt < C::kTokPerWarp; ++tt)
                    s[tt] += __shfl_xor_sync(0xffffffffu, s[tt], off);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int tt = 0; tt < C::kTokPerWarp; ++tt) {
                const int token = pg * kPageTokens + warp * C::kTokPerWarp + tt;
                if (token >= n) s[tt] = -INFINITY;  // past the sequence's last token
                mx = fmaxf(mx, s[tt]);
            }
            const float m_new = fmaxf(m, mx);
            if (m_new != -INFINITY) {  // (all of this warp's tokens so far may be masked)
                const float alpha = (m == -INFINITY) ? 0.0f : ex2_approx(m - m_new);
                float pr[C::kTokPerWarp], psum = 0.0f;
#pragma unroll
                for (int tt = 0; tt < C::kTokPerWarp; ++tt) {
                    pr[tt] = ex2_approx(s[tt] - m_new);
                    psum += pr[tt];
                }
                l = l * alpha + psum;
#pragma unroll
                for (int e = 0; e < C::kPer; ++e) o[e] *= alpha;
#pragma unroll
                for (int tt = 0; tt < C::kTokPerWarp; ++tt) {
                    const int t = warp * C::kTokPerWarp + tt;
                    float vv[C::kPer];
                    load_row16<BF16, C::kPer>(vp + (t * D + lane * C::kPer) * 2, vv);
#pragma unroll
                    for (int e = 0; e < C::kPer; ++e) o[e] = fmaf(pr[tt], vv[e], o[e]);
                }
                m = m_new;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_empty[st]);  // this warp is done with the stage
        }
        // Merge the four warps' partial results.
        if (lane == 0) {
            red_m[warp] = m;
            red_l[warp] = l;
        }
#pragma unroll
        for (int e = 0; e < C::kPer; ++e) red_o[warp][lane * C::kPer + e] = o[e];
        asm volatile("bar.sync 1, %0;" ::"r"(C::kComputeWarps * 32) : "memory");
        const int tid = threadIdx.x;
        if (tid < D) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::kComputeWarps; ++w) M = fmaxf(M, red_m[w]);
            float L = 0.0f, O = 0.0f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < C::kComputeWarps; ++w) {
                    const float f = (red_m[w] == -INFINITY) ? 0.0f : ex2_approx(red_m[w] - M);
                    L = fmaf(red_l[w], f, L);
                    O = fmaf(red_o[w][tid], f, O);
                }
            }
            const float out = L > 0.0f ? O / L : 0.0f;
            const float lse2 = L > 0.0f ? M + log2f(L) : -INFINITY;  // log2 domain
            const size_t row = (size_t)b * p.H + h;
            if (p.splits == 1) {
                uint16_t* dst = reinterpret_cast<uint16_t*>(p.o) + row * D + tid;
                const uint32_t pk = pack2<BF16>(out, 0.0f);
                *dst = (uint16_t)(pk & 0xffffu);
                if (tid == 0) p.lse[row] = lse2 * kLn2;
            } else {
                const size_t part = row * p.splits + split;
                p.part_o[part * D + tid] = out;
                if (tid == 0) p.part_lse[part] = lse2;
            }
        }
    }
    __syncthreads();
}

// Merges the splits of each (sequence, head): O = sum_s w_s O_s / sum_s w_s and
// LSE = log sum_s exp(LSE_s), with w_s = 2^(LSE2_s - max).  Splits past a sequence's pages carry
// LSE = -inf and weigh nothing; a sequence with no token gets O = 0, LSE = -inf.
template <int D, bool BF16>
__global__ void __launch_bounds__(D) fa_decode_combine_kernel(const DecodeParams p) {
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const size_t row = (size_t)b * p.H + h;
    const size_t base = row * p.splits;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, p.part_lse[base + s]);
    float W = 0.0f, O = 0.0f;
    if (M != -INFINITY) {
        for (int s = 0; s < p.splits; ++s) {
            const float l2 = p.part_lse[base + s];
            const float w = (l2 == -INFINITY) ? 0.0f : ex2_approx(l2 - M);
            W += w;
            O = fmaf(w, p.part_o[(base + s) * D + tid], O);
        }
    }
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.o) + row * D + tid;
    *dst = (uint16_t)(pack2<BF16>(W > 0.0f ? O / W : 0.0f, 0.0f) & 0xffffu);
    if (tid == 0) p.lse[row] = W > 0.0f ? (M + log2f(W)) * kLn2 : -INFINITY;
}

template <int D, bool BF16>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t s) {
    using C = DecCfg<D>;
    auto kern = fa_decode_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = launch_kernel(kern, dim3((unsigned)p.splits, (unsigned)p.H, (unsigned)p.B),
                      dim3(C::kThreads), C::kSmemBytes, s, p);
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_kernel(fa_decode_combine_kernel<D, BF16>, dim3((unsigned)p.H, (unsigned)p.B),
                         dim3(D), 0, s, p);
}

}  // namespace

int decode_splits(int B, int H, int max_pages) {
    // Enough CTAs for about four per SM of a 152-SM part (a fixed target, so that the workspace
    // size does not depend on the device); never more splits than pages.
    const long long units = (long long)B * H;
    const long long target = 4LL * 152;
    if (units <= 0 || units >= target || max_pages <= 1) return 1;
    long long splits = (target + units - 1) / units;
    if (splits > max_pages) splits = max_pages;
    const int per = (int)((max_pages + splits - 1) / splits);
    return (max_pages + per - 1) / per;  // splits that each hold at least one page
}

cudaError_t launch_decode(const DecodeParams& p, int D, bool bf16, cudaStream_t s) {
    if (D == 64) return bf16 ? launch_t<64, true>(p, s) : launch_t<64, false>(p, s);
    return bf16 ? launch_t<128, true>(p, s) : launch_t<128, false>(p, s);
}

}  // namespace fa
