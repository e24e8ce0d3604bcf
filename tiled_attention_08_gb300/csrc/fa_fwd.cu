// fa_fwd.cu -- fused attention forward for sm_103a (TMA + tcgen05/TMEM, online softmax).
//
// Method ("FlashAttention data-flow optimisation: MI50 memory and bandwidth bottlenecks",
// section 2.2): Q is split into 128-row tiles that stay on chip; K/V stream through shared
// memory in 128-key tiles; each row keeps a running max and a running sum of exponentials
// while the tiles arrive, the partial output is rescaled when the max grows, and only O and
// the per-row statistics (folded into one log-sum-exp) are written.  QK^T, the softmax and
// PV run in this one kernel ("FlashAttention principles and engineering practice",
// section 1, kernel fusion), so S and P never reach global memory.
//
// CTA roles (one CTA per (b*h, query tile)), with kSplit softmax warps per TMEM lane quadrant:
//   warps 0 .. 4*kSplit-1  softmax: warp w owns TMEM lanes 32*(w%4).. (query rows) and the
//              key columns [kCols*(w/4), +kCols) of each S tile (kCols = 128/kSplit); the
//              kSplit warps sharing a lane quadrant combine their partial row maxima through
//              shared memory at a named barrier;
//   next warp  TMA producer of Q (once) and the K_j ring;
//   next warp  MMA issuer (one thread) and TMEM owner;
//   last warp  TMA producer of the V_j ring (V_j is consumed a softmax later than K_j, so the
//              two rings advance independently and K runs further ahead).
// TMEM columns: S double buffer at [0,128) and [128,256) (fp32); the 16-bit P of a tile
// overwrites the first 64 columns of its S buffer and feeds the PV MMA straight from TMEM;
// O (fp32, D columns) at [256, 256+D).
//
// Online softmax in the log2 domain: y = s * scale * log2(e).  The running reference max m
// is only raised when a tile's max exceeds it by more than kRescaleThreshold (2^8 headroom
// for P), so O is rescaled rarely; the result is unchanged because O and the running sum
// always share the same reference.  LSE = (m + log2(l)) * ln(2).
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, bool BF16, bool CAUSAL>
struct FwdCfg {
    static constexpr int kChunks = D / kChunkElems;            // swizzle boxes per tile row
    static constexpr int kTileBytes = kTileRows * D * 2;       // one 128 x D tile
    static constexpr int kKStages = (D == 128) ? 3 : 4;        // K ring depth
    static constexpr int kVStages = (D == 128) ? 2 : 4;        // V ring depth
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kSmemBytes = kOffV + kVStages * kTileBytes + 1024;  // + alignment slack
    static constexpr int kSplit = 4;                          // softmax warps per lane quadrant
    static constexpr int kSoftmaxWarps = 4 * kSplit;
    static constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
    static constexpr int kProducerWarp = kSoftmaxWarps;
    static constexpr int kMmaWarp = kSoftmaxWarps + 1;
    static constexpr int kVProducerWarp = kSoftmaxWarps + 2;
    static constexpr int kThreads = (kSoftmaxWarps + 3) * 32;
    static constexpr int kCols = 128 / kSplit;                // S columns per softmax warp
    static constexpr int kOCols = D / kSplit;                 // O columns per softmax warp
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmS = 0;    // S buffer b at kTmS + 128*b
    static constexpr uint32_t kTmO = 256;  // O accumulator
    static constexpr uint32_t kIdescS = idesc_f16(BF16, 128, 128, false, false);
    static constexpr uint32_t kIdescO = idesc_f16(BF16, 128, D, false, true);
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(FwdCfg<D, BF16, CAUSAL>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = FwdCfg<D, BF16, CAUSAL>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ uint64_t bar_q, bar_kf[C::kKStages], bar_ke[C::kKStages], bar_vf[C::kVStages],
        bar_ve[C::kVStages], bar_sf[2], bar_pf[2], bar_od, bar_oready, bar_fin;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ float red_max[2][C::kSplit][128];  // [tile parity][column slice][row]
    __shared__ float red_sum[C::kSplit][128];     // [column slice][row]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Heads in L2-sized groups; inside a group the heaviest query tiles (most key tiles under
    // the causal mask) go first.
    int bh, rank;
    tile_coords(blockIdx.x, p.BH, p.n_tiles, p.group, bh, rank);
    const int qt = p.n_tiles - 1 - rank;
    const int n_kv = CAUSAL ? (qt + 1) : p.n_tiles;
    volatile int* abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar_q, 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&bar_kf[s], 1);
            mbar_init(&bar_ke[s], 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(&bar_vf[s], 1);
            mbar_init(&bar_ve[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar_sf[b], 1);
            mbar_init(&bar_pf[b], C::kSoftmaxThreads);
        }
        mbar_init(&bar_od, 1);
        mbar_init(&bar_oready, 1);
        mbar_init(&bar_fin, 1);
        mbar_fence_init();
    }
    if (warp == C::kMmaWarp) tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    if (warp == C::kProducerWarp || warp == C::kVProducerWarp) {
        // ------------------------------ TMA producers ------------------------------
        // One ring per warp: Q + K on kProducerWarp, V on kVProducerWarp.
        if (lane == 0) {
            const bool is_k = warp == C::kProducerWarp;
            const CUtensorMap* map = is_k ? &p.tm_k : &p.tm_v;
            const int stages = is_k ? C::kKStages : C::kVStages;
            uint64_t* full = is_k ? bar_kf : bar_vf;
            uint64_t* empty = is_k ? bar_ke : bar_ve;
            uint8_t* ring = smem + (is_k ? C::kOffK : C::kOffV);
            tma_prefetch_desc(map);
            if (is_k) {
                tma_prefetch_desc(&p.tm_q);
                mbar_arrive_expect_tx(&bar_q, C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(smem + C::kOffQ + c * kChunkBytes, &p.tm_q, &bar_q,
                                c * kChunkElems, qt * kTileRows, bh);
            }
            bool ok = true;
            int issued = 0;  // fills handed to the TMA unit
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % stages;
                const uint32_t ph = (uint32_t)(j / stages) & 1u;
                if (j >= stages && !wait_bounded(&empty[st], ph ^ 1u, abort_v, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[st], C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(ring + st * C::kTileBytes + c * kChunkBytes, map, &full[st],
                                c * kChunkElems, j * kTileRows, bh);
                issued = j + 1;
            }
            if (!ok) record_timeout(p.status, abort_v);
            // Drain: the newest fill of every stage must have landed before the CTA exits.
            // (These waits return at once on the normal path.)
            if (is_k) wait_bounded(&bar_q, 0, nullptr, p.timeout_ns);
            for (int j = issued - 1; j >= 0 && j >= issued - stages; --j)
                wait_bounded(&full[j % stages], (uint32_t)(j / stages) & 1u, nullptr, p.timeout_ns);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            const uint32_t q_base = smem_u32(smem + C::kOffQ);
            bool ok = wait_bounded(&bar_q, 0, abort_v, p.timeout_ns);
            auto issue_pv = [&](int jj) -> bool {
                const int b = jj & 1;
                const int st = jj % C::kVStages;
                const uint32_t ph = (uint32_t)(jj / C::kVStages) & 1u;
                if (!wait_bounded(&bar_pf[b], (uint32_t)(jj >> 1) & 1u, abort_v, p.timeout_ns))
                    return false;
                if (!wait_bounded(&bar_vf[st], ph, abort_v, p.timeout_ns)) return false;
                tc_fence_after_sync();
                const uint32_t v_base = smem_u32(smem + C::kOffV + st * C::kTileBytes);
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk) {
                    const uint64_t bd = sdesc_mnmajor_sw128(v_base + kk * 2048, kChunkBytes);
                    mma_ts(tmem + C::kTmO, tmem + C::kTmS + 128 * b + kk * 8, bd, C::kIdescO,
                           (jj > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bar_ve[st]);
                mma_commit(&bar_od);
                return true;
            };
            for (int j = 0; j < n_kv && ok; ++j) {
                const int st = j % C::kKStages;
                const uint32_t ph = (uint32_t)(j / C::kKStages) & 1u;
                const int b = j & 1;
                if (!wait_bounded(&bar_kf[st], ph, abort_v, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t k_base = smem_u32(smem + C::kOffK + st * C::kTileBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    mma_ss(tmem + C::kTmS + 128 * b, sdesc_kmajor_sw128(q_base + off),
                           sdesc_kmajor_sw128(k_base + off), C::kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar_ke[st]);
                mma_commit(&bar_sf[b]);
                if (j > 0 && !issue_pv(j - 1)) ok = false;
            }
            if (ok && n_kv > 0 && !issue_pv(n_kv - 1)) ok = false;
            // O is final once every PV has completed.  The epilogue cannot use bar_od for
            // this: S_{n-1} is issued before PV_{n-2}, so when the softmax finishes the last
            // tile bar_od may still be two phases short, and its parity cannot tell n-2 from n.
            if (ok) mma_commit(&bar_oready);
            if (!ok) record_timeout(p.status, abort_v);
            // Every issued MMA must finish before TMEM is released.
            mma_commit(&bar_fin);
            wait_bounded(&bar_fin, 0, nullptr, p.timeout_ns);
        }
    } else {
        // ------------------------------ softmax warps ------------------------------
        constexpr int kC = C::kCols;
        const int quad = warp & 3;                       // TMEM lane quadrant
        const int part = warp >> 2;                      // which kC key columns of the tile
        const uint32_t grp_bar = 1 + quad;               // named barrier of the quadrant
        constexpr uint32_t kGrpThreads = 32 * C::kSplit;
        const int row = quad * 32 + lane;                // row inside the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int q_row = qt * kTileRows + row;
        const int c0 = part * kC;
        float m_ref = -INFINITY;
        float l_sum = 0.0f;  // over this warp's columns only
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int b = j & 1;
            ok = wait_bounded(&bar_sf[b], (uint32_t)(j >> 1) & 1u, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            const uint32_t s_addr = tmem + lane_off + C::kTmS + 128 * b;
            float s[kC];
            float mx = -INFINITY;
            if (ok) {
                tc_fence_after_sync();
                uint32_t r[kC];
                tmem_ld_cols<kC>(s_addr + c0, r);
#pragma unroll
                for (int i = 0; i < kC; ++i) s[i] = __uint_as_float(r[i]);
                const int key0 = j * kTileRows + c0;
                if ((CAUSAL && j == n_kv - 1) || j * kTileRows + kTileRows > p.L) {
                    const int lim = CAUSAL ? min(p.L - 1, q_row) : (p.L - 1);
#pragma unroll
                    for (int c = 0; c < kC; ++c)
                        if (key0 + c > lim) s[c] = -INFINITY;
                }
                float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int c = 4; c < kC; c += 4) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) m4[u] = fmaxf(m4[u], s[c + u]);
                }
                mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
            red_max[b][part][row] = mx;
            // All slices have read their S columns (P may now overwrite them) and published
            // their partial maxima.
            ok = bar_and(grp_bar, kGrpThreads, ok);
            if (!ok) break;
#pragma unroll
            for (int q = 0; q < C::kSplit; ++q) mx = fmaxf(mx, red_max[b][q][row]);
            const float m_cand = mx * p.scale_log2;
            float m_new = m_ref;
            if (m_cand > m_ref + kRescaleThreshold) m_new = m_cand;
            const bool rescale = (j > 0) && (m_new != m_ref);
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            const float alpha = rescale ? ex2_approx(m_ref - m_new) : 1.0f;
            float sum4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            uint32_t pk[kC / 2];
#pragma unroll
            for (int i = 0; i < kC / 2; ++i) {
                const float p0 = ex2_approx(fmaf(s[2 * i], p.scale_log2, -m_use));
                const float p1 = ex2_approx(fmaf(s[2 * i + 1], p.scale_log2, -m_use));
                sum4[i & 3] += p0 + p1;
                pk[i] = pack2<BF16>(p0, p1);
            }
            tmem_st<kC / 2>(tmem + lane_off + C::kTmS + 128 * b + part * (kC / 2), pk);
            l_sum = l_sum * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
            bool okr = true;
            if (__any_sync(0xffffffffu, rescale)) {
                // O holds the sum up to tile j-1: wait for that PV, then rescale in place.
                okr = wait_bounded(&bar_od, (uint32_t)(j - 1) & 1u, abort_v, p.timeout_ns);
                okr = __all_sync(0xffffffffu, okr);
                if (okr) {
                    tc_fence_after_sync();
                    tmem_row_scale<C::kOCols>(tmem + lane_off + C::kTmO + part * C::kOCols, alpha);
                }
            }
            okr = bar_and(grp_bar, kGrpThreads, okr);
            if (!okr) {
                ok = false;
                break;
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bar_pf[b]);
            m_ref = m_new;
        }
        if (ok && n_kv > 0) {
            ok = wait_bounded(&bar_oready, 0, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
        }
        red_sum[part][row] = l_sum;
        ok = bar_and(grp_bar, kGrpThreads, ok);
        if (!ok) {
            if (lane == 0) record_timeout(p.status, abort_v);
        } else {
            tc_fence_after_sync();
            float l_tot = 0.0f;
#pragma unroll
            for (int q = 0; q < C::kSplit; ++q) l_tot += red_sum[q][row];
            const bool valid = q_row < p.L;
            if (valid && part == 0) p.lse[(size_t)bh * p.L + q_row] = (m_ref + log2f(l_tot)) * kLn2;
            uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) + ((size_t)bh * p.L + q_row) * D * 2 +
                            part * C::kOCols * 2;
            tmem_row_to_global<BF16, C::kOCols>(tmem + lane_off + C::kTmO + part * C::kOCols, orow,
                                                1.0f / l_tot, valid);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_t(const FwdParams& p, cudaStream_t s) {
    using C = FwdCfg<D, BF16, CAUSAL>;
    auto kern = fa_fwd_kernel<D, BF16, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)p.n_tiles * (unsigned)p.BH;
    kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, int D, bool bf16, bool causal, cudaStream_t s) {
    if (D == 64) {
        if (bf16) return causal ? launch_t<64, true, true>(p, s) : launch_t<64, true, false>(p, s);
        return causal ? launch_t<64, false, true>(p, s) : launch_t<64, false, false>(p, s);
    }
    if (bf16) return causal ? launch_t<128, true, true>(p, s) : launch_t<128, true, false>(p, s);
    return causal ? launch_t<128, false, true>(p, s) : launch_t<128, false, false>(p, s);
}

}  // namespace fa
