// fa_fwd_pair.cu -- the attention forward at D = 128 on CTA pairs (tcgen05 cta_group::2).
//
// Same method as fa_fwd.cu ("FlashAttention data-flow optimisation: MI50 memory and bandwidth
// bottlenecks", section 2.2: Q tiles kept on chip, K/V streamed, online softmax, only O and
// the log-sum-exp written), laid out for the pair form of the tensor core: a cluster of two
// CTAs on two SMs, and every contraction is one M = 256 MMA issued by the even CTA whose A rows
// 0-127 come from the even CTA and rows 128-255 from the odd one, and whose B operand is split
// between the two CTAs' shared memory by columns (N / 2 each); each CTA's tensor memory receives
// its own 128 rows.  So each CTA loads only half of every K tile (64 keys) and half of every V
// tile (64 of the 128 value columns): half the shared-memory bytes and L2 -> SM traffic per
// FLOP of the one-CTA kernel, and half the MMA instructions (one per pair).
//
// Work item: one cluster per four consecutive query tiles 4m..4m+3 of one head.  Super-tile A
// (M = 256) is query tiles 4m (even CTA) and 4m+1 (odd CTA), super-tile B is 4m+2 and 4m+3; a
// super-tile streams the key tiles of its later query tile (the earlier tile's rows mask the
// extra keys).  Tiles past the last query read zeros (tensor-copy out-of-bounds fill) and are
// not stored.
//
// CTA roles (352 threads), in both CTAs:
//   warps 0-7   softmax, four per super-tile (one row of S per thread, this CTA's rows);
//   warp 8      TMA producer: this CTA's two Q tiles, then its halves of K_j into a 4-slot ring;
//   warp 9      even CTA: MMA issuer; odd CTA: relay -- it waits for each of its own copies and
//               forwards the arrival to the even CTA's barrier of the same slot, so the issuer
//               sees both halves;
//   warp 10     TMA producer of this CTA's halves of V_j (4-slot ring).
// TMEM (allocated for the pair): S_A [0,128), S_B [128,256) (the 16-bit P overwrites the
// first 64 columns of its S), O_A [256,384), O_B [384,512).
// Completion of the even CTA's MMAs is signalled to both CTAs by two plain commits (one per
// CTA's barrier, no multicast); the odd CTA's softmax publishes P to the even CTA's barrier
// with remote arrives (one per warp).  MMA order and the reasoning that makes the in-place O rescale safe are
// those of fa_fwd.cu (S_t(j+1) is issued after PV_t(j)).
//
// No persistent form and no dropout variant.  fa_fwd_ex runs it only after
// fa_set_forward_pair(1): on this GPU a pair TS step (the PV contraction) runs at 78% of the
// single-CTA rate and the pair couples the two CTAs' softmax every step, so the single-CTA
// forward is faster and stays the default.
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_sched.h"

namespace fa {
namespace {

constexpr float kRescaleThresholdPair = 8.0f;
constexpr float kLn2Pair = 0.6931471805599453f;

template <bool BF16, bool CAUSAL>
struct PairCfg {
    static constexpr int D = 128;
    static constexpr int kQBytes = kTileRows * D * 2;     // one Q tile (2 chunks of 16 KB)
    static constexpr int kKHalf = 64 * D * 2;             // 64 keys x 128: 2 chunks of 8 KB
    static constexpr int kKChunk = 64 * 128;              // 64 rows of 128 bytes
    static constexpr int kVHalf = kTileRows * 64 * 2;     // 128 keys x 64 value columns
    static constexpr int kKStages = 4, kVStages = 4;
    static constexpr int kOffQ = 0;                       // Q_A, then Q_B (this CTA's rows)
    static constexpr int kOffK = 2 * kQBytes;
    static constexpr int kOffV = kOffK + kKStages * kKHalf;
    // One 4 KB buffer per softmax warp for the O read-out (32 rows x 64 columns, 16-bit).
    static constexpr int kStageBytes = 32 * 64 * 2;
    static constexpr int kOffStage = kOffV + kVStages * kVHalf;
    static constexpr int kSmemBytes = kOffStage + 8 * kStageBytes + 1024;  // + alignment slack
    static constexpr int kGroupWarps = 4;
    static constexpr int kGroupThreads = kGroupWarps * 32;
    static constexpr int kSoftmaxWarps = 2 * kGroupWarps;
    static constexpr int kProducerWarp = kSoftmaxWarps;
    static constexpr int kMmaWarp = kSoftmaxWarps + 1;
    static constexpr int kVProducerWarp = kSoftmaxWarps + 2;
    static constexpr int kThreads = (kSoftmaxWarps + 3) * 32;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmS = 0, kTmO = 256;
    static_assert(kSmemBytes <= 232448, "shared memory over the 227 KB per-block limit");
    static constexpr uint32_t kIdescS = idesc_f16(BF16, 256, 128, false, false);
    static constexpr uint32_t kIdescO = idesc_f16(BF16, 256, D, false, true);
};

// ---- CTA-pair primitives -------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of the variable at shared::cta address `saddr` in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ __forceinline__ void arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
__device__ __forceinline__ bool try_wait_cl(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// wait_bounded with cluster-scope acquire: for the barriers whose arrivals from the other CTA
// publish shared-memory data (relayed copies) or tensor-memory data written by the other CTA's
// threads (P).  Barriers that only the tensor core's commits complete (S, O ready, ring slots
// read) are waited on with the CTA-scope wait: the data they announce is ordered by the
// tcgen05 fences, not by the barrier's memory semantics.
__device__ __forceinline__ bool wait_cl(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                        uint64_t timeout_ns) {
    if (try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (try_wait_cl(bar, parity)) return true;
        if (abort != nullptr && *abort) return false;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}
__device__ __forceinline__ bool wait_cl_warp(uint64_t* bar, uint32_t parity,
                                             const volatile int* abort, uint64_t timeout_ns) {
    return __all_sync(0xffffffffu, wait_cl(bar, parity, abort, timeout_ns));
}
__device__ __forceinline__ void alloc_pair(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void mma_pair_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_pair_ts(uint32_t d, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// Arrives once on `bar` (a shared::cluster address) when the pair MMAs issued so far by this
// thread have completed.
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(
            bar)
        : "memory");
}

struct PairItem {
    int bh, quad;            // head, query tiles 4*quad .. 4*quad + 3
    int nk[2], n_kv;         // key tiles of super-tiles A and B (0: no row sees a key / absent)
};

template <bool CAUSAL>
__device__ __forceinline__ PairItem pair_item(const FwdParams& p) {
    PairItem it;
    const int n_quads = (p.n_qtiles + 3) >> 2;
    int rank;
    tile_coords((int)(blockIdx.x >> 1), p.BH, n_quads, p.group, it.bh, rank);
    it.quad = n_quads - 1 - rank;  // heaviest (most key tiles) first
    for (int t = 0; t < 2; ++t) {
        const int first = 4 * it.quad + 2 * t;
        it.nk[t] = first < p.n_qtiles ? q_tile_kv(first + 1, p.Lq, p.Lk, CAUSAL) : 0;
    }
    it.n_kv = it.nk[0] > it.nk[1] ? it.nk[0] : it.nk[1];
    return it;
}

template <bool BF16, bool CAUSAL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<BF16, CAUSAL>::kThreads, 1)
    fa_fwd_pair_kernel(const __grid_constant__ FwdParams p) {
    using C = PairCfg<BF16, CAUSAL>;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ uint64_t bar_qf, bar_kf[C::kKStages], bar_ke[C::kKStages], bar_vf[C::kVStages],
        bar_ve[C::kVStages], bar_sf[2], bar_pf[2], bar_oready[2], bar_fin;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    volatile int* abort_v = &abort_flag;
    const PairItem it = pair_item<CAUSAL>(p);
    const int hb = it.bh / p.H, hh = it.bh - hb * p.H;  // batch and head

    if (threadIdx.x == 0) {
        abort_flag = 0;
        // The even CTA's "full" barriers also wait for the odd CTA's relayed arrival.
        const uint32_t fills = leader ? 2u : 1u;
        mbar_init(&bar_qf, fills);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&bar_kf[s], fills);
            mbar_init(&bar_ke[s], 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(&bar_vf[s], fills);
            mbar_init(&bar_ve[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar_sf[t], 1);
            // P_t published: the even CTA's 128 softmax threads, and one arrive per warp of the
            // odd CTA's group (a remote arrive is a cluster-scope release: one per warp).
            mbar_init(&bar_pf[t], C::kGroupThreads + C::kGroupWarps);
            mbar_init(&bar_oready[t], 1);
        }
        mbar_init(&bar_fin, 1);
        mbar_fence_init();
    }
    if (warp == C::kMmaWarp) alloc_pair(&tmem_base_sh, C::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    const uint32_t peer = rank ^ 1u;
    // Commits from the even CTA: to its own barrier and to the odd CTA's copy of it.
    auto commit_both = [&](uint64_t* bar) {
        commit_pair(smem_u32(bar));
        commit_pair(peer_addr(smem_u32(bar), peer));
    };

    if (it.n_kv > 0 && (warp == C::kProducerWarp || warp == C::kVProducerWarp)) {
        // ------------------------------ TMA producers ------------------------------
        if (lane == 0) {
            const bool is_k = warp == C::kProducerWarp;
            const CUtensorMap* map = is_k ? &p.tm_k_half : &p.tm_v;
            const int stages = is_k ? C::kKStages : C::kVStages;
            uint64_t* full = is_k ? bar_kf : bar_vf;
            uint64_t* empty = is_k ? bar_ke : bar_ve;
            const int slot_bytes = is_k ? C::kKHalf : C::kVHalf;
            uint8_t* ring = smem + (is_k ? C::kOffK : C::kOffV);
            tma_prefetch_desc(map);
            bool ok = true;
            if (is_k) {  // this CTA's rows of super-tiles A and B
                tma_prefetch_desc(&p.tm_q);
                mbar_arrive_expect_tx(&bar_qf, 2 * C::kQBytes);
                for (int t = 0; t < 2; ++t)
                    for (int c = 0; c < 2; ++c)
                        tma_load_4d(smem + C::kOffQ + t * C::kQBytes + c * kChunkBytes, &p.tm_q,
                                    &bar_qf, c * kChunkElems,
                                    (4 * it.quad + 2 * t + (int)rank) * kTileRows, hh, hb);
            }
            for (int j = 0; ok && j < it.n_kv; ++j) {
                const int st = j % stages;
                if (j >= stages && !wait_bounded(&empty[st], ((uint32_t)(j / stages) & 1u) ^ 1u,
                                                 abort_v, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[st], (uint32_t)slot_bytes);
                uint8_t* dst = ring + st * slot_bytes;
                if (is_k) {  // keys 128 j + 64 rank .. + 63, both 64-column chunks
                    for (int c = 0; c < 2; ++c)
                        tma_load_4d(dst + c * C::kKChunk, map, &full[st], c * kChunkElems,
                                    j * kTileRows + 64 * (int)rank, hh, hb);
                } else {     // value columns 64 rank .. + 63 of keys 128 j .. + 127
                    tma_load_4d(dst, map, &full[st], 64 * (int)rank, j * kTileRows, hh, hb);
                }
            }
            if (!ok) record_timeout(p.status, abort_v);
            // Drain: the newest fill of every slot must have landed before the CTA exits.
            // (These waits return at once on the normal path; the even CTA's full barriers
            // also count the relayed arrival, so after a failure they wait out the limit.)
            if (is_k) wait_cl(&bar_qf, 0, nullptr, p.timeout_ns);
            for (int g = it.n_kv - 1; g >= 0 && g >= it.n_kv - stages; --g)
                wait_cl(&full[g % stages], (uint32_t)(g / stages) & 1u, nullptr, p.timeout_ns);
        }
    } else if (it.n_kv > 0 && warp == C::kMmaWarp && !leader) {
        // ------------------------------ relay (odd CTA) ------------------------------
        // Forwards every landed copy of this CTA to the even CTA's barrier of the same slot,
        // in fill order: Q, then K_0, V_0, K_1, V_1, ...
        if (lane == 0) {
            bool ok = wait_bounded(&bar_qf, 0, abort_v, p.timeout_ns);
            if (ok) arrive_remote(peer_addr(smem_u32(&bar_qf), 0));
            for (int j = 0; ok && j < it.n_kv; ++j) {
                const int ks = j % C::kKStages, vs = j % C::kVStages;
                ok = wait_bounded(&bar_kf[ks], (uint32_t)(j / C::kKStages) & 1u, abort_v,
                                  p.timeout_ns);
                if (ok) arrive_remote(peer_addr(smem_u32(&bar_kf[ks]), 0));
                ok = ok && wait_bounded(&bar_vf[vs], (uint32_t)(j / C::kVStages) & 1u, abort_v,
                                        p.timeout_ns);
                if (ok) arrive_remote(peer_addr(smem_u32(&bar_vf[vs]), 0));
            }
            if (!ok) record_timeout(p.status, abort_v);
        }
    } else if (it.n_kv > 0 && warp == C::kMmaWarp) {
        // ------------------------------ MMA issuer (even CTA) ------------------------------
        bool ok = true;
        int k_ready = -1;
        auto wait_k = [&](int j) -> bool {
            if (k_ready >= j) return true;
            if (!wait_cl_warp(&bar_kf[j % C::kKStages], (uint32_t)(j / C::kKStages) & 1u, abort_v,
                              p.timeout_ns))
                return false;
            tc_fence_after_sync();
            k_ready = j;
            return true;
        };
        auto issue_s = [&](int t, int j) {  // S_t = Q_t K_j^T (M = 256 over the pair)
            const uint64_t qd = sdesc_kmajor_sw128(smem_u32(smem + C::kOffQ + t * C::kQBytes));
            const uint64_t kd = sdesc_kmajor_sw128(
                smem_u32(smem + C::kOffK + (j % C::kKStages) * C::kKHalf));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t a_off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                const uint32_t b_off = (kk >> 2) * C::kKChunk + (kk & 3) * 32;
                mma_pair_ss(tmem + C::kTmS + 128 * t, sdesc_advance(qd, a_off),
                            sdesc_advance(kd, b_off), C::kIdescS | p.s_negate, kk > 0 ? 1u : 0u);
            }
            commit_both(&bar_sf[t]);
        };
        auto issue_pv = [&](int t, int j) -> bool {  // O_t += P_t V_j
            if (!wait_cl_warp(&bar_pf[t], (uint32_t)j & 1u, abort_v, p.timeout_ns)) return false;
            tc_fence_after_sync();
            const uint64_t vd = sdesc_mnmajor_sw128(
                smem_u32(smem + C::kOffV + (j % C::kVStages) * C::kVHalf), kChunkBytes);
#pragma unroll
            for (int kk = 0; kk < kTileRows / 16; ++kk)
                mma_pair_ts(tmem + C::kTmO + 128 * t, tmem + C::kTmS + 128 * t + kk * 8,
                            sdesc_advance(vd, kk * 2048), C::kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
            if (j + 1 == it.nk[t]) commit_both(&bar_oready[t]);  // O_t is final
            return true;
        };
        ok = wait_cl_warp(&bar_qf, 0, abort_v, p.timeout_ns);
        tc_fence_after_sync();
        ok = ok && wait_k(0);
        if (ok) {
            if (it.nk[0] > 0) issue_s(0, 0);
            if (it.nk[1] > 0) issue_s(1, 0);
            commit_both(&bar_ke[0]);  // K_0 read
        }
        for (int j = 0; ok && j < it.n_kv; ++j) {
            const bool next = j + 1 < it.n_kv;
            if (!wait_cl_warp(&bar_vf[j % C::kVStages], (uint32_t)(j / C::kVStages) & 1u, abort_v,
                              p.timeout_ns) ||
                (next && !wait_k(j + 1))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (!ok) break;
                if (j < it.nk[t] && !issue_pv(t, j)) {
                    ok = false;
                    break;
                }
                if (next && j + 1 < it.nk[t]) issue_s(t, j + 1);
            }
            if (!ok) break;
            commit_both(&bar_ve[j % C::kVStages]);                    // V_j read
            if (next) commit_both(&bar_ke[(j + 1) % C::kKStages]);    // K_{j+1} read
        }
        if (!ok && lane == 0) record_timeout(p.status, abort_v);
        // Every issued MMA must finish before the pair's TMEM is released.
        commit_pair(smem_u32(&bar_fin));
        wait_warp(&bar_fin, 0, nullptr, p.timeout_ns);
    } else if (it.n_kv > 0 && warp < C::kSoftmaxWarps) {
        // ------------------------------ softmax warps ------------------------------
        const int t = warp / C::kGroupWarps;
        const int quad = warp % C::kGroupWarps;
        const int row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + C::kTmS + 128 * t;
        const uint32_t o_addr = tmem + lane_off + C::kTmO + 128 * t;
        const uint64_t scale2 = f2_make(p.scale_log2, p.scale_log2);
        const int n_mine = it.nk[t];
        const int q_row = (4 * it.quad + 2 * t + (int)rank) * kTileRows + row;
        const uint32_t pf_addr = leader ? 0u : peer_addr(smem_u32(&bar_pf[t]), 0);
        bool ok = true;
        float m_ref = -INFINITY;
        float l_sum = 0.0f;
        for (int j = 0; ok && j < n_mine; ++j) {
            ok = wait_bounded(&bar_sf[t], (uint32_t)j & 1u, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            float s[128];
            {
                uint32_t r[128];
                tmem_ld_cols<128>(s_addr, r);
#pragma unroll
                for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(r[i]);
            }
            const int key0 = j * kTileRows;
            if (key0 + kTileRows - 1 >
                (CAUSAL ? min(p.Lk - 1, (q_row & ~(kTileRows - 1)) + (p.Lk - p.Lq)) : p.Lk - 1)) {
                const int lim = CAUSAL ? min(p.Lk - 1, q_row + (p.Lk - p.Lq)) : p.Lk - 1;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (key0 + c > lim) s[c] = -INFINITY;
            }
            float m4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) m4[u] = fmaxf(s[u], s[u + 4]);
#pragma unroll
            for (int c = 8; c < 128; c += 8) {
#pragma unroll
                for (int u = 0; u < 4; ++u) m4[u] = fmax3(m4[u], s[c + u], s[c + 4 + u]);
            }
            const float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
            const float m_cand = mx * p.scale_log2;
            float m_new = m_ref;
            if (m_cand > m_ref + kRescaleThresholdPair) m_new = m_cand;
            const bool rescale = (j > 0) && (m_new != m_ref);
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            const float alpha = rescale ? ex2_approx(m_ref - m_new) : 1.0f;
            const uint64_t shift2 = f2_make(-m_use, -m_use);
            uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float y0, y1;
                    f2_split(f2_fma(f2_make(s[h * 32 + 2 * i], s[h * 32 + 2 * i + 1]), scale2,
                                    shift2),
                             y0, y1);
                    const float p0 = ex2_approx(y0);
                    const float p1 = ex2_approx(y1);
                    sum2[i & 1] = f2_add(sum2[i & 1], f2_make(p0, p1));
                    pk[i] = pack2<BF16>(p0, p1);
                }
                tmem_st16(s_addr + h * 16, pk);
            }
            float sa, sb, sc, sd;
            f2_split(sum2[0], sa, sb);
            f2_split(sum2[1], sc, sd);
            l_sum = l_sum * alpha + ((sa + sb) + (sc + sd));
            // S_t(j) was issued after PV_t(j-1): every PV into O_t has completed.
            if (__any_sync(0xffffffffu, rescale)) tmem_row_scale<D>(o_addr, alpha);
            tmem_st_wait();
            tc_fence_before_sync();
            if (leader) {
                mbar_arrive(&bar_pf[t]);
            } else {
                __syncwarp();
                if (lane == 0) arrive_remote(pf_addr);
            }
            m_ref = m_new;
        }
        if (ok && n_mine > 0) {
            ok = wait_bounded(&bar_oready[t], 0, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after_sync();
                const bool valid = q_row < p.Lq;
                if (valid)
                    p.lse[(size_t)it.bh * p.Lq + q_row] =
                        l_sum > 0.0f ? (m_ref + log2f(l_sum)) * kLn2Pair : -INFINITY;
                // This warp's 32 rows start at q_row - lane; those at or past Lq are not
                // written.  Coalesced through the warp's staging buffer.
                const int row0 = q_row - lane;
                uint8_t* orow0 =
                    reinterpret_cast<uint8_t*>(p.o) + row_offset(p.so, it.bh, p.H, row0);
                tmem_rows_to_global_staged<BF16, D>(
                    o_addr, smem_u32(smem + C::kOffStage + warp * C::kStageBytes), orow0,
                    (size_t)p.so.l * 2u, p.Lq - row0, l_sum > 0.0f ? 1.0f / l_sum : 0.0f, lane);
            }
        }
        if (!ok && lane == 0) record_timeout(p.status, abort_v);
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // the pair is done with both CTAs' TMEM, shared memory and barriers
    if (warp == C::kMmaWarp) {
        tc_fence_after_sync();
        dealloc_pair(tmem, C::kTmemCols);
    }
}

template <bool BF16, bool CAUSAL>
cudaError_t launch_pair_t(const FwdParams& p, cudaStream_t s) {
    using C = PairCfg<BF16, CAUSAL>;
    auto kern = fa_fwd_pair_kernel<BF16, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long clusters = (long long)((p.n_qtiles + 3) / 4) * p.BH;
    if (2 * clusters > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_kernel(kern, dim3((unsigned)(2 * clusters)), dim3(C::kThreads), C::kSmemBytes,
                         s, p);
}

}  // namespace

cudaError_t launch_fwd_pair(const FwdParams& p, bool bf16, bool causal, cudaStream_t s) {
    if (bf16) return causal ? launch_pair_t<true, true>(p, s) : launch_pair_t<true, false>(p, s);
    return causal ? launch_pair_t<false, true>(p, s) : launch_pair_t<false, false>(p, s);
}

}  // namespace fa
