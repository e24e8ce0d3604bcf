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
// GB300 layout.  A work item is TWO consecutive 128-row query tiles (A = 2p, B = 2p+1) of one
// head, so every K/V tile brought into shared memory feeds two tiles' worth of MMAs: the L2 ->
// SM traffic per FLOP is half of a one-tile item's, and each ring slot has twice as long to
// arrive.  The two tiles also give the tensor core independent work to interleave: while the
// softmax of tile A runs, the MMA warp computes tile B's PV and S, and the other way round.
//
// Scheduling (fwd_grid).  Items are ordered heaviest first inside L2-sized head groups
// (tile_coords).  For rows of few key tiles a CTA's fixed cost (launch, barrier and TMEM
// set-up, the first copies' latency, the pipeline fill, the O read-out) is a large share of
// its work, so the grid is one CTA per SM and each CTA takes items in the snake rounds of
// persistent_tile: the K/V ring runs on from one item to the next, the next item's Q is loaded
// as soon as the current item's S contractions have completed (at D = 64 into a second Q slot,
// at once), and the next item's first S contractions run while the softmax warps read out O.
// For long rows the grid is one CTA per item (each CTA runs its single round), which lets the
// hardware's block scheduler balance the causal items.
//
// CTA roles (352 threads at D = 128, 320 at D = 64):
//   warps 0-7    softmax, four per query tile (tile A first); warp w owns TMEM lanes
//                32*(w%4).. (query rows), so every thread owns one whole row of S;
//   warp 8       TMA producer of Q_A, Q_B (per item) and the K_j ring (at D = 64 K_j and V_j
//                together in one slot);
//   warp 9       MMA issuer (one elected thread) and TMEM owner;
//   warp 10      TMA producer of the V_j ring (D = 128 only).
// TMEM columns: S_A [0,128), S_B [128,256) (fp32; the 16-bit P of a tile overwrites the first
// 64 columns of its S and feeds the PV MMA straight from TMEM), O_A [256, 256+D),
// O_B [256+D, 256+2D).  MMA order per item: S_A0, S_B0, then for each key tile j: PV_Aj,
// S_A(j+1), PV_Bj, S_B(j+1).  S_t(j+1) is issued after PV_tj, so (tcgen05 MMAs of one thread
// run in issue order) it never overwrites a P still being read, and once the softmax sees
// S_t(j+1) every PV before it has finished: O_t may be rescaled in place with no further wait.
// The same order carries across items: S_t0 of the next item follows the last PV_t of this
// one, and the softmax warps finish reading O_t out before they publish P_t0 of the next item,
// so PV_t0 (which overwrites O_t) never starts before the read-out is done.
//
// Online softmax in the log2 domain: y = s * |scale| * log2(e), where s is the stored S.  For a
// negative scale the S contraction runs with its A operand negated (an exact sign flip set in
// the instruction descriptor), so s * |scale| = (Q K^T) * scale for either sign and the row
// maximum of the stored S is always the row maximum of the logits.  The running reference max m
// is only raised when a tile's max exceeds it by more than kRescaleThreshold (2^8 headroom
// for P), so O is rescaled rarely; the result is unchanged because O and the running sum
// always share the same reference.  LSE = (m + log2(l)) * ln(2).
//
// Barrier phases count completions over the CTA's lifetime: the S / P barriers of tile t once
// per key tile of every item that has tile t, the O barrier of tile t once per such item, the
// ring barriers once per fill, the Q barriers once per item using that slot.
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_sched.h"

namespace fa {
namespace {

constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, bool BF16, bool CAUSAL>
struct FwdCfg {
    static constexpr int kChunks = D / kChunkElems;            // swizzle boxes per tile row
    static constexpr int kTileBytes = kTileRows * D * 2;       // one 128 x D tile
    // D = 64: K_j and V_j share one slot of the K ring (one full and one empty barrier per
    // slot, one producer warp), and the Q pair has two slots, so the next item's Q lands while
    // this item runs.  D = 128: separate K and V rings of two slots each, so that K_{j+1} can
    // land while V_j is still being read (measured faster at that size), and one Q slot (the
    // tiles fill 192 KB).
    static constexpr bool kMergedKV = (D == 64);
    static constexpr int kQSlots = (D == 128) ? 1 : 2;         // Q_A/Q_B pairs in flight
    static constexpr int kKStages = (D == 128) ? 2 : 4;        // K (or K/V) ring depth
    static constexpr int kVStages = (D == 128) ? 2 : 4;        // V ring depth (separate rings)
    static constexpr int kOffQ = 0;                            // slot s: Q_A, then Q_B
    static constexpr int kOffK = kOffQ + kQSlots * 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    // One 4 KB buffer per softmax warp for the O read-out (32 rows x 64 columns, 16-bit).
    static constexpr int kStageBytes = 32 * 64 * 2;
    static constexpr int kOffStage = kOffV + kVStages * kTileBytes;
    static constexpr int kSmemBytes = kOffStage + 8 * kStageBytes + 1024;  // + alignment slack
    static constexpr int kGroupWarps = 4;                      // softmax warps per query tile
    static constexpr int kGroupThreads = kGroupWarps * 32;
    static constexpr int kSoftmaxWarps = 2 * kGroupWarps;
    static constexpr int kProducerWarp = kSoftmaxWarps;
    static constexpr int kMmaWarp = kSoftmaxWarps + 1;
    static constexpr int kVProducerWarp = kSoftmaxWarps + 2;
    static constexpr int kThreads = (kSoftmaxWarps + (kMergedKV ? 2 : 3)) * 32;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmS = 0;        // S of tile t at kTmS + 128*t
    static constexpr uint32_t kTmO = 256;      // O of tile t at kTmO + D*t
    static_assert(kTmO + 2 * D <= kTmemCols, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory over the 227 KB per-block limit");
    static constexpr uint32_t kIdescS = idesc_f16(BF16, 128, 128, false, false);
    static constexpr uint32_t kIdescO = idesc_f16(BF16, 128, D, false, true);
};

// One work item: a pair of query tiles of one head and the key tiles each of them sees.
struct FwdItem {
    int bh, q_a, q_b;
    int n_kv_a, n_kv_b, n_kv;  // key tiles of tile A, of tile B (0 also when there is no tile
                               // B) and of the pair; 0 when no row of the tile (pair) sees a key
};

template <bool CAUSAL>
__device__ __forceinline__ bool fwd_item(const FwdParams& p, int round, FwdItem& it) {
    const int n_pairs = (p.n_qtiles + 1) >> 1;
    const int id = persistent_tile(round, (int)blockIdx.x, (int)gridDim.x, n_pairs * p.BH);
    if (id < 0) return false;
    int rank;
    tile_coords(id, p.BH, n_pairs, p.group, it.bh, rank);
    const int pair = n_pairs - 1 - rank;  // heaviest pairs (most key tiles) first
    it.q_a = 2 * pair;
    it.q_b = 2 * pair + 1;
    const bool has_b = it.q_b < p.n_qtiles;
    it.n_kv_a = q_tile_kv(it.q_a, p.Lq, p.Lk, CAUSAL);
    it.n_kv_b = has_b ? q_tile_kv(it.q_b, p.Lq, p.Lk, CAUSAL) : 0;
    it.n_kv = it.n_kv_b > it.n_kv_a ? it.n_kv_b : it.n_kv_a;  // n_kv_a <= n_kv_b
    return true;
}

// DROP: dropout on P (p.drop): the PV operand carries the kept entries only, the running sum
// all of them, and the final 1/l includes 1/(1-p).
template <int D, bool BF16, bool CAUSAL, bool DROP>
__global__ void __launch_bounds__(FwdCfg<D, BF16, CAUSAL>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = FwdCfg<D, BF16, CAUSAL>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ uint64_t bar_qf[C::kQSlots], bar_qe[C::kQSlots];  // Q pair landed / read by S
    __shared__ uint64_t bar_kf[C::kKStages], bar_ke[C::kKStages], bar_vf[C::kVStages],
        bar_ve[C::kVStages], bar_sf[2], bar_pf[2], bar_oready[2], bar_fin;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::kQSlots; ++s) {
            mbar_init(&bar_qf[s], 1);
            mbar_init(&bar_qe[s], 1);
        }
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&bar_kf[s], 1);
            mbar_init(&bar_ke[s], 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(&bar_vf[s], 1);
            mbar_init(&bar_ve[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar_sf[t], 1);
            mbar_init(&bar_pf[t], C::kGroupThreads);
            mbar_init(&bar_oready[t], 1);
        }
        mbar_init(&bar_fin, 1);
        mbar_fence_init();
    }
    if (warp == C::kMmaWarp) tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    auto q_tile = [&](int slot, int t) { return smem + C::kOffQ + (slot * 2 + t) * C::kTileBytes; };

    if (warp == C::kProducerWarp || (!C::kMergedKV && warp == C::kVProducerWarp)) {
        // ------------------------------ TMA producers ------------------------------
        // kProducerWarp: per item the Q pair (once its slot is free), then K_j (D = 64: K_j and
        // V_j together) into the ring; kVProducerWarp (D = 128): V_j into its ring.  The rings
        // run on across items.
        if (lane == 0) {
            const bool is_k = warp == C::kProducerWarp;
            const CUtensorMap* map = is_k ? &p.tm_k : &p.tm_v;
            const int stages = is_k ? C::kKStages : C::kVStages;
            uint64_t* full = is_k ? bar_kf : bar_vf;
            uint64_t* empty = is_k ? bar_ke : bar_ve;
            uint8_t* ring = smem + (is_k ? C::kOffK : C::kOffV);
            constexpr uint32_t kFill = (C::kMergedKV ? 2 : 1) * C::kTileBytes;
            tma_prefetch_desc(map);
            if (is_k) {
                tma_prefetch_desc(&p.tm_q);
                if (C::kMergedKV) tma_prefetch_desc(&p.tm_v);
            }
            bool ok = true;
            int issued = 0;  // ring fills handed to the TMA unit
            int n_q = 0;     // Q pair fills handed to the TMA unit
            FwdItem it;
            for (int round = 0; ok && fwd_item<CAUSAL>(p, round, it); ++round) {
                if (it.n_kv == 0) continue;  // no row sees a key: the softmax warps write it
                const int hb = it.bh / p.H, hh = it.bh - hb * p.H;  // batch and head
                if (is_k) {
                    const int qs = n_q % C::kQSlots;
                    const int use = n_q / C::kQSlots;  // earlier uses of this slot
                    if (use > 0 && !wait_bounded(&bar_qe[qs], (uint32_t)(use - 1) & 1u, abort_v,
                                                 p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const int nt = it.n_kv_b > 0 ? 2 : 1;
                    mbar_arrive_expect_tx(&bar_qf[qs], nt * C::kTileBytes);
                    for (int t = 0; t < nt; ++t)
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_4d(q_tile(qs, t) + c * kChunkBytes, &p.tm_q, &bar_qf[qs],
                                        c * kChunkElems, (t ? it.q_b : it.q_a) * kTileRows, hh, hb);
                    ++n_q;
                }
                for (int j = 0; j < it.n_kv; ++j) {
                    const int st = issued % stages;
                    const uint32_t ph = (uint32_t)(issued / stages) & 1u;
                    if (issued >= stages &&
                        !wait_bounded(&empty[st], ph ^ 1u, abort_v, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[st], kFill);
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_4d(ring + st * C::kTileBytes + c * kChunkBytes, map, &full[st],
                                    c * kChunkElems, j * kTileRows, hh, hb);
                        if constexpr (C::kMergedKV)
                            tma_load_4d(smem + C::kOffV + st * C::kTileBytes + c * kChunkBytes,
                                        &p.tm_v, &full[st], c * kChunkElems, j * kTileRows, hh, hb);
                    }
                    ++issued;
                }
            }
            if (!ok) record_timeout(p.status, abort_v);
            // Drain: the newest fill of every slot must have landed before the CTA exits.
            // (These waits return at once on the normal path.)
            for (int n = n_q - 1; n >= 0 && n >= n_q - C::kQSlots; --n)
                wait_bounded(&bar_qf[n % C::kQSlots], (uint32_t)(n / C::kQSlots) & 1u, nullptr,
                             p.timeout_ns);
            for (int g = issued - 1; g >= 0 && g >= issued - stages; --g)
                wait_bounded(&full[g % stages], (uint32_t)(g / stages) & 1u, nullptr, p.timeout_ns);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------ MMA issuer ------------------------------
        // The whole warp walks the loop (warp-uniform values); one elected lane issues.  A wait
        // between MMA groups can let the tensor pipe's short queue run dry, so each key tile
        // starts with the ring waits (D = 64: the merged slot j+1; D = 128: V_j and K_{j+1})
        // while the warp would idle until P of tile A anyway; after that only the two P waits
        // sit between MMA groups.  g counts key tiles over the CTA's lifetime (ring slot and
        // phase), ps[t] the S / P completions of tile t.
        bool ok = true;
        int g = 0, n_item = 0, ps[2] = {0, 0};
        int k_ready = -1;  // newest ring fill (K, or K/V) known to have landed
        auto wait_k = [&](int gk) -> bool {
            if (k_ready >= gk) return true;
            if (!wait_warp(&bar_kf[gk % C::kKStages], (uint32_t)(gk / C::kKStages) & 1u, abort_v,
                           p.timeout_ns))
                return false;
            tc_fence_after_sync();
            k_ready = gk;
            return true;
        };
        FwdItem it;
        for (int round = 0; ok && fwd_item<CAUSAL>(p, round, it); ++round) {
            if (it.n_kv == 0) continue;  // no row of the pair sees a key
            const int qs = n_item % C::kQSlots;
            const int n_kv = it.n_kv;
            const int nk[2] = {it.n_kv_a, it.n_kv_b};
            auto issue_s = [&](int t, int gk) {  // S_t = Q_t K^T for ring fill gk
                const uint64_t qd = sdesc_kmajor_sw128(smem_u32(q_tile(qs, t)));
                const uint64_t kd =
                    sdesc_kmajor_sw128(smem_u32(smem + C::kOffK + (gk % C::kKStages) * C::kTileBytes));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    mma_ss_w(tmem + C::kTmS + 128 * t, sdesc_advance(qd, off), sdesc_advance(kd, off),
                             C::kIdescS | p.s_negate, kk > 0 ? 1u : 0u);
                }
                mma_commit_w(&bar_sf[t]);
            };
            auto issue_pv = [&](int t, int j) -> bool {  // O_t += P_t V_j (V_j already landed)
                if (!wait_warp(&bar_pf[t], (uint32_t)(ps[t] + j) & 1u, abort_v, p.timeout_ns))
                    return false;
                tc_fence_after_sync();
                const int gv = g + j;
                const int vst = C::kMergedKV ? gv % C::kKStages : gv % C::kVStages;
                const uint64_t vd =
                    sdesc_mnmajor_sw128(smem_u32(smem + C::kOffV + vst * C::kTileBytes), kChunkBytes);
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk) {
                    const uint64_t bd = sdesc_advance(vd, kk * 2048);
                    mma_ts_w(tmem + C::kTmO + D * t, tmem + C::kTmS + 128 * t + kk * 8, bd,
                             C::kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                if (j + 1 == nk[t]) mma_commit_w(&bar_oready[t]);  // O_t is final
                return true;
            };
            // Q pair of this item landed, and K_0 (D = 64: K_0 and V_0).
            ok = wait_warp(&bar_qf[qs], (uint32_t)(n_item / C::kQSlots) & 1u, abort_v,
                           p.timeout_ns);
            tc_fence_after_sync();
            ok = ok && wait_k(g);
            if (!ok) break;
            if (nk[0] > 0) issue_s(0, g);
            if (nk[1] > 0) issue_s(1, g);
            if (n_kv == 1) mma_commit_w(&bar_qe[qs]);  // every S of the item issued
            if constexpr (!C::kMergedKV) mma_commit_w(&bar_ke[g % C::kKStages]);  // K_0 read
            for (int j = 0; ok && j < n_kv; ++j) {
                const bool next = j + 1 < n_kv;
                const int gj = g + j;
                if constexpr (C::kMergedKV) {
                    // Slot j+1 first, while this warp idles until P_A(j) anyway.
                    if (next && !wait_k(gj + 1)) {
                        ok = false;
                        break;
                    }
                } else {
                    // Ring waits first: then each P wait is followed by PV and the next S with
                    // no wait in between.
                    if (!wait_warp(&bar_vf[gj % C::kVStages], (uint32_t)(gj / C::kVStages) & 1u,
                                   abort_v, p.timeout_ns) ||
                        (next && !wait_k(gj + 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                }
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!ok) break;
                    if (j < nk[t] && !issue_pv(t, j)) {
                        ok = false;
                        break;
                    }
                    if (next && j + 1 < nk[t]) issue_s(t, gj + 1);
                }
                if (!ok) break;
                if (j + 2 == n_kv) mma_commit_w(&bar_qe[qs]);  // the item's last S issued
                if constexpr (C::kMergedKV) {
                    mma_commit_w(&bar_ke[gj % C::kKStages]);  // K_j (S_j) and V_j (PV_j) read
                } else {
                    mma_commit_w(&bar_ve[gj % C::kVStages]);                  // V_j read
                    if (next) mma_commit_w(&bar_ke[(gj + 1) % C::kKStages]);  // K_{j+1} read
                }
            }
            g += n_kv;
            ps[0] += nk[0];
            ps[1] += nk[1];
            ++n_item;
        }
        if (!ok && lane == 0) record_timeout(p.status, abort_v);
        // Every issued MMA must finish before TMEM is released.
        mma_commit_w(&bar_fin);
        wait_warp(&bar_fin, 0, nullptr, p.timeout_ns);
    } else {
        // ------------------------------ softmax warps ------------------------------
        const int t = warp / C::kGroupWarps;  // query tile of this group
        const int quad = warp % C::kGroupWarps;  // TMEM lane quadrant
        const int row = quad * 32 + lane;     // row inside the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + C::kTmS + 128 * t;
        const uint32_t o_addr = tmem + lane_off + C::kTmO + D * t;
        const uint64_t scale2 = f2_make(p.scale_log2, p.scale_log2);
        bool ok = true;
        int ps = 0;      // S / P completions of this tile so far
        int n_done = 0;  // items of this tile finished (O barrier phase)
        FwdItem it;
        for (int round = 0; ok && fwd_item<CAUSAL>(p, round, it); ++round) {
            const int n_mine = t ? it.n_kv_b : it.n_kv_a;
            const int q_row = (t ? it.q_b : it.q_a) * kTileRows + row;
            // No tile B, or no row of this tile sees a key (fa_fwd_empty_rows_kernel writes it).
            if (n_mine == 0) continue;
            float m_ref = -INFINITY;
            float l_sum = 0.0f;
            for (int j = 0; j < n_mine; ++j) {
                ok = wait_bounded(&bar_sf[t], (uint32_t)(ps + j) & 1u, abort_v, p.timeout_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;  // warp-uniform: the warp owns its rows alone
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
                // Row max: four independent chains of three-input maxima.
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
                if (m_cand > m_ref + kRescaleThreshold) m_new = m_cand;
                const bool rescale = (j > 0) && (m_new != m_ref);
                const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
                const float alpha = rescale ? ex2_approx(m_ref - m_new) : 1.0f;
                // Two columns per instruction for the scale-and-shift and the running sum.
                const uint64_t shift2 = f2_make(-m_use, -m_use);
                uint64_t sum2[2] = {0ull, 0ull};  // (+0.0f, +0.0f)
#pragma unroll
                for (int h = 0; h < 4; ++h) {  // 32 columns -> 16 packed TMEM columns at a time
                    uint32_t pk[16];
                    uint32_t keep = 0xfu;  // dropout: keep bits of the current 4 columns
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float y0, y1;
                        f2_split(f2_fma(f2_make(s[h * 32 + 2 * i], s[h * 32 + 2 * i + 1]), scale2,
                                        shift2),
                                 y0, y1);
                        const float p0 = ex2_approx(y0);
                        const float p1 = ex2_approx(y1);
                        sum2[i & 1] = f2_add(sum2[i & 1], f2_make(p0, p1));
                        if constexpr (DROP) {
                            if ((i & 1) == 0)
                                keep = dropout_keep4((uint32_t)(key0 + h * 32 + 2 * i),
                                                     (uint32_t)q_row, (uint32_t)it.bh,
                                                     p.drop.seed_lo, p.drop.seed_hi,
                                                     p.drop.threshold);
                            const uint32_t b2 = keep >> (2 * (i & 1));
                            pk[i] = pack2<BF16>((b2 & 1u) ? p0 : 0.0f, (b2 & 2u) ? p1 : 0.0f);
                        } else {
                            pk[i] = pack2<BF16>(p0, p1);
                        }
                    }
                    tmem_st16(s_addr + h * 16, pk);
                }
                float sa, sb, sc, sd;
                f2_split(sum2[0], sa, sb);
                f2_split(sum2[1], sc, sd);
                l_sum = l_sum * alpha + ((sa + sb) + (sc + sd));
                // S_t(j) was issued after PV_t(j-1), so every PV into O_t has completed: rescale
                // in place without waiting.
                if (__any_sync(0xffffffffu, rescale)) tmem_row_scale<D>(o_addr, alpha);
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(&bar_pf[t]);
                m_ref = m_new;
            }
            if (!ok) break;
            ok = wait_bounded(&bar_oready[t], (uint32_t)n_done & 1u, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            const bool valid = q_row < p.Lq;
            if (valid)
                p.lse[(size_t)it.bh * p.Lq + q_row] =
                    l_sum > 0.0f ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
            // This warp's 32 rows start at q_row - lane; those at or past Lq are not written.
            const int row0 = q_row - lane;
            uint8_t* orow0 = reinterpret_cast<uint8_t*>(p.o) + row_offset(p.so, it.bh, p.H, row0);
            const size_t row_bytes = (size_t)p.so.l * 2u;
            // The read-out finishes (tcgen05.ld waits) before this group publishes P_t0 of the
            // next item, which is what lets PV_t0 overwrite O_t.
            const float inv_l = l_sum > 0.0f ? (DROP ? p.drop.keep_scale : 1.0f) / l_sum : 0.0f;
            tmem_rows_to_global_staged<BF16, D>(
                o_addr, smem_u32(smem + C::kOffStage + warp * C::kStageBytes), orow0, row_bytes,
                p.Lq - row0, inv_l, lane);
            ps += n_mine;
            ++n_done;
        }
        if (!ok && lane == 0) record_timeout(p.status, abort_v);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Rows that see no key (the first Lq - Lk query rows under the causal mask when Lq > Lk): O = 0
// and LSE = -inf.  Enqueued only for such shapes; the attention kernel skips the query tiles in
// which no row sees a key and writes the same values for such rows of the tiles it does run.
template <int D>
__global__ void __launch_bounds__(256) fa_fwd_empty_rows_kernel(const FwdParams p, int rows) {
    constexpr int kChunks16 = D / 8;  // 16-byte pieces of a row
    const long long total = (long long)p.BH * rows * kChunks16;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(e % kChunks16);
        const long long r_all = e / kChunks16;
        const int bh = (int)(r_all / rows), r = (int)(r_all - (long long)bh * rows);
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.o) +
                                              row_offset(p.so, bh, p.H, r));
        dst[c] = make_uint4(0u, 0u, 0u, 0u);
        if (c == 0) p.lse[(size_t)bh * p.Lq + r] = -INFINITY;
    }
}

template <int D, bool BF16, bool CAUSAL, bool DROP>
cudaError_t launch_t(const FwdParams& p, cudaStream_t s) {
    using C = FwdCfg<D, BF16, CAUSAL>;
    auto kern = fa_fwd_kernel<D, BF16, CAUSAL, DROP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = fwd_grid(p.Lq, p.Lk, p.BH, CAUSAL, sm_count());
    return launch_kernel(kern, dim3((unsigned)grid), dim3(C::kThreads), C::kSmemBytes, s, p);
}

template <int D, bool BF16>
cudaError_t launch_d(const FwdParams& p, bool causal, bool drop, cudaStream_t s) {
    if (drop) return causal ? launch_t<D, BF16, true, true>(p, s) : launch_t<D, BF16, false, true>(p, s);
    return causal ? launch_t<D, BF16, true, false>(p, s) : launch_t<D, BF16, false, false>(p, s);
}

}  // namespace

cudaError_t launch_fwd_empty_rows(const FwdParams& p, int D, int rows, cudaStream_t s) {
    const long long work = (long long)p.BH * rows * (D / 8);
    const int sms = sm_count() > 0 ? sm_count() : 148;
    long long blocks = (work + 255) / 256;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    if (blocks < 1) blocks = 1;
    return D == 64 ? launch_kernel(fa_fwd_empty_rows_kernel<64>, dim3((unsigned)blocks), dim3(256),
                                   0, s, p, rows)
                   : launch_kernel(fa_fwd_empty_rows_kernel<128>, dim3((unsigned)blocks),
                                   dim3(256), 0, s, p, rows);
}

cudaError_t launch_fwd(const FwdParams& p, int D, bool bf16, bool causal, bool drop,
                       cudaStream_t s) {
    if (D == 64)
        return bf16 ? launch_d<64, true>(p, causal, drop, s) : launch_d<64, false>(p, causal, drop, s);
    return bf16 ? launch_d<128, true>(p, causal, drop, s) : launch_d<128, false>(p, causal, drop, s);
}

}  // namespace fa
