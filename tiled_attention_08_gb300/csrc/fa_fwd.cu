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
// GB300 layout.  One CTA owns TWO consecutive 128-row query tiles (A = 2p, B = 2p+1) of one
// head, so every K/V tile brought into shared memory feeds two tiles' worth of MMAs: the L2 ->
// SM traffic per FLOP is half of a one-tile CTA's, and each ring slot has twice as long to
// arrive.  The two tiles also give the tensor core independent work to interleave: while the
// softmax of tile A runs, the MMA warp computes tile B's PV and S, and the other way round.
//
// CTA roles (kSplit = 1: 352 threads at D = 128, 320 at D = 64):
//   softmax warps, one group of 4*kSplit per query tile (tile A first).  In a group, warp w
//                owns TMEM lanes 32*(w%4).. (query rows) and key columns
//                [kCols*(w/4), +kCols) of the tile's S (kCols = 128/kSplit); with kSplit > 1
//                the warps of a lane quadrant combine partial row maxima through shared memory
//                at a named barrier, with kSplit = 1 every thread owns a whole row;
//   next warp    TMA producer of Q_A, Q_B (once) and the K_j ring (at D = 64 K_j and V_j
//                together in one slot);
//   next warp    MMA issuer (one elected thread) and TMEM owner;
//   last warp    TMA producer of the V_j ring (D = 128 only).
// TMEM columns: S_A [0,128), S_B [128,256) (fp32; the 16-bit P of a tile overwrites the first
// 64 columns of its S and feeds the PV MMA straight from TMEM), O_A [256, 256+D),
// O_B [256+D, 256+2D).  MMA order: S_A0, S_B0, then for each key tile j: PV_Aj, S_A(j+1),
// PV_Bj, S_B(j+1).  S_t(j+1) is issued after PV_tj, so (tcgen05 MMAs of one thread run in
// issue order) it never overwrites a P still being read, and once the softmax sees S_t(j+1)
// every PV before it has finished: O_t may be rescaled in place with no further wait.
//
// Online softmax in the log2 domain: y = s * |scale| * log2(e), where s is the stored S.  For a
// negative scale the S contraction runs with its A operand negated (an exact sign flip set in
// the instruction descriptor), so s * |scale| = (Q K^T) * scale for either sign and the row
// maximum of the stored S is always the row maximum of the logits.  The running reference max m
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
    // D = 64: K_j and V_j share one slot of the K ring (one full and one empty barrier per
    // slot, one producer warp).  D = 128: separate K and V rings of two slots each, so that
    // K_{j+1} can land while V_j is still being read (measured faster at that size).
    static constexpr bool kMergedKV = (D == 64);
    static constexpr int kKStages = (D == 128) ? 2 : 4;        // K (or K/V) ring depth
    static constexpr int kVStages = (D == 128) ? 2 : 4;        // V ring depth (separate rings)
    static constexpr int kOffQ = 0;                            // Q_A, then Q_B
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kSmemBytes = kOffV + kVStages * kTileBytes + 1024;  // + alignment slack
    static constexpr int kSplit = 1;                           // softmax warps per lane quadrant
    static constexpr int kGroupWarps = 4 * kSplit;             // softmax warps per query tile
    static constexpr int kGroupThreads = kGroupWarps * 32;
    static constexpr int kSoftmaxWarps = 2 * kGroupWarps;
    static constexpr int kProducerWarp = kSoftmaxWarps;
    static constexpr int kMmaWarp = kSoftmaxWarps + 1;
    static constexpr int kVProducerWarp = kSoftmaxWarps + 2;
    static constexpr int kThreads = (kSoftmaxWarps + (kMergedKV ? 2 : 3)) * 32;
    static constexpr int kCols = 128 / kSplit;                 // S columns per softmax warp
    static constexpr int kOCols = D / kSplit;                  // O columns per softmax warp
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmS = 0;        // S of tile t at kTmS + 128*t
    static constexpr uint32_t kTmO = 256;      // O of tile t at kTmO + D*t
    static_assert(kTmO + 2 * D <= kTmemCols, "TMEM budget");
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
        bar_ve[C::kVStages], bar_sf[2], bar_pf[2], bar_oready[2], bar_fin;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    // Partial row maxima / sums exchanged between the column slices of a lane quadrant
    // (kSplit > 1 only; one element otherwise).
    constexpr int kRedRows = C::kSplit > 1 ? 128 : 1;
    __shared__ float red_max[2][2][C::kSplit][kRedRows];  // [tile][parity][column slice][row]
    __shared__ float red_sum[2][C::kSplit][kRedRows];     // [tile][column slice][row]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Heads in L2-sized groups; inside a group the heaviest tile pairs (most key tiles under
    // the causal mask) go first.
    const int n_pairs = (p.n_tiles + 1) >> 1;
    int bh, rank;
    tile_coords(blockIdx.x, p.BH, n_pairs, p.group, bh, rank);
    const int pair = n_pairs - 1 - rank;
    const int q_a = 2 * pair, q_b = 2 * pair + 1;  // the two query tiles
    const bool has_b = q_b < p.n_tiles;
    const int n_kv_a = CAUSAL ? q_a + 1 : p.n_tiles;  // key tiles each query tile sees
    const int n_kv_b = has_b ? (CAUSAL ? q_b + 1 : p.n_tiles) : 0;
    const int n_kv = has_b ? n_kv_b : n_kv_a;  // n_kv_a <= n_kv_b
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

    if (warp == C::kProducerWarp || (!C::kMergedKV && warp == C::kVProducerWarp)) {
        if constexpr (C::kMergedKV) {
            // ------------------------------ TMA producer ------------------------------
            // Q_A, Q_B once, then K_j and V_j together into ring slot j % kKStages.
            if (lane == 0) {
                tma_prefetch_desc(&p.tm_q);
                tma_prefetch_desc(&p.tm_k);
                tma_prefetch_desc(&p.tm_v);
                mbar_arrive_expect_tx(&bar_q, (has_b ? 2 : 1) * C::kTileBytes);
                for (int t = 0; t < (has_b ? 2 : 1); ++t)
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(smem + C::kOffQ + t * C::kTileBytes + c * kChunkBytes, &p.tm_q,
                                    &bar_q, c * kChunkElems, (t ? q_b : q_a) * kTileRows, bh);
                bool ok = true;
                int issued = 0;  // fills handed to the TMA unit
                for (int j = 0; j < n_kv; ++j) {
                    const int st = j % C::kKStages;
                    const uint32_t ph = (uint32_t)(j / C::kKStages) & 1u;
                    if (j >= C::kKStages && !wait_bounded(&bar_ke[st], ph ^ 1u, abort_v, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar_kf[st], 2 * C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_3d(smem + C::kOffK + st * C::kTileBytes + c * kChunkBytes, &p.tm_k,
                                    &bar_kf[st], c * kChunkElems, j * kTileRows, bh);
                        tma_load_3d(smem + C::kOffV + st * C::kTileBytes + c * kChunkBytes, &p.tm_v,
                                    &bar_kf[st], c * kChunkElems, j * kTileRows, bh);
                    }
                    issued = j + 1;
                }
                if (!ok) record_timeout(p.status, abort_v);
                // Drain: the newest fill of every slot must have landed before the CTA exits.
                // (These waits return at once on the normal path.)
                wait_bounded(&bar_q, 0, nullptr, p.timeout_ns);
                for (int j = issued - 1; j >= 0 && j >= issued - C::kKStages; --j)
                    wait_bounded(&bar_kf[j % C::kKStages], (uint32_t)(j / C::kKStages) & 1u, nullptr,
                                 p.timeout_ns);
            }
        } else {
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
                    mbar_arrive_expect_tx(&bar_q, (has_b ? 2 : 1) * C::kTileBytes);
                    for (int t = 0; t < (has_b ? 2 : 1); ++t)
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d(smem + C::kOffQ + t * C::kTileBytes + c * kChunkBytes, &p.tm_q,
                                        &bar_q, c * kChunkElems, (t ? q_b : q_a) * kTileRows, bh);
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
        }
    } else if (warp == C::kMmaWarp) {
        if constexpr (C::kMergedKV) {
            // ------------------------------ MMA issuer ------------------------------
            // The whole warp walks the loop (warp-uniform values); one elected lane issues.  A
            // wait between MMA groups can let the tensor pipe's short queue run dry, so each key
            // tile starts with the wait for the next K/V slot (the warp would idle until P of
            // tile A anyway); after that only P of tile A and P of tile B are waited for.
            bool ok = wait_warp(&bar_q, 0, abort_v, p.timeout_ns);
            auto wait_kv = [&](int j) -> bool {  // K_j and V_j landed
                if (!wait_warp(&bar_kf[j % C::kKStages], (uint32_t)(j / C::kKStages) & 1u, abort_v,
                               p.timeout_ns))
                    return false;
                tc_fence_after_sync();
                return true;
            };
            auto issue_s = [&](int t, int j) {
                const uint64_t qd = sdesc_kmajor_sw128(smem_u32(smem + C::kOffQ + t * C::kTileBytes));
                const uint64_t kd =
                    sdesc_kmajor_sw128(smem_u32(smem + C::kOffK + (j % C::kKStages) * C::kTileBytes));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    mma_ss_w(tmem + C::kTmS + 128 * t, sdesc_advance(qd, off), sdesc_advance(kd, off),
                           C::kIdescS | p.s_negate, kk > 0 ? 1u : 0u);
                }
                mma_commit_w(&bar_sf[t]);
            };
            auto issue_pv = [&](int t, int j) -> bool {
                if (!wait_warp(&bar_pf[t], (uint32_t)j & 1u, abort_v, p.timeout_ns))
                    return false;
                tc_fence_after_sync();
                const uint64_t vd = sdesc_mnmajor_sw128(
                    smem_u32(smem + C::kOffV + (j % C::kKStages) * C::kTileBytes), kChunkBytes);
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk) {
                    const uint64_t bd = sdesc_advance(vd, kk * 2048);
                    mma_ts_w(tmem + C::kTmO + D * t, tmem + C::kTmS + 128 * t + kk * 8, bd,
                           C::kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                if (j + 1 == (t ? n_kv_b : n_kv_a)) mma_commit_w(&bar_oready[t]);  // O_t is final
                return true;
            };
            if (ok && n_kv > 0) {
                ok = wait_kv(0);
                if (ok) {
                    issue_s(0, 0);
                    if (n_kv_b > 0) issue_s(1, 0);
                }
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const bool next = j + 1 < n_kv;
                // Slot j+1 first, while this warp idles until P_A(j) anyway.
                if (next && !wait_kv(j + 1)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int n_t = t ? n_kv_b : n_kv_a;
                    if (!ok) break;
                    if (j < n_t && !issue_pv(t, j)) {
                        ok = false;
                        break;
                    }
                    if (next && j + 1 < n_t) issue_s(t, j + 1);
                }
                if (!ok) break;
                mma_commit_w(&bar_ke[j % C::kKStages]);  // K_j (S_j) and V_j (both PV_j) consumed
            }
            if (!ok && lane == 0) record_timeout(p.status, abort_v);
            // Every issued MMA must finish before TMEM is released.
            mma_commit_w(&bar_fin);
            wait_warp(&bar_fin, 0, nullptr, p.timeout_ns);
        } else {
            // ------------------------------ MMA issuer ------------------------------
            // The whole warp walks the loop (warp-uniform values); one elected lane issues.  Each
            // key tile starts with the ring waits (V_j, K_{j+1}) while the warp would idle until
            // P of tile A anyway; after that only the two P waits sit between MMA groups.
            bool ok = wait_warp(&bar_q, 0, abort_v, p.timeout_ns);
            int k_ready = -1;  // newest K tile known to have landed
            auto wait_k = [&](int j) -> bool {
                if (k_ready >= j) return true;
                const int st = j % C::kKStages;
                if (!wait_warp(&bar_kf[st], (uint32_t)(j / C::kKStages) & 1u, abort_v,
                                  p.timeout_ns))
                    return false;
                tc_fence_after_sync();
                k_ready = j;
                return true;
            };
            auto issue_s = [&](int t, int j) {
                const uint64_t qd = sdesc_kmajor_sw128(smem_u32(smem + C::kOffQ + t * C::kTileBytes));
                const uint64_t kd =
                    sdesc_kmajor_sw128(smem_u32(smem + C::kOffK + (j % C::kKStages) * C::kTileBytes));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    mma_ss_w(tmem + C::kTmS + 128 * t, sdesc_advance(qd, off), sdesc_advance(kd, off),
                           C::kIdescS | p.s_negate, kk > 0 ? 1u : 0u);
                }
                mma_commit_w(&bar_sf[t]);
            };
            auto issue_pv = [&](int t, int j) -> bool {  // V_j was waited for at the tile's start
                const int st = j % C::kVStages;
                if (!wait_warp(&bar_pf[t], (uint32_t)j & 1u, abort_v, p.timeout_ns))
                    return false;
                tc_fence_after_sync();
                const uint64_t vd =
                    sdesc_mnmajor_sw128(smem_u32(smem + C::kOffV + st * C::kTileBytes), kChunkBytes);
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk) {
                    const uint64_t bd = sdesc_advance(vd, kk * 2048);
                    mma_ts_w(tmem + C::kTmO + D * t, tmem + C::kTmS + 128 * t + kk * 8, bd,
                           C::kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                if (j + 1 == (t ? n_kv_b : n_kv_a)) mma_commit_w(&bar_oready[t]);  // O_t is final
                return true;
            };
            if (ok && n_kv > 0) {
                ok = wait_k(0);
                if (ok) {
                    issue_s(0, 0);
                    if (n_kv_b > 0) issue_s(1, 0);
                    mma_commit_w(&bar_ke[0]);
                }
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const bool next = j + 1 < n_kv;
                // Ring waits first, while this warp idles until P_A(j) anyway: then each P wait
                // is followed by PV and the next S with no wait in between.
                if (!wait_warp(&bar_vf[j % C::kVStages], (uint32_t)(j / C::kVStages) & 1u, abort_v,
                               p.timeout_ns) ||
                    (next && !wait_k(j + 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int n_t = t ? n_kv_b : n_kv_a;
                    if (!ok) break;
                    if (j < n_t && !issue_pv(t, j)) {
                        ok = false;
                        break;
                    }
                    if (next && j + 1 < n_t) {
                        if (!wait_k(j + 1)) {
                            ok = false;
                            break;
                        }
                        issue_s(t, j + 1);
                    }
                }
                if (!ok) break;
                mma_commit_w(&bar_ve[j % C::kVStages]);                // V_j read by both PVs
                if (next) mma_commit_w(&bar_ke[(j + 1) % C::kKStages]);  // K_{j+1} read by both S
            }
            if (!ok && lane == 0) record_timeout(p.status, abort_v);
            // Every issued MMA must finish before TMEM is released.
            mma_commit_w(&bar_fin);
            wait_warp(&bar_fin, 0, nullptr, p.timeout_ns);
        }
    } else {
        // ------------------------------ softmax warps ------------------------------
        constexpr int kC = C::kCols;
        const int t = warp / C::kGroupWarps;             // query tile of this group
        const int gw = warp % C::kGroupWarps;
        const int quad = gw & 3;                         // TMEM lane quadrant
        const int part = gw >> 2;                        // which kC key columns of the tile
        const uint32_t grp_bar = 1 + t * 4 + quad;       // named barrier of the quadrant
        constexpr uint32_t kGrpThreads = 32 * C::kSplit;
        const int row = quad * 32 + lane;                // row inside the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int q_row = (t ? q_b : q_a) * kTileRows + row;
        const int n_mine = t ? n_kv_b : n_kv_a;
        const int c0 = part * kC;
        const uint32_t s_addr = tmem + lane_off + C::kTmS + 128 * t;
        const uint32_t o_addr = tmem + lane_off + C::kTmO + D * t + part * C::kOCols;
        float m_ref = -INFINITY;
        float l_sum = 0.0f;  // over this warp's columns only
        bool ok = true;
        for (int j = 0; j < n_mine; ++j) {
            const int par = j & 1;  // parity slot of the shared-memory max exchange
            ok = wait_bounded(&bar_sf[t], (uint32_t)j & 1u, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            float s[kC];
            float mx = -INFINITY;
            if (ok) {
                tc_fence_after_sync();
                uint32_t r[kC];
                tmem_ld_cols<kC>(s_addr + c0, r);
#pragma unroll
                for (int i = 0; i < kC; ++i) s[i] = __uint_as_float(r[i]);
                const int key0 = j * kTileRows + c0;
                if ((CAUSAL && j == n_mine - 1) || j * kTileRows + kTileRows > p.L) {
                    const int lim = CAUSAL ? min(p.L - 1, q_row) : (p.L - 1);
#pragma unroll
                    for (int c = 0; c < kC; ++c)
                        if (key0 + c > lim) s[c] = -INFINITY;
                }
                // Row max: four independent chains of three-input maxima.
                float m4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) m4[u] = fmaxf(s[u], s[u + 4]);
#pragma unroll
                for (int c = 8; c < kC; c += 8) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) m4[u] = fmax3(m4[u], s[c + u], s[c + 4 + u]);
                }
                mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
            }
            if constexpr (C::kSplit > 1) {
                red_max[t][par][part][row] = mx;
                // All slices have read their S columns (P may now overwrite them) and
                // published their partial maxima.
                ok = bar_and(grp_bar, kGrpThreads, ok);
                if (!ok) break;
#pragma unroll
                for (int q = 0; q < C::kSplit; ++q) mx = fmaxf(mx, red_max[t][par][q][row]);
            } else {
                if (!ok) break;  // warp-uniform: the warp owns its rows alone
            }
            const float m_cand = mx * p.scale_log2;
            float m_new = m_ref;
            if (m_cand > m_ref + kRescaleThreshold) m_new = m_cand;
            const bool rescale = (j > 0) && (m_new != m_ref);
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            const float alpha = rescale ? ex2_approx(m_ref - m_new) : 1.0f;
            // Two columns per instruction for the scale-and-shift and the running sum.
            const uint64_t scale2 = f2_make(p.scale_log2, p.scale_log2);
            const uint64_t shift2 = f2_make(-m_use, -m_use);
            uint64_t sum2[2] = {0ull, 0ull};  // (+0.0f, +0.0f)
#pragma unroll
            for (int h = 0; h < kC / 32; ++h) {  // 32 columns -> 16 packed TMEM columns at a time
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
                tmem_st16(s_addr + part * (kC / 2) + h * 16, pk);
            }
            float sa, sb, sc, sd;
            f2_split(sum2[0], sa, sb);
            f2_split(sum2[1], sc, sd);
            l_sum = l_sum * alpha + ((sa + sb) + (sc + sd));
            // S_t(j) was issued after PV_t(j-1), so every PV into O_t has completed: rescale
            // in place without waiting.
            if (__any_sync(0xffffffffu, rescale)) tmem_row_scale<C::kOCols>(o_addr, alpha);
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bar_pf[t]);
            m_ref = m_new;
        }
        if (ok && n_mine > 0) {
            ok = wait_bounded(&bar_oready[t], 0, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
        }
        if constexpr (C::kSplit > 1) {
            red_sum[t][part][row] = l_sum;
            ok = bar_and(grp_bar, kGrpThreads, ok);
        }
        if (!ok) {
            if (lane == 0) record_timeout(p.status, abort_v);
        } else if (n_mine > 0) {
            tc_fence_after_sync();
            float l_tot = l_sum;
            if constexpr (C::kSplit > 1) {
                l_tot = 0.0f;
#pragma unroll
                for (int q = 0; q < C::kSplit; ++q) l_tot += red_sum[t][q][row];
            }
            const bool valid = q_row < p.L;
            if (valid && part == 0) p.lse[(size_t)bh * p.L + q_row] = (m_ref + log2f(l_tot)) * kLn2;
            uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) + ((size_t)bh * p.L + q_row) * D * 2 +
                            part * C::kOCols * 2;
            tmem_row_to_global<BF16, C::kOCols>(o_addr, orow, 1.0f / l_tot, valid);
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
    const unsigned grid = (unsigned)((p.n_tiles + 1) / 2) * (unsigned)p.BH;
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
