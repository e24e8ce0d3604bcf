// fa_bwd_dkdv.cu -- attention backward, dK and dV: per (b*h, 128-key tile), one CTA each or
// persistent.
//
// Recompute-based backward ("FlashAttention data-flow optimisation: MI50 memory and bandwidth
// bottlenecks", section 2.2, third layer): P is rebuilt tile by tile from Q, K and the saved
// log-sum-exp instead of being stored.  For a key tile j and every query tile i that can see it
// (i >= j under the causal mask):
//   S^T  = K_j Q_i^T                      (tcgen05, both operands K-major in shared memory)
//   dP^T = V_j dO_i^T
//   P^T  = exp2(S^T * scale*log2e - LSE_i*log2e)        (per column: query)
//   dS^T = P^T o (dP^T - Delta_i)
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i   (A operand = 16-bit P^T / dS^T written back to TMEM)
// and at the end dK_j is multiplied by the softmax scale.
//
// CTA roles: 4*kSplit elementwise warps (warp w: key rows 32*(w%4).. == TMEM lanes, query
// columns [kCols*(w/4), +kCols)), then one TMA producer warp (per work item K_j and V_j; then
// Q_i with -LSE_i*log2e into a Q ring and dO_i with Delta_i into a dO ring one slot shallower,
// Q one tile ahead) and one MMA-issuer warp that also owns TMEM.
// TMEM: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D, 256+2D).
//
// Pipeline.  The elementwise warps read S^T into registers (P^T stays there) and at once
// release the S^T columns, so the MMA warp issues S^T of the NEXT query tile right away.
// Once dP^T has been read too, the 16-bit P^T and dS^T are written side by side into the
// dP^T columns (P^T at [128,192), dS^T at [192,256)), which feed the dK and dV MMAs (dK first:
// it releases Q_i, whose slot the next-but-one S^T needs); the next dP^T is issued after
// those.  So the P phase of query tile i+1 runs while the tensor core does dK_i, dV_i and
// dP^T_{i+1}, instead of waiting for them.
//
// Scheduling (dkdv_grid).  A work item is one key tile of one head, ordered heaviest first
// (key tile 0 sees every query tile under the causal mask) inside L2-sized head groups
// (tile_coords).  For rows of few query tiles the grid is one CTA per SM, each taking the next
// item from the pass's work counter whenever it is ready for one (fa_queue.cuh), so a CTA's
// fixed cost is paid once per SM and the items stay balanced: the Q / dO
// rings run on from one item to the next, the next item's K_j / V_j are loaded as soon as the
// current item's last S^T and dP^T have completed (at D = 64 into a second K/V slot, at once),
// and the next item's first S^T and dP^T run while the elementwise warps read out dK and dV.
// Those warps publish P^T / dS^T of the next item's first query tile only after the read-out,
// and dK / dV of that tile (which overwrite the accumulators) wait for that, so no extra
// barrier guards the accumulators.  For long rows the grid is one CTA per item.  Barrier
// phases count query tiles (ring slots, S^T / dP^T / P^T) or items (K/V slots, done) over the
// CTA's lifetime.
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_queue.cuh"
#include "fa_sched.h"

namespace fa {
namespace {

// DQA: the dK/dV pass also computes dQ_i += dS_i K_j and reduces it into an fp32 accumulator in
// global memory (the deterministic alternative is the separate dQ pass).
template <int D, bool BF16, bool CAUSAL, bool DQA = false>
struct DkdvCfg {
    static constexpr int kChunks = D / kChunkElems;
    static constexpr int kTileBytes = kTileRows * D * 2;
    // Q_i is needed early (by S^T) and late (by dK), dO_i only in between, so the Q ring is one
    // slot deeper than the dO ring (D = 64: five and four slots; six and five ran slower).  At
    // D = 128 the tiles then fill 224 KB of the 227 KB a block may have, so everything else
    // (the -LSE*log2e and Delta vectors, the barriers) lives in the same 1024-aligned dynamic
    // allocation and no alignment slack is requested.
    static constexpr int kQStages = (D == 128 || DQA) ? 3 : 5;
    static constexpr int kOStages = (D == 128) ? 2 : 4;
    // K_j / V_j slots: two at D = 64, so the next item's key tile lands while this one runs;
    // one at D = 128, where the tiles already take 224 KB.
    static constexpr int kKVSlots = (D == 128 || DQA) ? 1 : 2;
    // With three or more dO slots the MMA warp waits for dO_{t+1} before issuing dK_t, and the
    // producer issues dO_{t+1} only after Q_{t+2}, whose slot dK_{t+2-kQStages} frees: with two
    // Q slots that is dK_t itself, a circular wait.
    static_assert(kOStages < 3 || kQStages >= 3, "early dO wait needs three or more Q slots");
    static constexpr int kVecBytes = kTileRows * 4;  // one fp32 vector of a 128-row tile
    static constexpr int kOffK = 0;           // slot s: K at kOffK + 2*s*kTileBytes, then V
    static constexpr int kOffQ = 2 * kKVSlots * kTileBytes;
    static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
    // DQA: dS_i (128 queries x 128 keys, 16-bit), the A operand of dQ_i = dS_i K_j, written by
    // the elementwise warps in the MN-major 128-byte-swizzled layout (queries contiguous); two
    // buffers (query tile i in buffer i % 2), so dS_{i+1} never waits for dQ_i.  They take the
    // room of two Q slots (three instead of five).
    static constexpr int kOffDS = kOffDO + kOStages * kTileBytes;
    static constexpr int kDSTile = kTileRows * kTileRows * 2;
    static constexpr int kDSBytes = DQA ? 2 * kDSTile : 0;
    static constexpr int kOffNlse = kOffDS + kDSBytes;                // per Q slot
    static constexpr int kOffDelta = kOffNlse + kQStages * kVecBytes;  // per dO slot
    static constexpr int kOffBar = kOffDelta + kOStages * kVecBytes;
    static constexpr int kSplit = 4;  // elementwise warps per TMEM lane quadrant
    static constexpr int kEwWarps = 4 * kSplit;
    static constexpr int kEwThreads = kEwWarps * 32;
    static constexpr int kProducerWarp = kEwWarps;
    static constexpr int kMmaWarp = kEwWarps + 1;
    static constexpr int kThreads = (kEwWarps + 2) * 32;
    static constexpr int kCols = 128 / kSplit;  // query columns per elementwise warp
    static constexpr int kOutCols = D / kSplit;  // dK/dV columns per elementwise warp
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmST = 0, kTmDPT = 128, kTmDV = 256, kTmDK = 256 + D;
    static constexpr uint32_t kIdescS = idesc_f16(BF16, 128, 128, false, false);
    static constexpr uint32_t kIdescG = idesc_f16(BF16, 128, D, false, true);
    // DQA: two dQ accumulators of D columns after dK (TMEM has room for them at D = 64 only).
    static constexpr uint32_t kTmDQ = 256 + 2 * D;
    static constexpr uint32_t kIdescQ = idesc_f16(BF16, 128, D, true, true);
    static_assert(!DQA || D == 64, "dQ by reduction needs 2*D more TMEM columns: D = 64 only");
};

// Barriers and small shared state, placed after the tiles in dynamic shared memory.  dqf / dqe
// (DQA only): dQ accumulator b computed / read out.
template <int KVS, int QS, int OS>
struct DkdvBars {
    uint64_t kvf[KVS], kve[KVS], qf[QS], qe[QS], of[OS], oe[OS], sf, df, sr, ppd, done, fin;
    uint64_t dqf[2], dqe[2];
    WorkQueue queue;  // persistent kernel: the items, fetched from the pass's counter
    uint32_t tmem_base;
    int abort;
};

template <int D, bool BF16, bool CAUSAL, bool DQA = false>
using DkdvBarsT = DkdvBars<DkdvCfg<D, BF16, CAUSAL, DQA>::kKVSlots,
                           DkdvCfg<D, BF16, CAUSAL, DQA>::kQStages,
                           DkdvCfg<D, BF16, CAUSAL, DQA>::kOStages>;

template <int D, bool BF16, bool CAUSAL, bool DQA = false>
constexpr int dkdv_smem_bytes() {
    using C = DkdvCfg<D, BF16, CAUSAL, DQA>;
    return C::kOffBar + (int)sizeof(DkdvBarsT<D, BF16, CAUSAL, DQA>);
}

// One work item: key tile kt of head bh and the query tiles [it0, it0 + n_it) that see it.
struct DkdvItem {
    int bh, b, h, kt, it0, n_it;
};

// Work id -> item: ids follow tile_coords (heads in L2-sized groups, key tile 0, the heaviest,
// first).  The persistent kernel takes its ids from the pass's counter (fa_queue.cuh).
template <bool CAUSAL>
__device__ __forceinline__ void dkdv_item(const BwdParams& p, int id, DkdvItem& it) {
    tile_coords(id, p.BH, p.n_ktiles, p.group, it.bh, it.kt);  // key tile 0 (heaviest) first
    it.b = it.bh / p.H;
    it.h = it.bh - it.b * p.H;
    it.it0 = k_tile_q0(it.kt, p.Lq, p.Lk, CAUSAL);
    it.n_it = p.n_qtiles - it.it0;
}

// One CTA per (b*h, key tile), in tile_coords order (the hardware's block scheduler balances
// the causal tiles): for rows of many query tiles, where a CTA's fixed cost is a small share.
// DROP: dropout on P (p.drop): dV accumulates (P o keep)^T dO and is scaled by 1/(1-p) on the
// way out; dS^T = P^T o (dP^T o Z^T - Delta) with Z the keep mask times 1/(1-p).
// DQA: also dQ_i += dS_i K_j into p.dq_acc.  The elementwise warps write dS_i to shared memory
// (buffer i % 2) beside the 16-bit dS_i^T they put in TMEM; the MMA warp issues dQ_i = dS_i K_j
// (A = dS_i from shared memory, B = the K tile read MN-major) into TMEM accumulator i % 2 after
// dP^T of the next query tile; the elementwise warps wait for it, read it out and reduce it
// into global memory with 16-byte red.add after publishing P^T / dS^T of the next query tile,
// then free the accumulator.  Buffer i % 2 is written again (dS_{i+2}) only after that
// read-out has seen dQ_i complete.
template <int D, bool BF16, bool CAUSAL, bool DROP, bool DQA>
__global__ void __launch_bounds__(DkdvCfg<D, BF16, CAUSAL, DQA>::kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using C = DkdvCfg<D, BF16, CAUSAL, DQA>;
    // The kernel declares no static shared memory, so its dynamic shared memory starts at the
    // block's shared window, which is 1024-byte aligned; checked here (the 128-byte swizzle
    // needs it) before any barrier, TMEM or copy is touched.
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, (int)kDevBadShared);  // -> FA_ERR_CUDA
        return;
    }
    // Q_i (+ LSE_i) and dO_i (+ Delta_i) have their own rings and full/empty barriers: Q_i is
    // released by dK_i, issued first, so the load of a later Q tile (needed early, by S^T)
    // starts sooner.
    auto& bars = *reinterpret_cast<DkdvBarsT<D, BF16, CAUSAL, DQA>*>(smem + C::kOffBar);
    uint64_t& bar_kv = bars.kvf[0];
    uint64_t* bar_qf = bars.qf;
    uint64_t* bar_qe = bars.qe;
    uint64_t* bar_of = bars.of;
    uint64_t* bar_oe = bars.oe;
    uint64_t& bar_sf = bars.sf;
    uint64_t& bar_df = bars.df;
    uint64_t& bar_sr = bars.sr;
    uint64_t& bar_ppd = bars.ppd;
    uint64_t& bar_done = bars.done;
    uint64_t& bar_fin = bars.fin;
    uint32_t& tmem_base_sh = bars.tmem_base;
    int& abort_flag = bars.abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Heads in L2-sized groups (their Q/dO/LSE/Delta are streamed by every key tile); inside
    // a group key tile 0 first: it has the most query tiles under the causal mask.
    int bh, kt;
    tile_coords(blockIdx.x, p.BH, p.n_ktiles, p.group, bh, kt);
    const int hb = bh / p.H, hh = bh - hb * p.H;  // batch and head of bh
    const int it0 = k_tile_q0(kt, p.Lq, p.Lk, CAUSAL);
    const int n_it = p.n_qtiles - it0;
    volatile int* abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar_kv, 1);
        for (int s = 0; s < C::kQStages; ++s) {
            mbar_init(&bar_qf[s], 1);
            mbar_init(&bar_qe[s], 1);
        }
        for (int s = 0; s < C::kOStages; ++s) {
            mbar_init(&bar_of[s], 1);
            mbar_init(&bar_oe[s], 1);
        }
        mbar_init(&bar_sf, 1);
        mbar_init(&bar_df, 1);
        mbar_init(&bar_sr, C::kEwThreads);   // S^T read: its columns may be overwritten
        mbar_init(&bar_ppd, C::kEwThreads);  // P^T and dS^T written into the dP^T columns
        mbar_init(&bar_done, 1);
        mbar_init(&bar_fin, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.dqf[b], 1);
            mbar_init(&bars.dqe[b], C::kEwThreads);
        }
        mbar_fence_init();
    }
    if (warp == C::kMmaWarp) tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    if (warp == C::kProducerWarp) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_do);
            mbar_arrive_expect_tx(&bar_kv, 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_4d(smem + C::kOffK + c * kChunkBytes, &p.tm_k, &bar_kv, c * kChunkElems,
                            kt * kTileRows, hh, hb);
                tma_load_4d(smem + C::kOffK + C::kTileBytes + c * kChunkBytes, &p.tm_v, &bar_kv,
                            c * kChunkElems, kt * kTileRows, hh, hb);
            }
            bool ok = true;
            int issued_q = 0, issued_o = 0;
            auto load_q = [&](int t) -> bool {  // Q_t and -LSE_t*log2e into Q slot t % kQStages
                const int st = t % C::kQStages;
                if (t >= C::kQStages &&
                    !wait_bounded(&bar_qe[st], ((uint32_t)(t / C::kQStages) & 1u) ^ 1u, abort_v,
                                  p.timeout_ns))
                    return false;
                const int it = it0 + t;
                mbar_arrive_expect_tx(&bar_qf[st], C::kTileBytes + C::kVecBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(smem + C::kOffQ + st * C::kTileBytes + c * kChunkBytes, &p.tm_q,
                                &bar_qf[st], c * kChunkElems, it * kTileRows, hh, hb);
                bulk_load(smem + C::kOffNlse + st * C::kVecBytes,
                          p.nlse2_pad + (size_t)bh * p.Lqpad + (size_t)it * kTileRows, C::kVecBytes,
                          &bar_qf[st]);
                issued_q = t + 1;
                return true;
            };
            auto load_do = [&](int t) -> bool {  // dO_t and Delta_t into dO slot t % kOStages
                const int st = t % C::kOStages;
                if (t >= C::kOStages &&
                    !wait_bounded(&bar_oe[st], ((uint32_t)(t / C::kOStages) & 1u) ^ 1u, abort_v,
                                  p.timeout_ns))
                    return false;
                const int it = it0 + t;
                mbar_arrive_expect_tx(&bar_of[st], C::kTileBytes + C::kVecBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(smem + C::kOffDO + st * C::kTileBytes + c * kChunkBytes, &p.tm_do,
                                &bar_of[st], c * kChunkElems, it * kTileRows, hh, hb);
                bulk_load(smem + C::kOffDelta + st * C::kVecBytes,
                          p.delta_pad + (size_t)bh * p.Lqpad + (size_t)it * kTileRows, C::kVecBytes,
                          &bar_of[st]);
                issued_o = t + 1;
                return true;
            };
            // Q runs one tile ahead of dO: Q_{t+1} only waits for dK_{t+1-kQStages}.
            if (n_it > 0) ok = load_q(0);
            for (int t = 0; ok && t < n_it; ++t) {
                if (t + 1 < n_it) ok = load_q(t + 1);
                ok = ok && load_do(t);
            }
            if (!ok) record_timeout(p.status, abort_v);
            // Drain: no copy may still be landing when the CTA exits.
            wait_bounded(&bar_kv, 0, nullptr, p.timeout_ns);
            for (int t = issued_q - 1; t >= 0 && t >= issued_q - C::kQStages; --t)
                wait_bounded(&bar_qf[t % C::kQStages], (uint32_t)(t / C::kQStages) & 1u, nullptr,
                             p.timeout_ns);
            for (int t = issued_o - 1; t >= 0 && t >= issued_o - C::kOStages; --t)
                wait_bounded(&bar_of[t % C::kOStages], (uint32_t)(t / C::kOStages) & 1u, nullptr,
                             p.timeout_ns);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------ MMA issuer ------------------------------
        // The whole warp walks the loop (warp-uniform values); one elected lane issues.
        const uint32_t k_base = smem_u32(smem + C::kOffK);
        const uint32_t v_base = smem_u32(smem + C::kOffK + C::kTileBytes);
        auto q_base = [&](int t) {
            return smem_u32(smem + C::kOffQ + (t % C::kQStages) * C::kTileBytes);
        };
        auto do_base = [&](int t) {
            return smem_u32(smem + C::kOffDO + (t % C::kOStages) * C::kTileBytes);
        };
        auto wait_q = [&](int t) {  // Q_t landed
            const bool r = wait_warp(&bar_qf[t % C::kQStages], (uint32_t)(t / C::kQStages) & 1u,
                                     abort_v, p.timeout_ns);
            tc_fence_after_sync();
            return r;
        };
        auto wait_do = [&](int t) {  // dO_t landed
            const bool r = wait_warp(&bar_of[t % C::kOStages], (uint32_t)(t / C::kOStages) & 1u,
                                     abort_v, p.timeout_ns);
            tc_fence_after_sync();
            return r;
        };
        const uint64_t kdesc = sdesc_kmajor_sw128(k_base);
        const uint64_t vdesc = sdesc_kmajor_sw128(v_base);
        auto issue_st = [&](int t) {  // S^T = K Q_t^T
            const uint64_t qd = sdesc_kmajor_sw128(q_base(t));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                mma_ss_w(tmem + C::kTmST, sdesc_advance(kdesc, off), sdesc_advance(qd, off),
                       C::kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bar_sf);
        };
        auto issue_dpt = [&](int t) {  // dP^T = V dO_t^T
            const uint64_t dd = sdesc_kmajor_sw128(do_base(t));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                mma_ss_w(tmem + C::kTmDPT, sdesc_advance(vdesc, off), sdesc_advance(dd, off),
                       C::kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bar_df);
        };
        bool ok = wait_warp(&bar_kv, 0, abort_v, p.timeout_ns);
        if (ok && n_it > 0) {
            ok = wait_q(0);
            if (ok) issue_st(0);
            ok = ok && wait_do(0);
            if (ok) issue_dpt(0);
        }
        for (int t = 0; t < n_it && ok; ++t) {
            const uint32_t par = (uint32_t)t & 1u;
            if (t + 1 < n_it) {
                // S^T of the next query tile as soon as this one's S^T has been read.
                if (!wait_warp(&bar_sr, par, abort_v, p.timeout_ns) || !wait_q(t + 1)) {
                    ok = false;
                    break;
                }
                issue_st(t + 1);
            }
            // With three or more dO slots, dO_{t+1} has normally landed by now: wait for it here
            // so dK_t, dV_t and dP^T_{t+1} go out as one batch.  With two it may still be in
            // flight, and waiting here would hold up dK_t and dV_t (measured slower).
            constexpr bool kEarlyDo = C::kOStages >= 3;
            if ((kEarlyDo && t + 1 < n_it && !wait_do(t + 1)) ||
                !wait_warp(&bar_ppd, par, abort_v, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t acc0 = t > 0 ? 1u : 0u;
            const uint64_t dod = sdesc_mnmajor_sw128(do_base(t), kChunkBytes);
            const uint64_t qmd = sdesc_mnmajor_sw128(q_base(t), kChunkBytes);
#pragma unroll
            for (int kk = 0; kk < kTileRows / 16; ++kk)
                mma_ts_w(tmem + C::kTmDK, tmem + C::kTmDPT + 64 + kk * 8,
                       sdesc_advance(qmd, kk * 2048), C::kIdescG, (acc0 || kk > 0) ? 1u : 0u);
            mma_commit_w(&bar_qe[t % C::kQStages]);  // Q_t fully read
#pragma unroll
            for (int kk = 0; kk < kTileRows / 16; ++kk)
                mma_ts_w(tmem + C::kTmDV, tmem + C::kTmDPT + kk * 8,
                       sdesc_advance(dod, kk * 2048), C::kIdescG, (acc0 || kk > 0) ? 1u : 0u);
            mma_commit_w(&bar_oe[t % C::kOStages]);  // dO_t fully read
            if (t + 1 < n_it) {                     // after dV_t, dK_t read the dP^T columns
                if (!kEarlyDo && !wait_do(t + 1)) {
                    ok = false;
                    break;
                }
                issue_dpt(t + 1);
            }
            if constexpr (DQA) {  // dQ_t = dS_t K into accumulator t % 2, once read out twice ago
                const int b = t & 1;
                if (t >= 2 && !wait_warp(&bars.dqe[b], ((uint32_t)(t - 2) >> 1) & 1u, abort_v,
                                         p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t dsd =
                    sdesc_mnmajor_sw128(smem_u32(smem + C::kOffDS + b * C::kDSTile), kChunkBytes);
                const uint64_t kmd = sdesc_mnmajor_sw128(k_base, kChunkBytes);
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk)
                    mma_ss_w(tmem + C::kTmDQ + b * D, sdesc_advance(dsd, kk * 2048),
                             sdesc_advance(kmd, kk * 2048), C::kIdescQ, kk > 0 ? 1u : 0u);
                mma_commit_w(&bars.dqf[b]);
            }
        }
        if (ok) mma_commit_w(&bar_done);
        if (!ok && lane == 0) record_timeout(p.status, abort_v);
        mma_commit_w(&bar_fin);
        wait_warp(&bar_fin, 0, nullptr, p.timeout_ns);
    } else {
        // ------------------------------ elementwise warps ------------------------------
        constexpr int kC = C::kCols;
        const int quad = warp & 3;              // TMEM lane quadrant (key rows)
        const int part = warp >> 2;             // which kC query columns
        const uint32_t grp_bar = 1 + quad;      // named barrier of the quadrant
        constexpr uint32_t kGrpThreads = 32 * C::kSplit;
        const int row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int key = kt * kTileRows + row;
        const int c0 = part * kC;
        // DQA: dQ_tq (TMEM accumulator tq % 2; lane = query row (it0 + tq) * 128 + lane) into
        // p.dq_acc.  A TMEM load gives each thread 16 columns of one row, and 16-byte
        // reductions from 32 rows at once would touch 32 memory lines per instruction; so the
        // quadrant's four warps stage their rows in shared memory (the dS buffer of query tile
        // tq, which dQ_tq has finished reading: the 8 KB that this quadrant's dS rows occupy,
        // rows 256 B apart with the 16-byte unit index XORed by row % 16) and each warp then
        // reduces 8 whole rows, two 256-byte rows per instruction.  Every warp of the quadrant
        // calls it the same number of times (it holds the quadrant's named barrier); `go`
        // false skips the work, and the result is the quadrant's AND of it.
        auto dq_reduce = [&](int tq, bool go) -> bool {
            constexpr int kQc = 16;
            static_assert(!DQA || D / C::kSplit == kQc, "16 dQ columns per warp slice");
            static_assert(!DQA || D == 64, "256-byte dQ rows");
            uint8_t* stage = smem + C::kOffDS + (tq & 1) * C::kDSTile + quad * 4096;
            auto unit = [&](int r, int u) {  // 16-byte unit u of the quadrant's row r
                return stage + (r >> 4) * kChunkBytes + (r & 15) * 256 + ((u ^ (r & 15)) << 4);
            };
            if (go) {
                tc_fence_after_sync();
                uint32_t r[kQc];
                tmem_ld16(tmem + lane_off + C::kTmDQ + (tq & 1) * D + part * kQc, r);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4*>(unit(lane, part * 4 + j)) =
                        make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            }
            go = bar_and(grp_bar, kGrpThreads, go);
            if (go) {
                const int r0 = part * 8 + (lane >> 4), u = lane & 15;
                float* dst = p.dq_acc +
                             ((size_t)bh * p.Lqpad + (size_t)(it0 + tq) * kTileRows + quad * 32) *
                                 D +
                             u * 4;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rr = r0 + 2 * i;
                    const float4 x = *reinterpret_cast<const float4*>(unit(rr, u));
                    red_add_v4(dst + (size_t)rr * D, x.x, x.y, x.z, x.w);
                }
            }
            return go;
        };
        bool ok = true;
        for (int t = 0; t < n_it; ++t) {
            const int it = it0 + t;
            const int qs = t % C::kQStages, os = t % C::kOStages;  // ring slots of Q_t, dO_t
            const uint32_t qph = (uint32_t)(t / C::kQStages) & 1u;
            const uint32_t oph = (uint32_t)(t / C::kOStages) & 1u;
            // -LSE*log2e and Delta of this warp's query columns (broadcast shared reads).
            const uint32_t nlse2_addr = smem_u32(smem + C::kOffNlse + qs * C::kVecBytes) + c0 * 4;
            const uint32_t dlt_addr = smem_u32(smem + C::kOffDelta + os * C::kVecBytes) + c0 * 4;
            const int q0 = it * kTileRows + c0;
            const bool masked = tile_masked(it, kt, p.Lq, p.Lk, CAUSAL);
            const int qlim = p.Lq - 1;  // last valid query
            // Phase 1: P^T = exp2(S^T * scale*log2e - LSE*log2e) on this warp's columns; kept
            // in registers, and the S^T columns are released at once.  (ok is false here only
            // after a failed wait of the dQ read-out.)
            ok = ok && wait_bounded(&bar_qf[qs], qph, abort_v, p.timeout_ns) &&
                 wait_bounded(&bar_sf, (uint32_t)t & 1u, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            float pv[kC];
            uint32_t pk_p[kC / 2];  // P^T, packed to 16 bits
            uint32_t keep_bits = 0xffffffffu;  // dropout: bit i keeps query column c0 + i
            static_assert(!DROP || kC <= 32, "one keep word per warp slice");
            if (ok) {
                tc_fence_after_sync();
                uint32_t r[kC];
                tmem_ld_cols<kC>(tmem + lane_off + C::kTmST + c0, r);
                tc_fence_before_sync();
                mbar_arrive(&bar_sr);
                const uint64_t scale2 = f2_make(p.scale_log2, p.scale_log2);
#pragma unroll
                for (int i = 0; i < kC; i += 4) {  // two columns per f32x2 instruction
                    const float4 l = lds_f32x4(nlse2_addr + i * 4);
                    float y0, y1, y2, y3;
                    f2_split(f2_fma(f2_make(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                    scale2, f2_make(l.x, l.y)),
                             y0, y1);
                    f2_split(f2_fma(f2_make(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])),
                                    scale2, f2_make(l.z, l.w)),
                             y2, y3);
                    pv[i + 0] = ex2_approx(y0);
                    pv[i + 1] = ex2_approx(y1);
                    pv[i + 2] = ex2_approx(y2);
                    pv[i + 3] = ex2_approx(y3);
                }
                if (masked) {
#pragma unroll
                    for (int i = 0; i < kC; ++i) {
                        const int qg = q0 + i;
                        if (qg > qlim || (CAUSAL && key > qg + (p.Lk - p.Lq))) pv[i] = 0.0f;
                    }
                }
                if constexpr (DROP) {
                    // One generator block holds keys 4m..4m+3 of one query: the four lanes of
                    // those keys each draw one query of a group of four and swap nibbles, so
                    // lane 4m+r ends up with key 4m+r's bits of all four queries.
                    const uint32_t r4 = (uint32_t)lane & 3u;
                    keep_bits = 0u;
#pragma unroll
                    for (int g = 0; g < kC; g += 4) {
                        uint32_t x = dropout_keep4((uint32_t)(key & ~3), (uint32_t)(q0 + g) + r4,
                                                   (uint32_t)bh, p.drop.seed_lo, p.drop.seed_hi,
                                                   p.drop.threshold)
                                     << (4u * r4);
                        x |= __shfl_xor_sync(0xffffffffu, x, 1);
                        x |= __shfl_xor_sync(0xffffffffu, x, 2);
                        // bit 4c + r4 of x: query q0 + g + c
                        const uint32_t b = ((x >> r4) & 1u) | ((x >> (r4 + 3u)) & 2u) |
                                           ((x >> (r4 + 6u)) & 4u) | ((x >> (r4 + 9u)) & 8u);
                        keep_bits |= b << g;
                    }
#pragma unroll
                    for (int i = 0; i < kC / 2; ++i)
                        pk_p[i] = pack2<BF16>((keep_bits >> (2 * i)) & 1u ? pv[2 * i] : 0.0f,
                                              (keep_bits >> (2 * i + 1)) & 1u ? pv[2 * i + 1] : 0.0f);
                } else {
#pragma unroll
                    for (int i = 0; i < kC / 2; ++i) pk_p[i] = pack2<BF16>(pv[2 * i], pv[2 * i + 1]);
                }
                // Phase 2: dS^T = P^T o (dP^T - Delta).
                ok = wait_bounded(&bar_of[os], oph, abort_v, p.timeout_ns) &&
                     wait_bounded(&bar_df, (uint32_t)t & 1u, abort_v, p.timeout_ns);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (ok) {
                tc_fence_after_sync();
                constexpr int kLd = kC >= 64 ? 32 : 16;  // dP^T columns per load (registers)
#pragma unroll
                for (int h = 0; h < kC / kLd; ++h) {
                    uint32_t r[kLd];
                    tmem_ld<kLd>(tmem + lane_off + C::kTmDPT + c0 + h * kLd, r);
                    if constexpr (DROP) {  // dP^T o Z^T: dropped entries 0, kept ones / (1 - p)
#pragma unroll
                        for (int i = 0; i < kLd; ++i)
                            r[i] = __float_as_uint((keep_bits >> (h * kLd + i)) & 1u
                                                       ? __uint_as_float(r[i]) * p.drop.keep_scale
                                                       : 0.0f);
                    }
#pragma unroll
                    for (int i = 0; i < kLd; i += 4) {  // P o (dP - Delta), two per instruction
                        const float4 d = lds_f32x4(dlt_addr + (h * kLd + i) * 4);
                        float* q = pv + h * kLd + i;
                        f2_split(f2_mul(f2_make(q[0], q[1]),
                                        f2_sub(f2_make(__uint_as_float(r[i]),
                                                       __uint_as_float(r[i + 1])),
                                               f2_make(d.x, d.y))),
                                 q[0], q[1]);
                        f2_split(f2_mul(f2_make(q[2], q[3]),
                                        f2_sub(f2_make(__uint_as_float(r[i + 2]),
                                                       __uint_as_float(r[i + 3])),
                                               f2_make(d.z, d.w))),
                                 q[2], q[3]);
                    }
                }
            }
            // Every slice of the quadrant has read its dP^T columns before any is overwritten.
            // (All warps reach this barrier once per query tile on every path.)
            ok = bar_and(grp_bar, kGrpThreads, ok);
            if (!ok) break;
            {
                tmem_st<kC / 2>(tmem + lane_off + C::kTmDPT + part * (kC / 2), pk_p);
                uint32_t pk[kC / 2];
#pragma unroll
                for (int i = 0; i < kC / 2; ++i) pk[i] = pack2<BF16>(pv[2 * i], pv[2 * i + 1]);
                tmem_st<kC / 2>(tmem + lane_off + C::kTmDPT + 64 + part * (kC / 2), pk);
                if constexpr (DQA) {
                    // dS row `row` (a key), queries c0..c0+31: four 16-byte units of the
                    // MN-major tile (64-query chunks 16 KB apart, 128-byte rows per key, the
                    // unit index XORed with key % 8).
                    static_assert(kC == 32, "four 16-byte units per warp slice");
                    uint8_t* ds_row = smem + C::kOffDS + (t & 1) * C::kDSTile +
                                      (c0 >> 6) * kChunkBytes + (row >> 3) * 1024 + (row & 7) * 128;
                    const int u0 = (c0 & 63) >> 3;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4*>(ds_row + (((u0 + j) ^ (row & 7)) << 4)) =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    fence_proxy_async_smem();
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bar_ppd);
            if constexpr (DQA) {  // dQ_{t-1}: read out and reduce, then free its accumulator
                if (t > 0) {
                    ok = wait_warp(&bars.dqf[(t - 1) & 1], ((uint32_t)(t - 1) >> 1) & 1u, abort_v,
                                   p.timeout_ns);
                    ok = dq_reduce(t - 1, ok);
                    if (ok) {
                        tc_fence_before_sync();
                        mbar_arrive(&bars.dqe[(t - 1) & 1]);
                    }
                }
            }
        }
        if (ok) {
            ok = wait_bounded(&bar_done, 0, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
        }
        if constexpr (DQA) ok = dq_reduce(n_it - 1, ok);  // every warp of the quadrant
        if (!ok) {
            if (lane == 0) record_timeout(p.status, abort_v);
        } else {
            tc_fence_after_sync();
            // The warp's 32 key rows from key - lane, stored coalesced across the warp.
            const int key0 = key - lane;
            const size_t coff = (size_t)part * C::kOutCols * 2;
            tmem_rows_to_global_xpose<BF16, C::kOutCols>(
                tmem + lane_off + C::kTmDV + part * C::kOutCols,
                reinterpret_cast<uint8_t*>(p.dv) + row_offset(p.sdv, bh, p.H, key0) + coff,
                (size_t)p.sdv.l * 2u, p.Lk - key0, DROP ? p.drop.keep_scale : 1.0f, lane);
            tmem_rows_to_global_xpose<BF16, C::kOutCols>(
                tmem + lane_off + C::kTmDK + part * C::kOutCols,
                reinterpret_cast<uint8_t*>(p.dk) + row_offset(p.sdk, bh, p.H, key0) + coff,
                (size_t)p.sdk.l * 2u, p.Lk - key0, p.scale, lane);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Persistent CTAs (see the file header): for rows of few query tiles.
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(DkdvCfg<D, BF16, CAUSAL>::kThreads, 1)
    fa_bwd_dkdv_kernel_persistent(const __grid_constant__ BwdParams p) {
    using C = DkdvCfg<D, BF16, CAUSAL>;
    // The kernel declares no static shared memory, so its dynamic shared memory starts at the
    // block's shared window, which is 1024-byte aligned; checked here (the 128-byte swizzle
    // needs it) before any barrier, TMEM or copy is touched.
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, (int)kDevBadShared);  // -> FA_ERR_CUDA
        return;
    }
    // Q_i (+ LSE_i) and dO_i (+ Delta_i) have their own rings and full/empty barriers: Q_i is
    // released by dK_i, issued first, so the load of a later Q tile (needed early, by S^T)
    // starts sooner.
    auto& bars = *reinterpret_cast<DkdvBarsT<D, BF16, CAUSAL>*>(smem + C::kOffBar);
    uint64_t* bar_kvf = bars.kvf;
    uint64_t* bar_kve = bars.kve;
    uint64_t* bar_qf = bars.qf;
    uint64_t* bar_qe = bars.qe;
    uint64_t* bar_of = bars.of;
    uint64_t* bar_oe = bars.oe;
    uint64_t& bar_sf = bars.sf;
    uint64_t& bar_df = bars.df;
    uint64_t& bar_sr = bars.sr;
    uint64_t& bar_ppd = bars.ppd;
    uint64_t& bar_done = bars.done;
    uint64_t& bar_fin = bars.fin;
    uint32_t& tmem_base_sh = bars.tmem_base;
    int& abort_flag = bars.abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::kKVSlots; ++s) {
            mbar_init(&bar_kvf[s], 1);
            mbar_init(&bar_kve[s], 1);
        }
        for (int s = 0; s < C::kQStages; ++s) {
            mbar_init(&bar_qf[s], 1);
            mbar_init(&bar_qe[s], 1);
        }
        for (int s = 0; s < C::kOStages; ++s) {
            mbar_init(&bar_of[s], 1);
            mbar_init(&bar_oe[s], 1);
        }
        mbar_init(&bar_sf, 1);
        mbar_init(&bar_df, 1);
        mbar_init(&bar_sr, C::kEwThreads);   // S^T read: its columns may be overwritten
        mbar_init(&bar_ppd, C::kEwThreads);  // P^T and dS^T written into the dP^T columns
        mbar_init(&bar_done, 1);             // every MMA of an item complete: dK, dV final
        mbar_init(&bar_fin, 1);
        queue_init(bars.queue, 1 + C::kEwWarps);  // read by the MMA and elementwise warps
        mbar_fence_init();
    }
    if (warp == C::kMmaWarp) tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    auto k_tile = [&](int slot) { return smem + C::kOffK + 2 * slot * C::kTileBytes; };
    auto v_tile = [&](int slot) { return smem + C::kOffK + (2 * slot + 1) * C::kTileBytes; };

    if (warp == C::kProducerWarp) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_do);
            bool ok = true;
            int issued_kv = 0, issued_q = 0, issued_o = 0;
            // Q_u and -LSE*log2e into Q slot u % kQStages (u counts query tiles over the CTA's
            // lifetime); query tile `qi` of head `bh`.
            auto load_q = [&](int u, const DkdvItem& it, int qi) -> bool {
                const int st = u % C::kQStages;
                if (u >= C::kQStages &&
                    !wait_bounded(&bar_qe[st], ((uint32_t)(u / C::kQStages) & 1u) ^ 1u, abort_v,
                                  p.timeout_ns))
                    return false;
                mbar_arrive_expect_tx(&bar_qf[st], C::kTileBytes + C::kVecBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(smem + C::kOffQ + st * C::kTileBytes + c * kChunkBytes, &p.tm_q,
                                &bar_qf[st], c * kChunkElems, qi * kTileRows, it.h, it.b);
                bulk_load(smem + C::kOffNlse + st * C::kVecBytes,
                          p.nlse2_pad + (size_t)it.bh * p.Lqpad + (size_t)qi * kTileRows,
                          C::kVecBytes,
                          &bar_qf[st]);
                issued_q = u + 1;
                return true;
            };
            auto load_do = [&](int u, const DkdvItem& it, int qi) -> bool {  // dO_u, Delta_u
                const int st = u % C::kOStages;
                if (u >= C::kOStages &&
                    !wait_bounded(&bar_oe[st], ((uint32_t)(u / C::kOStages) & 1u) ^ 1u, abort_v,
                                  p.timeout_ns))
                    return false;
                mbar_arrive_expect_tx(&bar_of[st], C::kTileBytes + C::kVecBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(smem + C::kOffDO + st * C::kTileBytes + c * kChunkBytes, &p.tm_do,
                                &bar_of[st], c * kChunkElems, qi * kTileRows, it.h, it.b);
                bulk_load(smem + C::kOffDelta + st * C::kVecBytes,
                          p.delta_pad + (size_t)it.bh * p.Lqpad + (size_t)qi * kTileRows,
                          C::kVecBytes,
                          &bar_of[st]);
                issued_o = u + 1;
                return true;
            };
            int u = 0;
            DkdvItem it;
            // Item ids are fetched one round ahead of the loads (fa_queue.cuh).
            int next_id = queue_push(bars.queue, 0, p.sched, p.n_ktiles * p.BH, false, abort_v,
                                     p.timeout_ns);
            for (int round = 0; ok; ++round) {
                const int id = next_id;
                if (id == -2) ok = false;
                if (id < 0) break;
                next_id = queue_push(bars.queue, round + 1, p.sched, p.n_ktiles * p.BH, false,
                                     abort_v, p.timeout_ns);
                dkdv_item<CAUSAL>(p, id, it);
                // K_j and V_j into K/V slot round % kKVSlots, once the item that used it last has
                // completed its S^T and dP^T contractions.
                const int kvs = round % C::kKVSlots;
                const int use = round / C::kKVSlots;
                if (use > 0 && !wait_bounded(&bar_kve[kvs], (uint32_t)(use - 1) & 1u, abort_v,
                                             p.timeout_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bar_kvf[kvs], 2 * C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_4d(k_tile(kvs) + c * kChunkBytes, &p.tm_k, &bar_kvf[kvs],
                                c * kChunkElems, it.kt * kTileRows, it.h, it.b);
                    tma_load_4d(v_tile(kvs) + c * kChunkBytes, &p.tm_v, &bar_kvf[kvs],
                                c * kChunkElems, it.kt * kTileRows, it.h, it.b);
                }
                issued_kv = round + 1;
                // Q runs one tile ahead of dO: Q_{t+1} only waits for dK_{t+1-kQStages}.
                ok = load_q(u, it, it.it0);
                for (int t = 0; ok && t < it.n_it; ++t) {
                    if (t + 1 < it.n_it) ok = load_q(u + t + 1, it, it.it0 + t + 1);
                    ok = ok && load_do(u + t, it, it.it0 + t);
                }
                u += it.n_it;
            }
            if (!ok) record_timeout(p.status, abort_v);
            // Drain: no copy may still be landing when the CTA exits.
            for (int n = issued_kv - 1; n >= 0 && n >= issued_kv - C::kKVSlots; --n)
                wait_bounded(&bar_kvf[n % C::kKVSlots], (uint32_t)(n / C::kKVSlots) & 1u, nullptr,
                             p.timeout_ns);
            for (int t = issued_q - 1; t >= 0 && t >= issued_q - C::kQStages; --t)
                wait_bounded(&bar_qf[t % C::kQStages], (uint32_t)(t / C::kQStages) & 1u, nullptr,
                             p.timeout_ns);
            for (int t = issued_o - 1; t >= 0 && t >= issued_o - C::kOStages; --t)
                wait_bounded(&bar_of[t % C::kOStages], (uint32_t)(t / C::kOStages) & 1u, nullptr,
                             p.timeout_ns);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------ MMA issuer ------------------------------
        // The whole warp walks the loop (warp-uniform values); one elected lane issues.  u counts
        // query tiles over the CTA's lifetime (ring slots and the per-tile barrier phases).
        auto q_base = [&](int uu) {
            return smem_u32(smem + C::kOffQ + (uu % C::kQStages) * C::kTileBytes);
        };
        auto do_base = [&](int uu) {
            return smem_u32(smem + C::kOffDO + (uu % C::kOStages) * C::kTileBytes);
        };
        auto wait_q = [&](int uu) {  // Q_uu landed
            const bool r = wait_warp(&bar_qf[uu % C::kQStages], (uint32_t)(uu / C::kQStages) & 1u,
                                     abort_v, p.timeout_ns);
            tc_fence_after_sync();
            return r;
        };
        auto wait_do = [&](int uu) {  // dO_uu landed
            const bool r = wait_warp(&bar_of[uu % C::kOStages], (uint32_t)(uu / C::kOStages) & 1u,
                                     abort_v, p.timeout_ns);
            tc_fence_after_sync();
            return r;
        };
        bool ok = true;
        int u = 0;
        DkdvItem it;
        for (int round = 0; ok; ++round) {
            const int id = queue_pop_warp(bars.queue, round, abort_v, p.timeout_ns);
            if (id == -2) ok = false;
            if (id < 0) break;
            dkdv_item<CAUSAL>(p, id, it);
            const int kvs = round % C::kKVSlots;
            const int n = it.n_it;
            const uint64_t kdesc = sdesc_kmajor_sw128(smem_u32(k_tile(kvs)));
            const uint64_t vdesc = sdesc_kmajor_sw128(smem_u32(v_tile(kvs)));
            auto issue_st = [&](int uu) {  // S^T = K Q_uu^T
                const uint64_t qd = sdesc_kmajor_sw128(q_base(uu));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    mma_ss_w(tmem + C::kTmST, sdesc_advance(kdesc, off), sdesc_advance(qd, off),
                             C::kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit_w(&bar_sf);
            };
            auto issue_dpt = [&](int uu) {  // dP^T = V dO_uu^T
                const uint64_t dd = sdesc_kmajor_sw128(do_base(uu));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    mma_ss_w(tmem + C::kTmDPT, sdesc_advance(vdesc, off), sdesc_advance(dd, off),
                             C::kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit_w(&bar_df);
            };
            // K_j / V_j of this item landed; the previous item's last S^T has been read (its
            // columns are reused).  The dP^T columns were last read by the previous item's last
            // dK / dV, issued before this point.
            ok = wait_warp(&bar_kvf[kvs], (uint32_t)(round / C::kKVSlots) & 1u, abort_v,
                           p.timeout_ns);
            if (ok && u > 0) ok = wait_warp(&bar_sr, (uint32_t)(u - 1) & 1u, abort_v, p.timeout_ns);
            ok = ok && wait_q(u);
            if (!ok) break;
            issue_st(u);
            if (!wait_do(u)) {
                ok = false;
                break;
            }
            issue_dpt(u);
            if (n == 1) mma_commit_w(&bar_kve[kvs]);  // the item's only S^T and dP^T issued
            for (int t = 0; t < n && ok; ++t) {
                const int uu = u + t;
                const uint32_t par = (uint32_t)uu & 1u;
                if (t + 1 < n) {
                    // S^T of the next query tile as soon as this one's S^T has been read.
                    if (!wait_warp(&bar_sr, par, abort_v, p.timeout_ns) || !wait_q(uu + 1)) {
                        ok = false;
                        break;
                    }
                    issue_st(uu + 1);
                }
                // With three or more dO slots, dO_{t+1} has normally landed by now: wait for it
                // here so dK_t, dV_t and dP^T_{t+1} go out as one batch.  With two it may still
                // be in flight, and waiting here would hold up dK_t and dV_t (measured slower).
                constexpr bool kEarlyDo = C::kOStages >= 3;
                if ((kEarlyDo && t + 1 < n && !wait_do(uu + 1)) ||
                    !wait_warp(&bar_ppd, par, abort_v, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t acc0 = t > 0 ? 1u : 0u;
                const uint64_t dod = sdesc_mnmajor_sw128(do_base(uu), kChunkBytes);
                const uint64_t qmd = sdesc_mnmajor_sw128(q_base(uu), kChunkBytes);
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk)
                    mma_ts_w(tmem + C::kTmDK, tmem + C::kTmDPT + 64 + kk * 8,
                             sdesc_advance(qmd, kk * 2048), C::kIdescG, (acc0 || kk > 0) ? 1u : 0u);
                mma_commit_w(&bar_qe[uu % C::kQStages]);  // Q_t fully read
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk)
                    mma_ts_w(tmem + C::kTmDV, tmem + C::kTmDPT + kk * 8,
                             sdesc_advance(dod, kk * 2048), C::kIdescG, (acc0 || kk > 0) ? 1u : 0u);
                mma_commit_w(&bar_oe[uu % C::kOStages]);  // dO_t fully read
                if (t + 1 < n) {  // after dV_t, dK_t read the dP^T columns
                    if (!kEarlyDo && !wait_do(uu + 1)) {
                        ok = false;
                        break;
                    }
                    issue_dpt(uu + 1);
                    if (t + 2 == n) mma_commit_w(&bar_kve[kvs]);  // the item's last S^T, dP^T
                }
            }
            if (!ok) break;
            mma_commit_w(&bar_done);
            u += n;
        }
        if (!ok && lane == 0) record_timeout(p.status, abort_v);
        mma_commit_w(&bar_fin);
        wait_warp(&bar_fin, 0, nullptr, p.timeout_ns);
    } else {
        // ------------------------------ elementwise warps ------------------------------
        constexpr int kC = C::kCols;
        const int quad = warp & 3;              // TMEM lane quadrant (key rows)
        const int part = warp >> 2;             // which kC query columns
        const uint32_t grp_bar = 1 + quad;      // named barrier of the quadrant
        constexpr uint32_t kGrpThreads = 32 * C::kSplit;
        const int row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int c0 = part * kC;
        const uint64_t scale2 = f2_make(p.scale_log2, p.scale_log2);
        bool ok = true;
        int u = 0;                 // query tiles of earlier items
        uint32_t done_par = 0u;    // phase of the item's done barrier
        DkdvItem it;
        for (int round = 0; ok; ++round) {
            // The quadrant's warps agree on the outcome before any of them goes on: they meet
            // at named barriers below.
            const int id = queue_pop_warp(bars.queue, round, abort_v, p.timeout_ns);
            ok = bar_and(grp_bar, kGrpThreads, id != -2);
            if (!ok || id < 0) break;
            dkdv_item<CAUSAL>(p, id, it);
            const int key = it.kt * kTileRows + row;
            const int u_end = u + it.n_it;
            const int qi_off = it.it0 - u;  // query tile of ring index uu: uu + qi_off
            for (int uu = u; uu < u_end; ++uu) {
                const int qi = uu + qi_off;
                const int qs = uu % C::kQStages, os = uu % C::kOStages;  // ring slots of Q, dO
                const uint32_t qph = (uint32_t)(uu / C::kQStages) & 1u;
                const uint32_t oph = (uint32_t)(uu / C::kOStages) & 1u;
                // -LSE*log2e and Delta of this warp's query columns (broadcast shared reads).
                const uint32_t nlse2_addr =
                    smem_u32(smem + C::kOffNlse + qs * C::kVecBytes) + c0 * 4;
                const uint32_t dlt_addr = smem_u32(smem + C::kOffDelta + os * C::kVecBytes) + c0 * 4;
                const int q0 = qi * kTileRows + c0;
                const bool masked = tile_masked(qi, it.kt, p.Lq, p.Lk, CAUSAL);
                const int qlim = p.Lq - 1;  // last valid query
                // Phase 1: P^T = exp2(S^T * scale*log2e - LSE*log2e) on this warp's columns;
                // kept in registers, and the S^T columns are released at once.
                ok = wait_bounded(&bar_qf[qs], qph, abort_v, p.timeout_ns) &&
                     wait_bounded(&bar_sf, (uint32_t)uu & 1u, abort_v, p.timeout_ns);
                ok = __all_sync(0xffffffffu, ok);
                float pv[kC];
                uint32_t pk_p[kC / 2];  // P^T, packed to 16 bits
                if (ok) {
                    tc_fence_after_sync();
                    uint32_t r[kC];
                    tmem_ld_cols<kC>(tmem + lane_off + C::kTmST + c0, r);
                    tc_fence_before_sync();
                    mbar_arrive(&bar_sr);
#pragma unroll
                    for (int i = 0; i < kC; i += 4) {  // two columns per f32x2 instruction
                        const float4 l = lds_f32x4(nlse2_addr + i * 4);
                        float y0, y1, y2, y3;
                        f2_split(f2_fma(f2_make(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                        scale2, f2_make(l.x, l.y)),
                                 y0, y1);
                        f2_split(f2_fma(f2_make(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])),
                                        scale2, f2_make(l.z, l.w)),
                                 y2, y3);
                        pv[i + 0] = ex2_approx(y0);
                        pv[i + 1] = ex2_approx(y1);
                        pv[i + 2] = ex2_approx(y2);
                        pv[i + 3] = ex2_approx(y3);
                    }
                    if (masked) {
#pragma unroll
                        for (int i = 0; i < kC; ++i) {
                            const int qg = q0 + i;
                            if (qg > qlim || (CAUSAL && key > qg + (p.Lk - p.Lq))) pv[i] = 0.0f;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kC / 2; ++i) pk_p[i] = pack2<BF16>(pv[2 * i], pv[2 * i + 1]);
                    // Phase 2: dS^T = P^T o (dP^T - Delta).
                    ok = wait_bounded(&bar_of[os], oph, abort_v, p.timeout_ns) &&
                         wait_bounded(&bar_df, (uint32_t)uu & 1u, abort_v, p.timeout_ns);
                    ok = __all_sync(0xffffffffu, ok);
                }
                if (ok) {
                    tc_fence_after_sync();
                    constexpr int kLd = kC >= 64 ? 32 : 16;  // dP^T columns per load (registers)
#pragma unroll
                    for (int h = 0; h < kC / kLd; ++h) {
                        uint32_t r[kLd];
                        tmem_ld<kLd>(tmem + lane_off + C::kTmDPT + c0 + h * kLd, r);
#pragma unroll
                        for (int i = 0; i < kLd; i += 4) {  // P o (dP - Delta), two per instruction
                            const float4 d = lds_f32x4(dlt_addr + (h * kLd + i) * 4);
                            float* q = pv + h * kLd + i;
                            f2_split(f2_mul(f2_make(q[0], q[1]),
                                            f2_sub(f2_make(__uint_as_float(r[i]),
                                                           __uint_as_float(r[i + 1])),
                                                   f2_make(d.x, d.y))),
                                     q[0], q[1]);
                            f2_split(f2_mul(f2_make(q[2], q[3]),
                                            f2_sub(f2_make(__uint_as_float(r[i + 2]),
                                                           __uint_as_float(r[i + 3])),
                                                   f2_make(d.z, d.w))),
                                     q[2], q[3]);
                        }
                    }
                }
                // Every slice of the quadrant has read its dP^T columns before any is
                // overwritten.  (All warps reach this barrier once per query tile on every path.)
                ok = bar_and(grp_bar, kGrpThreads, ok);
                if (!ok) break;
                {
                    tmem_st<kC / 2>(tmem + lane_off + C::kTmDPT + part * (kC / 2), pk_p);
                    uint32_t pk[kC / 2];
#pragma unroll
                    for (int i = 0; i < kC / 2; ++i) pk[i] = pack2<BF16>(pv[2 * i], pv[2 * i + 1]);
                    tmem_st<kC / 2>(tmem + lane_off + C::kTmDPT + 64 + part * (kC / 2), pk);
                }
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(&bar_ppd);
            }
            if (!ok) break;
            ok = wait_bounded(&bar_done, done_par, abort_v, p.timeout_ns);
            done_par ^= 1u;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            // tcgen05.ld waits for its data: the read-out is complete before this warp publishes
            // P^T / dS^T of the next item, which is what lets dK / dV of that item start.
            // The warp's 32 key rows from key - lane, stored coalesced across the warp.
            const int key0 = key - lane;
            const size_t coff = (size_t)part * C::kOutCols * 2;
            tmem_rows_to_global_xpose<BF16, C::kOutCols>(
                tmem + lane_off + C::kTmDV + part * C::kOutCols,
                reinterpret_cast<uint8_t*>(p.dv) + row_offset(p.sdv, it.bh, p.H, key0) + coff,
                (size_t)p.sdv.l * 2u, p.Lk - key0, 1.0f, lane);
            tmem_rows_to_global_xpose<BF16, C::kOutCols>(
                tmem + lane_off + C::kTmDK + part * C::kOutCols,
                reinterpret_cast<uint8_t*>(p.dk) + row_offset(p.sdk, it.bh, p.H, key0) + coff,
                (size_t)p.sdk.l * 2u, p.Lk - key0, p.scale, lane);
            u = u_end;
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

template <int D, bool BF16, bool CAUSAL, bool DROP, bool DQA>
cudaError_t launch_t(const BwdParams& p, cudaStream_t s) {
    using C = DkdvCfg<D, BF16, CAUSAL, DQA>;
    constexpr int kSmem = dkdv_smem_bytes<D, BF16, CAUSAL, DQA>();
    static_assert(kSmem <= 232448, "dynamic shared memory over the 227 KB per-block limit");
    const int total = p.n_ktiles * p.BH;
    // The persistent kernel has neither a dropout nor a dQ-reduction variant.
    const int grid = (DROP || DQA) ? total : dkdv_grid(p.Lq, p.Lk, p.BH, CAUSAL, sm_count());
    auto kern = grid < total ? fa_bwd_dkdv_kernel_persistent<D, BF16, CAUSAL>
                             : fa_bwd_dkdv_kernel<D, BF16, CAUSAL, DROP, DQA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, (unsigned)grid, C::kThreads, kSmem, s, p);
}

template <int D, bool BF16>
cudaError_t launch_d(const BwdParams& p, bool causal, bool drop, cudaStream_t s) {
    if (drop)
        return causal ? launch_t<D, BF16, true, true, false>(p, s)
                      : launch_t<D, BF16, false, true, false>(p, s);
    return causal ? launch_t<D, BF16, true, false, false>(p, s)
                  : launch_t<D, BF16, false, false, false>(p, s);
}

}  // namespace

cudaError_t launch_bwd_dkdv(const BwdParams& p, int D, bool bf16, bool causal, bool drop,
                            cudaStream_t s) {
    if (D == 64)
        return bf16 ? launch_d<64, true>(p, causal, drop, s) : launch_d<64, false>(p, causal, drop, s);
    return bf16 ? launch_d<128, true>(p, causal, drop, s) : launch_d<128, false>(p, causal, drop, s);
}

cudaError_t launch_bwd_dkdv_dq_reduce(const BwdParams& p, bool bf16, bool causal, cudaStream_t s) {
    if (bf16)
        return causal ? launch_t<64, true, true, false, true>(p, s)
                      : launch_t<64, true, false, false, true>(p, s);
    return causal ? launch_t<64, false, true, false, true>(p, s)
                  : launch_t<64, false, false, false, true>(p, s);
}

}  // namespace fa
