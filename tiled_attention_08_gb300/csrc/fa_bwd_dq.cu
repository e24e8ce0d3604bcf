// fa_bwd_dq.cu -- attention backward, dQ: per (b*h, 128-query tile), one CTA each or persistent.
//
// The separate-pass form of the dQ accumulation: for each query tile i and every key
// tile j it can see (j <= i under the causal mask), P and dS are recomputed from the saved
// log-sum-exp ("FlashAttention data-flow optimisation: MI50 memory and bandwidth
// bottlenecks", section 2.2, third layer) and
//   S  = Q_i K_j^T,  dP = dO_i V_j^T
//   P  = exp2(S * scale*log2e - LSE_i*log2e),  dS = P o (dP - Delta_i)   (per row: scalars)
//   dQ_i += dS K_j
// dQ_i is scaled by the softmax scale and written once: no atomics, deterministic.
//
// GB300 layout.  dO_i is the A operand of dP for every key tile, so it is staged once into TMEM
// (16-bit, two values per column) and dP runs with A in TMEM.  Q_i stays in shared memory
// (loaded once by TMA) and S = Q K_j^T reads both operands from there: SS and TS contractions
// run at the same rate on this part, and the TMEM columns Q would take go to a dedicated dS
// region (staging Q into TMEM as well measured 1.3% slower at D = 64).  Shared memory
// otherwise holds the K_j / V_j ring.
//
// CTA roles: 4*kSplit elementwise warps (warp w: query rows 32*(w%4).. == TMEM lanes, key
// columns [kCols*(w/4), +kCols)), then one TMA producer warp (Q_i, the K_j / V_j ring) and
// one MMA-issuer warp that also owns TMEM.
// TMEM: S [0,128), dP [128,256), dQ [256,256+D), dO [256+D, +D/2), dS (64 columns).
//
// Pipeline.  The elementwise warps read S into registers and release its columns at once, so
// the MMA warp issues S for the next key tile right away.  dS has its own columns: dP_{j+1} is
// issued as soon as dP_j has been read, and the elementwise warps write dS_{j+1} once dQ_j has
// completed.  The P phase of key tile j+1 therefore runs while the tensor core does dQ_j and
// dP_{j+1}.
//
// Two schedules (dq_grid).  For rows of few key tiles (a mean of at most kPersistMaxKv per
// query tile) fa_bwd_dq_kernel_persistent runs one CTA per SM (a CTA fills an SM: all 512 TMEM
// columns and over 200 KB of shared memory), each taking the next query tile of a
// heaviest-first order from the pass's work counter whenever it is ready for one
// (fa_queue.cuh).  The fixed cost of a CTA (launch, barrier and TMEM set-up, the first copies'
// latency, the pipeline fill and the dQ read-out) is then paid once per SM instead of once per
// tile, and most of it overlaps the neighbouring tiles: the K_j / V_j ring runs on across
// tiles, Q of the next tile is loaded as soon as the S contractions of this one have
// completed, the elementwise warps stage the next dO right after reading this tile's last dP,
// and the next tile's first S and dP run while they read out dQ.  Its barrier phases count
// key-tile iterations (or tiles) over the CTA's lifetime.  For longer rows the fixed cost
// matters less than the per-tile speed of fa_bwd_dq_kernel, which runs one CTA per query tile.
// Measured: B8 H32 L4096 D128 causal (16.5 key tiles per query tile on average) 1.205 ms one
// CTA per tile, 1.109 persistent in fixed rounds, 1.047 persistent with the work counter;
// B1 H16 L16384 D64 causal (64.5) 0.688 one CTA per tile, 0.729 persistent with the counter.
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_queue.cuh"
#include "fa_sched.h"

namespace fa {
namespace {

template <int D, bool BF16, bool CAUSAL>
struct DqCfg {
    static constexpr int kChunks = D / kChunkElems;
    static constexpr int kTileBytes = kTileRows * D * 2;
    static constexpr int kStages = (D == 128) ? 3 : 6;  // K/V ring depth
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kSmemBytes = kOffV + kStages * kTileBytes + 1024;
    // Elementwise warps per TMEM lane quadrant: at D = 64 the tensor core spends half as long
    // per key tile, so the elementwise phase is split over twice as many warps.
    static constexpr int kSplit = (D == 64) ? 4 : 2;
    static constexpr int kEwWarps = 4 * kSplit;
    static constexpr int kEwThreads = kEwWarps * 32;
    static constexpr int kProducerWarp = kEwWarps;
    static constexpr int kMmaWarp = kEwWarps + 1;
    static constexpr int kThreads = (kEwWarps + 2) * 32;
    static constexpr int kCols = 128 / kSplit;   // key columns per elementwise warp
    static constexpr int kOutCols = D / kSplit;  // dQ columns per elementwise warp
    static constexpr int kStageCols = D / 2 / kSplit;  // packed dO columns each warp stages
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmS = 0, kTmDP = 128, kTmDQ = 256;
    // dS has its own 64 columns, so dP_{j+1} never waits for dQ_j to have read dS_j.
    static constexpr uint32_t kTmDO = 256 + D;
    static constexpr uint32_t kTmDS = kTmDO + D / 2;
    static_assert(kTmDS + 64 <= kTmemCols, "TMEM budget");
    static constexpr uint32_t kIdescS = idesc_f16(BF16, 128, 128, false, false);
    static constexpr uint32_t kIdescG = idesc_f16(BF16, 128, D, false, true);
};

// One CTA per (b*h, query tile), in tile_coords order (the hardware's block scheduler balances
// the causal tiles): for rows of many key tiles, where a CTA's fixed cost is a small share.
// DROP: dropout on P (p.drop): dS = P o (dP o Z - Delta) with Z the keep mask times 1/(1-p).
template <int D, bool BF16, bool CAUSAL, bool DROP>
__global__ void __launch_bounds__(DqCfg<D, BF16, CAUSAL>::kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using C = DqCfg<D, BF16, CAUSAL>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ uint64_t bar_dpr, bar_dqd;  // dP read / dQ_j done (dS columns reusable)
    __shared__ uint64_t bar_q;             // Q_i landed in shared memory
    __shared__ uint64_t bar_qt, bar_kvf[C::kStages], bar_kve[C::kStages], bar_sf, bar_df, bar_sr,
        bar_pd, bar_done, bar_fin;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Heads in L2-sized groups (their K/V are streamed by every query tile); inside a group
    // the heaviest query tiles first.
    int bh, rank;
    tile_coords(blockIdx.x, p.BH, p.n_qtiles, p.group, bh, rank);
    const int hb = bh / p.H, hh = bh - hb * p.H;  // batch and head of bh
    const int qt = p.n_qtiles - 1 - rank;
    const int n_kv = q_tile_kv(qt, p.Lq, p.Lk, CAUSAL);
    // No row of this query tile sees a key (causal with Lq > Lk): the preprocess kernel has
    // written its dQ rows (zeros), so the whole CTA leaves before setting anything up.
    if (n_kv == 0) return;
    volatile int* abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar_qt, C::kEwThreads);  // dO_i staged into TMEM
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bar_kvf[s], 1);
            mbar_init(&bar_kve[s], 1);
        }
        mbar_init(&bar_sf, 1);
        mbar_init(&bar_df, 1);
        mbar_init(&bar_sr, C::kEwThreads);  // S read: its columns may be overwritten
        mbar_init(&bar_pd, C::kEwThreads);  // dS written
        mbar_init(&bar_dpr, C::kEwThreads);  // dP read: its columns may be overwritten
        mbar_init(&bar_q, 1);
        mbar_init(&bar_dqd, 1);              // dQ_j done: the dS columns may be overwritten
        mbar_init(&bar_done, 1);
        mbar_init(&bar_fin, 1);
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
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_q);
            mbar_arrive_expect_tx(&bar_q, C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(smem + C::kOffQ + c * kChunkBytes, &p.tm_q, &bar_q, c * kChunkElems,
                            qt * kTileRows, hh, hb);
            bool ok = true;
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % C::kStages;
                const uint32_t ph = (uint32_t)(j / C::kStages) & 1u;
                if (j >= C::kStages && !wait_bounded(&bar_kve[st], ph ^ 1u, abort_v, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bar_kvf[st], 2 * C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_4d(smem + C::kOffK + st * C::kTileBytes + c * kChunkBytes, &p.tm_k,
                                &bar_kvf[st], c * kChunkElems, j * kTileRows, hh, hb);
                    tma_load_4d(smem + C::kOffV + st * C::kTileBytes + c * kChunkBytes, &p.tm_v,
                                &bar_kvf[st], c * kChunkElems, j * kTileRows, hh, hb);
                }
                issued = j + 1;
            }
            if (!ok) record_timeout(p.status, abort_v);
            // Drain: no copy may still be landing when the CTA exits.
            wait_bounded(&bar_q, 0, nullptr, p.timeout_ns);
            for (int j = issued - 1; j >= 0 && j >= issued - C::kStages; --j)
                wait_bounded(&bar_kvf[j % C::kStages], (uint32_t)(j / C::kStages) & 1u, nullptr,
                             p.timeout_ns);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------ MMA issuer ------------------------------
        // The whole warp walks the loop (warp-uniform values); one elected lane issues.
        auto k_base = [&](int j) {
            return smem_u32(smem + C::kOffK + (j % C::kStages) * C::kTileBytes);
        };
        auto v_base = [&](int j) {
            return smem_u32(smem + C::kOffV + (j % C::kStages) * C::kTileBytes);
        };
        auto wait_stage = [&](int j) {
            const bool r = wait_warp(&bar_kvf[j % C::kStages],
                                        (uint32_t)(j / C::kStages) & 1u, abort_v, p.timeout_ns);
            tc_fence_after_sync();
            return r;
        };
        auto issue_s = [&](int j) {  // S = Q K_j^T, both operands in shared memory
            const uint64_t kd = sdesc_kmajor_sw128(k_base(j));
            const uint64_t qd = sdesc_kmajor_sw128(smem_u32(smem + C::kOffQ));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                mma_ss_w(tmem + C::kTmS, sdesc_advance(qd, off), sdesc_advance(kd, off),
                         C::kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bar_sf);
        };
        auto issue_dp = [&](int j) {  // dP = dO V_j^T, dO from TMEM
            const uint64_t vd = sdesc_kmajor_sw128(v_base(j));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                mma_ts_w(tmem + C::kTmDP, tmem + C::kTmDO + kk * 8, sdesc_advance(vd, off),
                       C::kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bar_df);
        };
        bool ok = wait_warp(&bar_qt, 0, abort_v, p.timeout_ns) &&
                  wait_warp(&bar_q, 0, abort_v, p.timeout_ns);
        tc_fence_after_sync();
        if (ok && n_kv > 0) {
            ok = wait_stage(0);
            if (ok) {
                issue_s(0);
                issue_dp(0);
            }
        }
        for (int j = 0; j < n_kv && ok; ++j) {
            const uint32_t par = (uint32_t)j & 1u;
            if (j + 1 < n_kv) {
                // S of the next key tile as soon as this one's S has been read.
                if (!wait_stage(j + 1) || !wait_warp(&bar_sr, par, abort_v, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                issue_s(j + 1);
                // dP_{j+1} as soon as dP_j has been read (dS has its own columns).
                if (!wait_warp(&bar_dpr, par, abort_v, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                issue_dp(j + 1);
            }
            if (!wait_warp(&bar_pd, par, abort_v, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint64_t kmd = sdesc_mnmajor_sw128(k_base(j), kChunkBytes);
#pragma unroll
            for (int kk = 0; kk < kTileRows / 16; ++kk)
                mma_ts_w(tmem + C::kTmDQ, tmem + C::kTmDS + kk * 8, sdesc_advance(kmd, kk * 2048),
                       C::kIdescG, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit_w(&bar_kve[j % C::kStages]);  // K_j, V_j fully read
            mma_commit_w(&bar_dqd);                  // dS_j consumed
        }
        if (ok) mma_commit_w(&bar_done);
        if (!ok && lane == 0) record_timeout(p.status, abort_v);
        mma_commit_w(&bar_fin);
        wait_warp(&bar_fin, 0, nullptr, p.timeout_ns);
    } else {
        // ------------------------------ elementwise warps ------------------------------
        constexpr int kC = C::kCols;
        const int quad = warp & 3;              // TMEM lane quadrant (query rows)
        const int part = warp >> 2;             // which kC key columns
        const int row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int q_row = qt * kTileRows + row;  // < Lqpad always
        const int c0 = part * kC;
        // Stage this warp's slice (D/kSplit elements) of the dO row into TMEM as packed 16-bit
        // pairs; rows past L are zeros.
        {
            constexpr int kE = D / C::kSplit;       // elements per warp slice
            constexpr int kW = C::kStageCols;       // packed 32-bit columns per slice
            const bool valid = q_row < p.Lq;
            const uint4* src = reinterpret_cast<const uint4*>(
                reinterpret_cast<const uint8_t*>(p.dout) + row_offset(p.sdo, bh, p.H, q_row) +
                (size_t)part * kE * 2);
            uint32_t w[kW];
#pragma unroll
            for (int v = 0; v < kW / 4; ++v) {
                const uint4 x = valid ? src[v] : make_uint4(0u, 0u, 0u, 0u);
                w[4 * v + 0] = x.x;
                w[4 * v + 1] = x.y;
                w[4 * v + 2] = x.z;
                w[4 * v + 3] = x.w;
            }
            tmem_st<kW>(tmem + lane_off + C::kTmDO + part * kW, w);
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bar_qt);
        }
        const float nlse2 = p.nlse2_pad[(size_t)bh * p.Lqpad + q_row];  // -LSE * log2(e)
        const float dlt = p.delta_pad[(size_t)bh * p.Lqpad + q_row];
        const uint64_t dlt2 = f2_make(dlt, dlt);
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int key0 = j * kTileRows + c0;
            const bool masked = tile_masked(qt, j, p.Lq, p.Lk, CAUSAL);
            const int klim = CAUSAL ? min(p.Lk - 1, q_row + (p.Lk - p.Lq)) : (p.Lk - 1);
            const uint32_t par = (uint32_t)j & 1u;
            float pv[kC];
            ok = wait_bounded(&bar_sf, par, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after_sync();
                uint32_t r[kC];
                tmem_ld_cols<kC>(tmem + lane_off + C::kTmS + c0, r);
                tc_fence_before_sync();
                mbar_arrive(&bar_sr);
                const uint64_t scale2 = f2_make(p.scale_log2, p.scale_log2);
                const uint64_t shift2 = f2_make(nlse2, nlse2);
#pragma unroll
                for (int i = 0; i < kC; i += 2) {  // two columns per f32x2 instruction
                    float y0, y1;
                    f2_split(f2_fma(f2_make(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                    scale2, shift2),
                             y0, y1);
                    pv[i] = ex2_approx(y0);
                    pv[i + 1] = ex2_approx(y1);
                }
                if (masked) {
#pragma unroll
                    for (int i = 0; i < kC; ++i)
                        if (key0 + i > klim) pv[i] = 0.0f;
                }
                ok = wait_bounded(&bar_df, par, abort_v, p.timeout_ns);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (ok) {
                tc_fence_after_sync();
                constexpr int kLd = kC >= 64 ? 32 : 16;  // dP columns per load (registers)
#pragma unroll
                for (int h = 0; h < kC / kLd; ++h) {
                    uint32_t r[kLd];
                    tmem_ld<kLd>(tmem + lane_off + C::kTmDP + c0 + h * kLd, r);
                    if constexpr (DROP) {  // dP o Z: dropped entries 0, kept ones / (1 - p)
#pragma unroll
                        for (int g = 0; g < kLd; g += 4) {
                            const uint32_t keep = dropout_keep4(
                                (uint32_t)(key0 + h * kLd + g), (uint32_t)q_row, (uint32_t)bh,
                                p.drop.seed_lo, p.drop.seed_hi, p.drop.threshold);
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                r[g + c] = __float_as_uint(
                                    (keep >> c) & 1u ? __uint_as_float(r[g + c]) * p.drop.keep_scale
                                                     : 0.0f);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kLd; i += 2) {  // P o (dP - Delta), two per instruction
                        float* q = pv + h * kLd + i;
                        f2_split(f2_mul(f2_make(q[0], q[1]),
                                        f2_sub(f2_make(__uint_as_float(r[i]),
                                                       __uint_as_float(r[i + 1])),
                                               dlt2)),
                                 q[0], q[1]);
                    }
                }
                tc_fence_before_sync();
                mbar_arrive(&bar_dpr);  // this thread's dP columns are read
            }
            // dS has its own columns: wait only until dQ_{j-1} has read dS_{j-1}.
            if (!ok) break;
            if (j > 0) {
                ok = wait_bounded(&bar_dqd, par ^ 1u, abort_v, p.timeout_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after_sync();
            }
            {
                uint32_t pk[kC / 2];
#pragma unroll
                for (int i = 0; i < kC / 2; ++i) pk[i] = pack2<BF16>(pv[2 * i], pv[2 * i + 1]);
                tmem_st<kC / 2>(tmem + lane_off + C::kTmDS + part * (kC / 2), pk);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bar_pd);
        }
        if (ok) {
            ok = wait_bounded(&bar_done, 0, abort_v, p.timeout_ns);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (!ok) {
            if (lane == 0) record_timeout(p.status, abort_v);
        } else {
            tc_fence_after_sync();
            uint8_t* dst_row = reinterpret_cast<uint8_t*>(p.dq) +
                               row_offset(p.sdq, bh, p.H, q_row) + part * C::kOutCols * 2;
            tmem_row_to_global<BF16, C::kOutCols>(tmem + lane_off + C::kTmDQ + part * C::kOutCols,
                                                  dst_row, p.scale, q_row < p.Lq);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Persistent CTAs (see the file header): for rows of few key tiles.
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(DqCfg<D, BF16, CAUSAL>::kThreads, 1)
    fa_bwd_dq_kernel_persistent(const __grid_constant__ BwdParams p) {
    using C = DqCfg<D, BF16, CAUSAL>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    // Per key-tile iteration (phase = running iteration count over all tiles of this CTA):
    __shared__ uint64_t bar_sf, bar_df;     // S / dP complete
    __shared__ uint64_t bar_sr, bar_dpr;    // S / dP read: their columns may be overwritten
    __shared__ uint64_t bar_pd;             // dS written
    __shared__ uint64_t bar_dqd;            // dQ += dS K done: the dS columns may be overwritten
    __shared__ uint64_t bar_kvf[C::kStages], bar_kve[C::kStages];  // K/V ring full / empty
    // Per query tile (phase = tile count of this CTA):
    __shared__ uint64_t bar_q;    // Q_i landed in shared memory
    __shared__ uint64_t bar_qe;   // every S of the tile complete: the Q buffer may be refilled
    __shared__ uint64_t bar_qt;   // dO_i staged into TMEM
    __shared__ uint64_t bar_done; // every MMA of the tile complete: dQ_i final
    __shared__ uint64_t bar_dqr;  // dQ_i read out: the accumulator may be overwritten
    __shared__ uint64_t bar_fin;
    __shared__ WorkQueue queue;  // this CTA's query tiles, fetched from the pass's counter
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort_v = &abort_flag;
    // Work ids 0 .. total-1 follow tile_coords (heads in L2-sized groups, heaviest query tiles
    // first); every CTA takes the next id when it is ready for one (fa_queue.cuh).  (The
    // launcher uses this kernel only when every query tile sees at least one key.)
    const int total = p.n_qtiles * p.BH;
    struct Tile {
        int bh, b, h, qt, n_kv;
    };
    auto tile_from = [&](int id, Tile& t) {
        int rank;
        tile_coords(id, p.BH, p.n_qtiles, p.group, t.bh, rank);
        t.b = t.bh / p.H;
        t.h = t.bh - t.b * p.H;
        t.qt = p.n_qtiles - 1 - rank;
        t.n_kv = q_tile_kv(t.qt, p.Lq, p.Lk, CAUSAL);
    };

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bar_kvf[s], 1);
            mbar_init(&bar_kve[s], 1);
        }
        mbar_init(&bar_sf, 1);
        mbar_init(&bar_df, 1);
        mbar_init(&bar_sr, C::kEwThreads);
        mbar_init(&bar_dpr, C::kEwThreads);
        mbar_init(&bar_pd, C::kEwThreads);
        mbar_init(&bar_dqd, 1);
        mbar_init(&bar_q, 1);
        mbar_init(&bar_qe, 1);
        mbar_init(&bar_qt, C::kEwThreads);
        mbar_init(&bar_done, 1);
        mbar_init(&bar_dqr, C::kEwThreads);
        mbar_init(&bar_fin, 1);
        queue_init(queue, 1 + C::kEwWarps);  // read by the MMA warp and the elementwise warps
        mbar_fence_init();
    }
    if (warp == C::kMmaWarp) tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    if (warp == C::kProducerWarp) {
        // ------------------------------ TMA producer ------------------------------
        // Fetches the tile ids (one round ahead).  Per tile: Q_i (once the previous tile's S
        // contractions have completed), then its K_j / V_j into the ring, which runs on across
        // tiles, so the next tile's first key tiles are already in flight while this one
        // finishes.
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_q);
            bool ok = true;
            int gk = 0;       // K/V fills handed to the TMA unit
            int q_loads = 0;  // Q fills handed to the TMA unit
            Tile t;
            int next_id = queue_push(queue, 0, p.sched + 1, total, false, abort_v, p.timeout_ns);
            for (int round = 0; ok; ++round) {
                const int id = next_id;
                if (id == -2) ok = false;
                if (id < 0) break;
                next_id = queue_push(queue, round + 1, p.sched + 1, total, false, abort_v,
                                     p.timeout_ns);
                tile_from(id, t);
                if (q_loads > 0 &&
                    !wait_bounded(&bar_qe, (uint32_t)(q_loads - 1) & 1u, abort_v, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bar_q, C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(smem + C::kOffQ + c * kChunkBytes, &p.tm_q, &bar_q,
                                c * kChunkElems, t.qt * kTileRows, t.h, t.b);
                ++q_loads;
                for (int j = 0; j < t.n_kv; ++j) {
                    const int st = gk % C::kStages;
                    const uint32_t ph = (uint32_t)(gk / C::kStages) & 1u;
                    if (gk >= C::kStages &&
                        !wait_bounded(&bar_kve[st], ph ^ 1u, abort_v, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar_kvf[st], 2 * C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_4d(smem + C::kOffK + st * C::kTileBytes + c * kChunkBytes,
                                    &p.tm_k, &bar_kvf[st], c * kChunkElems, j * kTileRows, t.h,
                                    t.b);
                        tma_load_4d(smem + C::kOffV + st * C::kTileBytes + c * kChunkBytes,
                                    &p.tm_v, &bar_kvf[st], c * kChunkElems, j * kTileRows, t.h,
                                    t.b);
                    }
                    ++gk;
                }
            }
            if (!ok) record_timeout(p.status, abort_v);
            // Drain: no copy may still be landing when the CTA exits.
            if (q_loads > 0)
                wait_bounded(&bar_q, (uint32_t)(q_loads - 1) & 1u, nullptr, p.timeout_ns);
            for (int g = gk - 1; g >= 0 && g >= gk - C::kStages; --g)
                wait_bounded(&bar_kvf[g % C::kStages], (uint32_t)(g / C::kStages) & 1u, nullptr,
                             p.timeout_ns);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------ MMA issuer ------------------------------
        // The whole warp walks the loop (warp-uniform values); one elected lane issues.  g is
        // the running key-tile iteration over all of this CTA's tiles (ring slot and phase).
        auto k_base = [&](int g) {
            return smem_u32(smem + C::kOffK + (g % C::kStages) * C::kTileBytes);
        };
        auto v_base = [&](int g) {
            return smem_u32(smem + C::kOffV + (g % C::kStages) * C::kTileBytes);
        };
        auto wait_stage = [&](int g) {
            const bool r = wait_warp(&bar_kvf[g % C::kStages], (uint32_t)(g / C::kStages) & 1u,
                                     abort_v, p.timeout_ns);
            tc_fence_after_sync();
            return r;
        };
        auto issue_s = [&](int g) {  // S = Q K^T, both operands in shared memory
            const uint64_t kd = sdesc_kmajor_sw128(k_base(g));
            const uint64_t qd = sdesc_kmajor_sw128(smem_u32(smem + C::kOffQ));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                mma_ss_w(tmem + C::kTmS, sdesc_advance(qd, off), sdesc_advance(kd, off),
                         C::kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bar_sf);
        };
        auto issue_dp = [&](int g) {  // dP = dO V^T, dO from TMEM
            const uint64_t vd = sdesc_kmajor_sw128(v_base(g));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                mma_ts_w(tmem + C::kTmDP, tmem + C::kTmDO + kk * 8, sdesc_advance(vd, off),
                         C::kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bar_df);
        };
        bool ok = true;
        int g = 0;
        int tc = 0;
        Tile t;
        for (int round = 0; ok; ++round, ++tc) {
            const int id = queue_pop_warp(queue, round, abort_v, p.timeout_ns);
            if (id == -2) ok = false;
            if (id < 0) break;
            tile_from(id, t);
            const int n = t.n_kv;
            // Q_i landed and dO_i staged; the previous tile's last S and dP have been read (their
            // columns are reused); K_0 / V_0 of this tile landed.
            ok = wait_warp(&bar_q, (uint32_t)tc & 1u, abort_v, p.timeout_ns) &&
                 wait_warp(&bar_qt, (uint32_t)tc & 1u, abort_v, p.timeout_ns);
            if (ok && g > 0)
                ok = wait_warp(&bar_sr, (uint32_t)(g - 1) & 1u, abort_v, p.timeout_ns) &&
                     wait_warp(&bar_dpr, (uint32_t)(g - 1) & 1u, abort_v, p.timeout_ns);
            if (ok) ok = wait_stage(g);
            if (!ok) break;
            issue_s(g);
            if (n == 1) mma_commit_w(&bar_qe);  // the tile's only S: Q free once it completes
            issue_dp(g);
            for (int j = 0; j < n; ++j) {
                const int gg = g + j;
                const uint32_t par = (uint32_t)gg & 1u;
                if (j + 1 < n) {
                    // S of the next key tile as soon as this one's S has been read.
                    if (!wait_stage(gg + 1) || !wait_warp(&bar_sr, par, abort_v, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    issue_s(gg + 1);
                    if (j + 2 == n) mma_commit_w(&bar_qe);  // the tile's last S issued
                    // dP_{j+1} as soon as dP_j has been read (dS has its own columns).
                    if (!wait_warp(&bar_dpr, par, abort_v, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    issue_dp(gg + 1);
                }
                if (!wait_warp(&bar_pd, par, abort_v, p.timeout_ns) ||
                    (j == 0 && tc > 0 &&
                     !wait_warp(&bar_dqr, (uint32_t)(tc - 1) & 1u, abort_v, p.timeout_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t kmd = sdesc_mnmajor_sw128(k_base(gg), kChunkBytes);
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk)
                    mma_ts_w(tmem + C::kTmDQ, tmem + C::kTmDS + kk * 8,
                             sdesc_advance(kmd, kk * 2048), C::kIdescG,
                             (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit_w(&bar_kve[gg % C::kStages]);  // K_j, V_j fully read
                mma_commit_w(&bar_dqd);                   // dS_j consumed
            }
            if (!ok) break;
            mma_commit_w(&bar_done);
            g += n;
        }
        if (!ok && lane == 0) record_timeout(p.status, abort_v);
        mma_commit_w(&bar_fin);
        wait_warp(&bar_fin, 0, nullptr, p.timeout_ns);
    } else {
        // ------------------------------ elementwise warps ------------------------------
        constexpr int kC = C::kCols;
        const int quad = warp & 3;              // TMEM lane quadrant (query rows)
        const int part = warp >> 2;             // which kC key columns
        const int row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int c0 = part * kC;
        // Stage this warp's slice (D/kSplit elements) of tile t's dO row into TMEM as packed
        // 16-bit pairs (rows past L are zeros), and read the row's -LSE*log2(e) and Delta.
        auto stage_do = [&](const Tile& t, float& nl, float& dl) {
            constexpr int kE = D / C::kSplit;       // elements per warp slice
            constexpr int kW = C::kStageCols;       // packed 32-bit columns per slice
            const int q_row = t.qt * kTileRows + row;  // < Lqpad always
            const bool valid = q_row < p.Lq;
            const uint4* src = reinterpret_cast<const uint4*>(
                reinterpret_cast<const uint8_t*>(p.dout) + row_offset(p.sdo, t.bh, p.H, q_row) +
                (size_t)part * kE * 2);
            uint32_t w[kW];
#pragma unroll
            for (int v = 0; v < kW / 4; ++v) {
                const uint4 x = valid ? src[v] : make_uint4(0u, 0u, 0u, 0u);
                w[4 * v + 0] = x.x;
                w[4 * v + 1] = x.y;
                w[4 * v + 2] = x.z;
                w[4 * v + 3] = x.w;
            }
            nl = p.nlse2_pad[(size_t)t.bh * p.Lqpad + q_row];
            dl = p.delta_pad[(size_t)t.bh * p.Lqpad + q_row];
            tmem_st<kW>(tmem + lane_off + C::kTmDO + part * kW, w);
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&bar_qt);
        };
        Tile cur, nxt;
        float nlse2 = 0.0f, dlt = 0.0f;  // -LSE * log2(e) and Delta of this thread's row
        const int id0 = queue_pop_warp(queue, 0, abort_v, p.timeout_ns);
        bool ok = id0 != -2;
        const bool any = id0 >= 0;  // a CTA that starts late may find no tile left
        if (any) {
            tile_from(id0, cur);
            stage_do(cur, nlse2, dlt);
        }
        int g = 0;
        for (int round = 0, tc = 0; ok && any; ++round, ++tc) {
            const int idn = queue_pop_warp(queue, round + 1, abort_v, p.timeout_ns);
            if (idn == -2) {
                ok = false;
                break;
            }
            const bool has_next = idn >= 0;
            if (has_next) tile_from(idn, nxt);
            const int n = cur.n_kv;
            const int q_row = cur.qt * kTileRows + row;
            const int klim = CAUSAL ? min(p.Lk - 1, q_row + (p.Lk - p.Lq)) : (p.Lk - 1);
            const uint64_t dlt2 = f2_make(dlt, dlt);
            float nlse2_n = 0.0f, dlt_n = 0.0f;
            for (int j = 0; j < n; ++j) {
                const int gg = g + j;
                const int key0 = j * kTileRows + c0;
                const bool masked = tile_masked(cur.qt, j, p.Lq, p.Lk, CAUSAL);
                const uint32_t par = (uint32_t)gg & 1u;
                float pv[kC];
                ok = wait_bounded(&bar_sf, par, abort_v, p.timeout_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    tc_fence_after_sync();
                    uint32_t r[kC];
                    tmem_ld_cols<kC>(tmem + lane_off + C::kTmS + c0, r);
                    tc_fence_before_sync();
                    mbar_arrive(&bar_sr);
                    const uint64_t scale2 = f2_make(p.scale_log2, p.scale_log2);
                    const uint64_t shift2 = f2_make(nlse2, nlse2);
#pragma unroll
                    for (int i = 0; i < kC; i += 2) {  // two columns per f32x2 instruction
                        float y0, y1;
                        f2_split(f2_fma(f2_make(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                        scale2, shift2),
                                 y0, y1);
                        pv[i] = ex2_approx(y0);
                        pv[i + 1] = ex2_approx(y1);
                    }
                    if (masked) {
#pragma unroll
                        for (int i = 0; i < kC; ++i)
                            if (key0 + i > klim) pv[i] = 0.0f;
                    }
                    ok = wait_bounded(&bar_df, par, abort_v, p.timeout_ns);
                    ok = __all_sync(0xffffffffu, ok);
                }
                if (ok) {
                    tc_fence_after_sync();
                    constexpr int kLd = kC >= 64 ? 32 : 16;  // dP columns per load (registers)
#pragma unroll
                    for (int h = 0; h < kC / kLd; ++h) {
                        uint32_t r[kLd];
                        tmem_ld<kLd>(tmem + lane_off + C::kTmDP + c0 + h * kLd, r);
#pragma unroll
                        for (int i = 0; i < kLd; i += 2) {  // P o (dP - Delta), two at a time
                            float* q = pv + h * kLd + i;
                            f2_split(f2_mul(f2_make(q[0], q[1]),
                                            f2_sub(f2_make(__uint_as_float(r[i]),
                                                           __uint_as_float(r[i + 1])),
                                                   dlt2)),
                                     q[0], q[1]);
                        }
                    }
                    tc_fence_before_sync();
                    mbar_arrive(&bar_dpr);  // this thread's dP columns are read
                }
                if (!ok) break;
                // dS has its own columns: wait until the previous dQ contraction (of this tile
                // or the last one of the previous tile) has read them.
                if (gg > 0) {
                    ok = wait_bounded(&bar_dqd, par ^ 1u, abort_v, p.timeout_ns);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after_sync();
                }
                {
                    uint32_t pk[kC / 2];
#pragma unroll
                    for (int i = 0; i < kC / 2; ++i) pk[i] = pack2<BF16>(pv[2 * i], pv[2 * i + 1]);
                    tmem_st<kC / 2>(tmem + lane_off + C::kTmDS + part * (kC / 2), pk);
                }
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(&bar_pd);
                // The tile's last dP has completed (it was read above), so the next tile's dO
                // may take the dO columns now: the MMA warp can start that tile's dP while
                // this tile's dQ is read out.
                if (j == n - 1 && has_next) stage_do(nxt, nlse2_n, dlt_n);
            }
            if (ok) {
                ok = wait_bounded(&bar_done, (uint32_t)tc & 1u, abort_v, p.timeout_ns);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (!ok) break;
            tc_fence_after_sync();
            uint8_t* dst_row = reinterpret_cast<uint8_t*>(p.dq) +
                               row_offset(p.sdq, cur.bh, p.H, q_row) + part * C::kOutCols * 2;
            tmem_row_to_global<BF16, C::kOutCols>(tmem + lane_off + C::kTmDQ + part * C::kOutCols,
                                                  dst_row, p.scale, q_row < p.Lq);
            tc_fence_before_sync();
            mbar_arrive(&bar_dqr);  // the accumulator is read: the next tile may overwrite it
            g += n;
            if (!has_next) break;
            cur = nxt;
            nlse2 = nlse2_n;
            dlt = dlt_n;
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

template <int D, bool BF16, bool CAUSAL, bool DROP>
cudaError_t launch_t(const BwdParams& p, cudaStream_t s) {
    using C = DqCfg<D, BF16, CAUSAL>;
    const int total = p.n_qtiles * p.BH;
    const int grid = dq_grid(p.Lq, p.Lk, p.BH, CAUSAL, sm_count());
    // The persistent kernel needs every query tile to see a key; only the first tile can fail to.
    // It has no dropout variant.
    if (!DROP && grid < total && q_tile_kv(0, p.Lq, p.Lk, CAUSAL) > 0) {
        // Persistent: one CTA per SM (each fills an SM).
        auto kern = fa_bwd_dq_kernel_persistent<D, BF16, CAUSAL>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        return launch_kernel(kern, (unsigned)grid, C::kThreads, C::kSmemBytes, s, p);
    }
    auto kern = fa_bwd_dq_kernel<D, BF16, CAUSAL, DROP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, (unsigned)total, C::kThreads, C::kSmemBytes, s, p);
}

template <int D, bool BF16>
cudaError_t launch_d(const BwdParams& p, bool causal, bool drop, cudaStream_t s) {
    if (drop) return causal ? launch_t<D, BF16, true, true>(p, s) : launch_t<D, BF16, false, true>(p, s);
    return causal ? launch_t<D, BF16, true, false>(p, s) : launch_t<D, BF16, false, false>(p, s);
}

// dQ by reduction: dQ = scale * dq_acc rounded to 16 bits, for every row < Lq (rows that see
// no key hold zeros).  HBM-bound: 16-byte stores, two 16-byte loads per store.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const BwdParams p) {
    constexpr int kPieces = D / 8;  // 8 elements (16 output bytes) per piece
    const long long total = (long long)p.BH * p.Lq * kPieces;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(e % kPieces);
        const long long r_all = e / kPieces;
        const int bh = (int)(r_all / p.Lq), i = (int)(r_all - (long long)bh * p.Lq);
        const float4* src = reinterpret_cast<const float4*>(
            p.dq_acc + ((size_t)bh * p.Lqpad + i) * D + c * 8);
        const float4 a = src[0], b = src[1];
        const float m = p.scale;
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.dq) +
                                  row_offset(p.sdq, bh, p.H, i) + c * 16) =
            make_uint4(pack2<BF16>(a.x * m, a.y * m), pack2<BF16>(a.z * m, a.w * m),
                       pack2<BF16>(b.x * m, b.y * m), pack2<BF16>(b.z * m, b.w * m));
    }
}

}  // namespace

cudaError_t launch_bwd_dq_convert(const BwdParams& p, int D, bool bf16, cudaStream_t s) {
    const long long work = (long long)p.BH * p.Lq * (D / 8);
    const int sms = sm_count() > 0 ? sm_count() : 148;
    long long blocks = (work + 255) / 256;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    if (blocks < 1) blocks = 1;
    const dim3 g((unsigned)blocks), b(256);
    if (D == 64)
        return bf16 ? launch_kernel(fa_bwd_dq_convert_kernel<64, true>, g, b, 0, s, p)
                    : launch_kernel(fa_bwd_dq_convert_kernel<64, false>, g, b, 0, s, p);
    return bf16 ? launch_kernel(fa_bwd_dq_convert_kernel<128, true>, g, b, 0, s, p)
                : launch_kernel(fa_bwd_dq_convert_kernel<128, false>, g, b, 0, s, p);
}

cudaError_t launch_bwd_dq(const BwdParams& p, int D, bool bf16, bool causal, bool drop,
                          cudaStream_t s) {
    if (D == 64)
        return bf16 ? launch_d<64, true>(p, causal, drop, s) : launch_d<64, false>(p, causal, drop, s);
    return bf16 ? launch_d<128, true>(p, causal, drop, s) : launch_d<128, false>(p, causal, drop, s);
}

}  // namespace fa
