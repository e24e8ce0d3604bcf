/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa.so).
 *
 * Operation.  Per (b,h) head, with Q, K, V, O of shape [L, D]:
 *     S = scale * Q K^T   (S_ij = -inf for j > i when causal)
 *     P = softmax(S) row by row,  O = P V,  LSE_i = log(sum_j exp(S_ij))
 * computed the tiled, streaming way: Q in 128-row tiles kept on chip, K/V streamed in 128-key
 * tiles, a running row max and row sum with the partial output rescaled as tiles arrive, and
 * only O and the per-row log-sum-exp written ("FlashAttention data-flow optimisation: MI50
 * memory and bandwidth bottlenecks", section 2.2, first and second layers;
 * "FlashAttention principles and engineering practice", section 2.1 for the plain
 * definition attn = softmax(q k^T * scale) v).  The backward pass recomputes P from the saved
 * LSE instead of storing the L x L matrix (data-flow page, section 2.2, third layer).
 *
 * Conventions shared by every entry point:
 *  - Tensors are DEVICE pointers to row-major [B, H, L, D] arrays (LSE: [B, H, L] fp32), each
 *    16-byte aligned: contiguous for fa_fwd / fa_bwd, strided (fa_strides) for fa_fwd_ex /
 *    fa_bwd_ex.  q, k, v, o, dO, dq, dk, dv all have the dtype `dtype`.
 *  - Supported: D in {64, 128}; B, H, L >= 0 (an empty problem returns FA_OK and launches
 *    nothing); causal in {0, 1} (query i sees key j iff j <= i); scale finite, of either sign
 *    or zero ("FlashAttention principles and engineering practice", section 2.1: the scale
 *    multiplies q k^T before the softmax), with scale * (q . k) inside the fp32 range.
 *  - The caller allocates and owns every buffer, including the backward workspace; the
 *    library never allocates or frees device memory in these calls.  The one exception is
 *    fa_bwd_noalloc's fixed scratch array, which is compiled into the library.
 *  - Calls are asynchronous: they validate, enqueue on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and return without synchronising.  Argument errors are reported
 *    before anything is enqueued and leave every output untouched.  A non-OK status from a
 *    launch leaves outputs undefined.  Kernels never spin without bound: a wait that exceeds
 *    its time limit records FA_ERR_TIMEOUT in a device status word, read by
 *    fa_get_device_status().
 *  - Outputs must not overlap inputs.  fa_bwd overwrites dq, dk, dv (it does not accumulate).
 *  - The library keeps no per-call state.  It caches the driver entry point used to build TMA
 *    descriptors and, per device index, the address of its status word, the address of
 *    fa_bwd_noalloc's scratch array and the SM count.  Those addresses belong to the device's
 *    primary context: after cudaDeviceReset (or anything else that destroys that context) the
 *    cached addresses are stale, so do not call into the library on that device again in the
 *    same process.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null/misaligned/overlapping pointer, bad size, bad flag */
    FA_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement (e.g. D) */
    FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed */
    FA_ERR_TIMEOUT = 4      /* a device-side bounded wait ran out (see fa_get_device_status) */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP16 = 1 } fa_dtype;

/*
 * Element strides of one [B, H, L, D] operand whose D elements are contiguous.  The layouts of
 * the flash_attn_func interface ("FlashAttention data-flow optimisation", section 4.1, step 3:
 * [B, L, H, D]) and of flash_attn_qkvpacked_func ("AIInfra notes 01: from TFLOPS to
 * FlashAttention", sections 4.2-4.3: [B, L, 3, H, D]) are both of this form:
 *     contiguous [B,H,L,D]:   {H*L*D, L*D,  D}
 *     [B,L,H,D]:              {L*H*D, D,    H*D}
 *     q/k/v of [B,L,3,H,D]:   {3*L*H*D, D,  3*H*D}, bases at +0, +H*D, +2*H*D elements.
 * Every stride is a positive multiple of 8 elements (16 bytes: the tensor-copy unit's rule) and
 * below 2^39; a stride of 0 is accepted for a dimension of size 1.
 */
typedef struct {
    int64_t batch, head, row;
} fa_strides;

/*
 * Forward.  Writes o [B,H,L,D] (dtype) and lse [B,H,L] (fp32, natural log).
 * Data-flow page, section 2.2 (tiling, streaming softmax, statistics kept for backward).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int L, int D, float scale, int causal, int dtype, void* stream);

/*
 * Forward with general layouts and lengths: q [B,H,Lq,D], k and v [B,H,Lk,D], o [B,H,Lq,D], each
 * addressed through its own strides (strides[0..3] = q, k, v, o); lse is contiguous [B,H,Lq].
 * Lq may differ from Lk.  Under the causal mask the queries are the last Lq positions of the
 * key sequence (a block of new tokens after Lk - Lq earlier ones): query i sees key j iff
 * j <= i + Lk - Lq.  A query row that sees no key (only when Lq > Lk) gets O = 0 and
 * LSE = -inf.  Lq = 0 returns FA_OK with nothing to do; Lk = 0 with Lq > 0 returns
 * FA_ERR_UNSUPPORTED.  Extents (first to last element) of the outputs must not overlap those of
 * the inputs or each other.  fa_fwd(..., L, ...) is fa_fwd_ex with Lq = Lk = L, contiguous
 * strides and no dropout.
 *
 * Dropout on P (flash_attn_func's dropout_p, data-flow page, section 4.1, step 3):
 * dropout_p in [0, 1) (NaN or outside: FA_ERR_INVALID_ARG); 0 runs the kernels without
 * dropout.  O = (P o Z) V with Z_ij = 0 for a dropped entry and 1 / (1 - dropout_p) for a kept
 * one; LSE stays that of P itself.  Entry (i, j) of head bh = b * H + h (query row i, key j) is
 * kept iff word j % 4 of the Philox-4x32-10 block (Salmon et al., "Parallel random numbers: as
 * easy as 1, 2, 3", SC 2011) at counter (j / 4, i, bh, 0) under key (seed & 0xffffffff,
 * seed >> 32) is at least floor(dropout_p * 2^32).  The pages fix no generator; this one is
 * counter-based, so the backward regenerates the mask from (dropout_p, seed) instead of storing
 * it.
 */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                    const fa_strides* strides, int B, int H, int Lq, int Lk, int D, float scale,
                    int causal, double dropout_p, uint64_t seed, int dtype, void* stream);

/*
 * Bytes of device workspace fa_bwd needs for this shape: two fp32 vectors per head padded to
 * a whole number of 128-row tiles (-LSE * log2(e) and Delta = rowsum(dO * O)), then 16 bytes
 * of work counters for the persistent passes.  Returns 0 for an empty problem or invalid sizes.
 * The pages have no such call: they keep the row maximum and the sum of exponentials for the
 * backward (data-flow page, section 2.2, third layer) without saying where the per-row
 * vectors the backward derives from them live.  Here the caller owns that memory, so the
 * library reports how much it needs.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int L, int D);

/*
 * Bytes of device workspace fa_bwd_ex needs for q of [B, H, Lq, D] and the given
 * `deterministic` flag (0 or 1; else 0 is returned): with deterministic = 0 at D = 64 the
 * backward reduces dQ into an fp32 accumulator [B*H, Lqpad, D] kept in the workspace after the
 * two per-row vectors (Lqpad = Lq rounded up to a multiple of 128; the work counters follow
 * it).  A workspace of this size
 * also serves the same shape with dropout (which always takes the deterministic path).
 * fa_bwd_workspace_bytes(B, H, L, D) = fa_bwd_workspace_bytes_ex(B, H, L, D, 1).
 * Pages: silent (as for fa_bwd_workspace_bytes).
 */
size_t fa_bwd_workspace_bytes_ex(int B, int H, int Lq, int D, int deterministic);

/*
 * Backward.  Given q, k, v, the forward's o and lse, and the output gradient dout, writes
 * dq, dk, dv [B,H,L,D] (dtype).  `workspace` is a device buffer of at least
 * fa_bwd_workspace_bytes(B,H,L,D) bytes, 16-byte aligned, owned by the caller; its contents
 * on entry do not matter.  Three kernels are enqueued on `stream`: the Delta/LSE preprocess,
 * the dK/dV pass (one CTA per key tile, or, when key tiles are seen by at most 32 query tiles
 * on average, one persistent CTA per SM) and the dQ pass (likewise per query tile, persistent
 * when query tiles see at most 32 key tiles on average); persistent CTAs take the next tile of
 * a heaviest-first order from a counter in the workspace whenever they are ready for one.  The
 * results are the same either way.
 * Data-flow page, section 2.2, third layer (recompute P from the saved statistics).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace,
                 size_t workspace_bytes, int B, int H, int L, int D, float scale, int causal,
                 int dtype, void* stream);

/*
 * Backward with general layouts and lengths (see fa_fwd_ex): strides[0..7] = q, k, v, o, dout,
 * dq, dk, dv; dq has the shape of q, dk and dv that of k.  The workspace is
 * fa_bwd_workspace_bytes(B, H, Lq, D).  Rows that see no key get dQ = 0.  Lq = Lk = 0 returns
 * FA_OK; only one of them 0 returns FA_ERR_UNSUPPORTED.  dq, dk and dv may be the three
 * interleaved parts of one packed [B,L,3,H,D] gradient (Lq = Lk, equal strides, the heads of a
 * row together, each part's heads ending before the next part's begin); otherwise no two
 * outputs' extents may overlap, and no output may overlap an input.  fa_bwd is fa_bwd_ex with
 * Lq = Lk = L, contiguous strides, no dropout and deterministic = 1.  dropout_p and seed must
 * be those of the forward that produced o and lse (the same mask is regenerated):
 * dV = (P o Z)^T dO and dS = P o ((dO V^T) o Z - Delta), Delta = rowsum(dO o O); the backward
 * under dropout always runs one CTA per tile.
 *
 * deterministic (0 or 1, else FA_ERR_INVALID_ARG): 1 computes dQ in its own pass, one CTA (or
 * persistent CTA) per query tile summing its key tiles in a fixed order, so every call gives
 * the same bits.  0 allows dQ to be computed inside the dK/dV pass ("dQ by atomics or a
 * separate pass", the method's two options): at D = 64 without dropout each (key tile, query
 * tile) pair adds its dS K into an fp32 accumulator in the workspace with vector reductions
 * (additions in arrival order: the result may differ in the last bits between calls) and a
 * third kernel converts it to dq; elsewhere 0 takes the deterministic path.  The workspace is
 * then fa_bwd_workspace_bytes_ex(B, H, Lq, D, 0) bytes.
 */
fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, void* workspace,
                    size_t workspace_bytes, const fa_strides* strides, int B, int H, int Lq,
                    int Lk, int D, float scale, int causal, double dropout_p, uint64_t seed,
                    int deterministic, int dtype, void* stream);

/* Size of the fixed device scratch array behind fa_bwd_noalloc: 16 MiB for the per-row
 * vectors and 256 bytes for the work counters. */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (((size_t)16 << 20) + 256)

/*
 * Backward for callers that cannot allocate device memory.  The pages describe no such entry
 * point; it has no counterpart in the method and exists only for callers that must not call
 * cudaMalloc themselves (for example a plugin whose host framework owns all device memory and
 * passes it only inputs and outputs, or a running latency-critical loop where an allocation
 * could synchronise the device at an unbounded cost).
 *
 * Same arguments, results and checks as fa_bwd, minus the workspace: the scratch fa_bwd would
 * take from `workspace` comes from a file-scope device array of FA_BWD_NOALLOC_SCRATCH_BYTES
 * compiled into the library, which every GPU that loads the library's code holds until the
 * process exits.  The limit: fa_bwd_workspace_bytes(B,H,L,D) = 8*B*H*ceil(L/128)*128 + 16
 * bytes must not exceed FA_BWD_NOALLOC_SCRATCH_BYTES (B*H*ceil(L/128)*128 <= 2^21 rows, e.g.
 * B*H = 256 heads at L = 8192); larger problems return FA_ERR_UNSUPPORTED before anything is
 * enqueued.  The call allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 *
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.  Every call on
 * a device shares the one array, so calls whose kernels overlap on the GPU (on different
 * streams, or from different threads) race on it and give undefined results: serialise them.
 * Nothing in the array needs clearing between calls; each call's first kernel overwrites
 * everything its later kernels read.  Checks run in fa_bwd's order (sizes and flags, then null
 * pointers), then the scratch limit, then fa_bwd's remaining checks; every outcome consumes a
 * trace arming made with fa_trace_next_call.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                         int H, int L, int D, float scale, int causal, int dtype, void* stream);

/* Tokens per page of the paged key/value cache of fa_decode_paged. */
#define FA_PAGE_TOKENS 16

/*
 * Bytes of device workspace fa_decode_paged needs for this shape: 0 when every (sequence, head)
 * pair is one CTA, else room for the per-split partial results (fp32).  0 for invalid sizes.
 */
size_t fa_decode_workspace_bytes(int B, int H, int D, int max_pages);

/*
 * One decode step over a paged key/value cache ("FlashAttention principles and engineering
 * practice", section 4.2: serving with PagedAttention, block_size 16, continuous batching).
 * Sequence b adds one token; its query rows q[b, h, :] attend to all seq_lens[b] tokens cached
 * for it (the new token's key and value already written to the cache by the caller):
 *     O[b,h] = softmax(scale * q[b,h] K_bh^T) V_bh,   LSE[b,h] = log sum_t exp(scale q.k_t),
 * with token t of sequence b in physical page block_tables[b*max_pages + t/16], slot t % 16.
 *   q, o:             [B, H, D] 16-bit (dtype), contiguous, 16-byte aligned;
 *   k_cache, v_cache: [num_pages, H, FA_PAGE_TOKENS, D] 16-bit, contiguous, 16-byte aligned
 *                     (the 16 tokens of one head in one page are contiguous);
 *   block_tables:     [B, max_pages] int32, device; entries past a sequence's pages are unread;
 *   seq_lens:         [B] int32, device, 0 <= seq_lens[b] <= 16 * max_pages;
 *   lse:              [B, H] fp32; workspace: fa_decode_workspace_bytes(B, H, D, max_pages).
 * A sequence with no cached token gets O = 0 and LSE = -inf.  Host-side argument errors return
 * before anything is enqueued; a page index outside [0, num_pages) or a length outside its range
 * (device data, checked by the kernel before any copy) is skipped and reported by
 * fa_get_device_status() as FA_ERR_INVALID_ARG, with the outputs of that call undefined.
 */
fa_status fa_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* seq_lens, void* o,
                          float* lse, void* workspace, size_t workspace_bytes, int B, int H, int D,
                          int num_pages, int max_pages, float scale, int dtype, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status word.  Returns
 * FA_OK, FA_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last call,
 * FA_ERR_INVALID_ARG if a decode kernel found a page index or sequence length out of range, or
 * FA_ERR_CUDA if synchronisation itself failed or a kernel refused to run (its dynamic shared
 * memory was not 1024-byte aligned; it then wrote nothing).
 * The pages are silent on failure detection; this call is the library's own way of making a
 * stalled kernel visible without faulting the GPU (every device-side wait is bounded).
 */
fa_status fa_get_device_status(void* stream);

/*
 * Selects the forward kernel at D = 128 without dropout: mode 1 runs it on CTA pairs (one
 * tensor-core contraction of 256 query rows over two SMs, tcgen05 cta_group::2, each CTA
 * loading half of every K and V tile), mode 0 (the default) on single CTAs.  The two give the
 * same results up to the order of nothing: every row's arithmetic is the same, so O and LSE are
 * bit for bit equal.  Process-wide; other head sizes and dropout always use single CTAs.
 * FA_ERR_INVALID_ARG for other modes.  The pages have no counterpart (TFLOPS page, sections
 * 3.2-3.3 size tiles for one SM).
 */
fa_status fa_set_forward_pair(int mode);

/* Time limit of every device-side wait, in nanoseconds (default 4e9).  0 restores the
 * default.  Applies to launches made after the call; returns FA_OK. */
fa_status fa_set_wait_timeout_ns(uint64_t timeout_ns);

/*
 * Self-test of the bounded-wait machinery: enqueues one tiny kernel that waits on a barrier
 * nothing will ever complete, with the given limit.  The kernel gives up, records
 * FA_ERR_TIMEOUT in the status word and returns, so the following fa_get_device_status()
 * reports FA_ERR_TIMEOUT and the context stays usable.
 */
fa_status fa_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * Kernel timing trace (the CUDA-event measurement the TFLOP/s figures rest on, per kernel).
 * Arms the next forward or backward call made by this host thread: the i-th kernel that call
 * enqueues is bracketed by cudaEventRecord(events[2*i], stream) and
 * cudaEventRecord(events[2*i+1], stream).  `events` holds n_pairs pairs of cudaEvent_t created
 * by the caller (with timing enabled); kernels beyond n_pairs are not traced.  The next call
 * consumes the arming.  A forward enqueues 1 kernel (2 under the causal mask with Lq > Lk: the
 * second writes the rows that see no key), a backward 3 (preprocess, dK/dV, dQ).
 */
fa_status fa_trace_next_call(void* const* events, int n_pairs);

/* Number of kernels this library has enqueued in this process so far. */
uint64_t fa_launch_count(void);

/* Static, human-readable name of a status code.  The pages have no counterpart (they
 * define no C interface); it names the fa_status values above. */
const char* fa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
