// fa_internal.h -- launch parameters shared between the C-ABI layer and the kernel units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Status codes a kernel records in the device status word (first error wins).
enum DeviceError : int {
    kDevOk = 0,
    kDevBadShared = 3,  // dynamic shared memory not 1024-byte aligned (kernel did nothing)
    kDevTimeout = 4,    // a bounded wait ran out
    kDevBadArg = 5,     // device-side argument out of range (a page index or sequence length)
};

// Tile geometry shared by every kernel: 128 query rows x 128 keys per tile; operands are
// staged in shared memory as 128-row x 64-element boxes with the 128-byte swizzle.
constexpr int kTileRows = 128;
constexpr int kChunkElems = 64;
constexpr int kChunkBytes = kTileRows * kChunkElems * 2;  // 16 KiB per box

// Tile schedule shared by the attention kernels.  Heads are taken in groups of `group`
// (chosen on the host so that a group's streamed operands fit in L2 with room to spare);
// inside a group, tiles go heaviest first across all of the group's heads.  Returns the head
// and the tile's rank by weight (0 = heaviest: the last query tile, or key tile 0, under the
// causal mask).
__host__ __device__ __forceinline__ void tile_coords(int tile_id, int BH, int n_tiles, int group,
                                                     int& bh, int& rank) {
    const int span = group * n_tiles;
    const int g = tile_id / span;
    const int r = tile_id - g * span;
    const int heads = (BH - g * group) < group ? (BH - g * group) : group;
    rank = r / heads;
    bh = g * group + (r - rank * heads);
}

// Element strides of a [B, H, L, D] view whose D elements are contiguous (a row): contiguous
// [B,H,L,D], [B,L,H,D] and the q/k/v parts of a packed [B,L,3,H,D] tensor are all of this form.
struct Strides {
    long long b, h, l;
};

// Byte offset of row `row` of head `bh` (= b*H + h) of a 16-bit tensor with strides `s`.
__host__ __device__ __forceinline__ size_t row_offset(const Strides& s, int bh, int H, int row) {
    const int b = bh / H, h = bh - b * H;
    return (size_t)((long long)b * s.b + (long long)h * s.h + (long long)row * s.l) * 2u;
}

// Dropout on P: entry (bh, i, j) is dropped iff word j % 4 of Philox-4x32-10 at counter
// (j / 4, i, bh, 0) under the key (seed_lo, seed_hi) is below `threshold` = floor(p * 2^32); kept
// entries count 1/(1-p) (`keep_scale`).  threshold = 0: no dropout.
struct Dropout {
    uint32_t threshold, seed_lo, seed_hi;
    float keep_scale;
};

struct FwdParams {
    CUtensorMap tm_q, tm_k, tm_v;  // 16-bit {D, L, H, B} (strided), box {64, 128, 1, 1}
    CUtensorMap tm_k_half;         // K with box {64, 64, 1, 1} (CTA-pair forward only)
    void* o;                       // [B, H, Lq, D] 16-bit, strides so
    Strides so;
    float* lse;                    // [B*H, Lq] natural-log LSE (contiguous)
    int Lq, Lk, H, BH;
    int n_qtiles, n_ktiles;  // ceil(Lq / 128), ceil(Lk / 128)
    int group;          // heads per schedule group (tile_coords)
    float scale_log2;   // |scale| * log2(e)
    uint32_t s_negate;  // kIdescNegateA when scale < 0 (S is computed as -Q K^T), else 0
    Dropout drop;
    int* status;        // device status word
    uint64_t timeout_ns;
};

struct BwdPreParams {
    const void* o;       // [B, H, Lq, D], strides so
    const void* dout;    // [B, H, Lq, D], strides sdo
    void* dq;            // [B, H, Lq, D], strides sdq: rows that see no key are zeroed here
    Strides so, sdo, sdq;
    const float* lse;    // [BH, Lq]
    float* nlse2_pad;    // [BH, Lqpad]: -LSE * log2(e), zero past Lq
    float* delta_pad;    // [BH, Lqpad]: rowsum(dO * O), zero past Lq
    float* dq_acc;       // [BH, Lqpad, D] fp32, zeroed here (dQ by reduction), or null
    int* sched;          // work counters of the persistent passes, zeroed here
    int Lq, Lqpad, H, BH, D;
    int first_seen_row;  // rows below this see no key (causal with Lq > Lk), else 0
    int bf16;
};

// Work counters of the persistent backward passes at the end of the backward workspace.
constexpr int kSchedCounters = 4;
constexpr size_t kSchedBytes = kSchedCounters * sizeof(int);

// Decode over a paged key/value cache: tokens per page.
constexpr int kPageTokens = 16;

struct DecodeParams {
    const void* q;             // [B, H, D] 16-bit: the new token's query rows
    const void* k_cache;       // [num_pages, H, kPageTokens, D] 16-bit
    const void* v_cache;       // [num_pages, H, kPageTokens, D] 16-bit
    const int* block_tables;   // [B, max_pages]: physical page of each sequence's page
    const int* seq_lens;       // [B]: cached tokens per sequence (the new one included)
    void* o;                   // [B, H, D] 16-bit
    float* lse;                // [B, H] natural log
    float* part_o;             // [B*H*splits, D] fp32 (splits > 1)
    float* part_lse;           // [B*H*splits] log2 domain (splits > 1)
    int B, H, num_pages, max_pages, splits, pages_per_split;
    float scale_log2;          // scale * log2(e), either sign
    int* status;
    uint64_t timeout_ns;
};

struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;  // 16-bit {D, L, H, B} (strided), box {64, 128, 1, 1}
    const void* dout;                     // rows staged into TMEM by the dQ pass
    Strides sdo;
    const float* nlse2_pad;               // [BH, Lqpad]: -LSE * log2(e)
    const float* delta_pad;               // [BH, Lqpad]
    void* dq;                             // [B, H, Lq, D]
    void* dk;                             // [B, H, Lk, D]
    void* dv;                             // [B, H, Lk, D]
    Strides sdq, sdk, sdv;
    int Lq, Lk, Lqpad, H, BH, n_qtiles, n_ktiles;
    int group;          // heads per schedule group (tile_coords)
    float scale;        // softmax scale (applied to dQ and dK)
    float scale_log2;   // scale * log2(e)
    Dropout drop;
    float* dq_acc;      // [BH, Lqpad, D] fp32: dQ by reduction in the dK/dV pass, or null
    int* sched;         // [kSchedCounters] work counters: [0] dK/dV pass, [1] dQ pass
    int* status;
    uint64_t timeout_ns;
};

// Host-side helpers of the C-ABI layer shared with the other entry-point units.
// Consumes the fa_trace_next_call arming of the calling thread (every public call ends so).
void trace_disarm();
// Number of SMs of the current device (looked up once per device index); 0 if unknown.
int sm_count();
// fa_bwd's checks of sizes, flags and null pointers (the workspace excepted), in fa_bwd's
// order; on FA_OK (an int fa_status) *ws_need is the workspace the shape needs (0: empty).
int bwd_check_args(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, const void* dq, const void* dk, const void* dv, int B, int H,
                   int L, int D, float scale, int causal, int dtype, size_t* ws_need);

// Enqueues kern<<<grid, block, smem, s>>>(args...) and returns the status of that launch alone.
// (cudaGetLastError after a <<<>>> launch would also report a stale error left on the calling
// thread by any earlier runtime call, for example by a framework's set-up of its own threads.)
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Launchers (one per kernel unit).  Return the launch error, if any.
cudaError_t launch_fwd(const FwdParams& p, int D, bool bf16, bool causal, bool drop,
                       cudaStream_t s);
// The forward at D = 128 on CTA pairs (fa_fwd_pair.cu); needs p.tm_k_half.
cudaError_t launch_fwd_pair(const FwdParams& p, bool bf16, bool causal, cudaStream_t s);
cudaError_t launch_fwd_empty_rows(const FwdParams& p, int D, int rows, cudaStream_t s);
cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t s);
cudaError_t launch_bwd_dkdv(const BwdParams& p, int D, bool bf16, bool causal, bool drop,
                            cudaStream_t s);
// The dK/dV pass that also reduces dQ = dS K into p.dq_acc (D = 64, no dropout), then the
// conversion of p.dq_acc (times the scale) into p.dq.
cudaError_t launch_bwd_dkdv_dq_reduce(const BwdParams& p, bool bf16, bool causal, cudaStream_t s);
cudaError_t launch_bwd_dq_convert(const BwdParams& p, int D, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dq(const BwdParams& p, int D, bool bf16, bool causal, bool drop,
                          cudaStream_t s);
cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, int D, bool bf16, cudaStream_t s);
// Splits of the page range per (sequence, head) for a decode step of this shape.
int decode_splits(int B, int H, int max_pages);

}  // namespace fa
