// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, TMA descriptors, launches,
// and the per-device status word that bounded device waits report into.
#include <cudaTypedefs.h>

#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_sched.h"

namespace fa {
namespace {

__device__ int g_status_word;  // first device-side error since the last fa_get_device_status

std::atomic<uint64_t> g_timeout_ns{4000000000ull};
std::atomic<int> g_fwd_pair{0};  // fa_set_forward_pair
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

// Device address of the status word of the current device (looked up once per device).
int* status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(ptr);
    }
    return g_status_ptr[dev];
}

// Makes the current device's primary context current on the calling thread.  The driver's
// tensor-map encoder needs a current context, and a thread may have none yet: a framework's
// worker thread (torch's autograd engine, for one) that has made no runtime call that creates
// or binds a context.  cudaSetDevice on the device the thread already uses does exactly that
// and allocates nothing.
bool bind_context() {
    int dev = 0;
    return cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess;
}

// [B, H, L, D] 16-bit tensor with element strides `st` (D contiguous) viewed as 4-D
// {D, L, H, B}; box = 64 elements x 128 rows x 1 x 1, with the 128-byte swizzle the tcgen05
// descriptors expect.  Rows past L read as zeros.  The strides are positive multiples of 8
// elements (16 bytes), checked by the caller.
bool make_map(CUtensorMap* m, const void* ptr, int B, int H, int L, int D, const Strides& st,
              bool bf16, int box_rows = kTileRows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)st.l * 2, (cuuint64_t)st.h * 2, (cuuint64_t)st.b * 2};
    cuuint32_t box[4] = {(cuuint32_t)kChunkElems, (cuuint32_t)box_rows, 1, 1};
    cuuint32_t elem[4] = {1, 1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     4, const_cast<void*>(ptr), dims, strides, box, elem,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Per-thread trace arming (fa_trace_next_call) and the process-wide launch counter.
constexpr int kMaxTracePairs = 8;
thread_local int t_trace_pairs = 0;
thread_local cudaEvent_t t_trace_events[2 * kMaxTracePairs];
std::atomic<uint64_t> g_launches{0};

// Enqueues one kernel through `launch`, bracketed by the armed trace events (if any).
template <typename F>
cudaError_t traced_launch(int index, cudaStream_t s, F&& launch) {
    const bool traced = index < t_trace_pairs;
    if (traced && cudaEventRecord(t_trace_events[2 * index], s) != cudaSuccess)
        return cudaErrorInvalidValue;
    cudaError_t e = launch();
    if (e != cudaSuccess) return e;
    g_launches.fetch_add(1);
    if (traced && cudaEventRecord(t_trace_events[2 * index + 1], s) != cudaSuccess)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

// Consumes the trace arming at the end of a public call, whatever its outcome.
struct TraceDisarm {
    ~TraceDisarm() { t_trace_pairs = 0; }
};

// Heads per schedule group: the streamed per-head operands (two [L, D] 16-bit tensors) of a
// group should take at most kGroupBytes of L2, so that tiles of the same head that run at the
// same time reuse them from L2 instead of HBM.
constexpr size_t kGroupBytes = size_t(48) << 20;
int schedule_group(int BH, int L, int D) {
    const size_t per_head = (size_t)2 * (size_t)L * (size_t)D * 2u;
    size_t g = per_head ? kGroupBytes / per_head : (size_t)BH;
    if (g < 1) g = 1;
    if (g > (size_t)BH) g = (size_t)BH;
    return (int)g;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
Range range(const void* p, size_t bytes) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

struct Shape {
    int BH = 0, H = 0, Lq = 0, Lk = 0, D = 0, n_qtiles = 0, n_ktiles = 0, Lqpad = 0;
    size_t lse_bytes = 0;
    bool empty = true;
};

// Checks sizes and flags shared by both passes.  Does not touch the GPU.
fa_status check_shape(int B, int H, int Lq, int Lk, int D, float scale, int causal, int dtype,
                      Shape* sh) {
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || D <= 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    const long long bh = (long long)B * (long long)H;
    const long long qtiles = ((long long)Lq + kTileRows - 1) / kTileRows;
    const long long ktiles = ((long long)Lk + kTileRows - 1) / kTileRows;
    if (bh > 0x7fffffffLL || qtiles * bh > 0x7fffffffLL || ktiles * bh > 0x7fffffffLL)
        return FA_ERR_UNSUPPORTED;
    sh->BH = (int)bh;
    sh->H = H;
    sh->Lq = Lq;
    sh->Lk = Lk;
    sh->D = D;
    sh->n_qtiles = (int)qtiles;
    sh->n_ktiles = (int)ktiles;
    sh->Lqpad = (int)(qtiles * kTileRows);
    sh->lse_bytes = (size_t)bh * (size_t)Lq * 4u;
    sh->empty = (bh == 0 || Lq == 0);  // no output row
    return FA_OK;
}

// A caller's strides, checked for the TMA rules (positive multiples of 8 elements = 16 bytes,
// below 2^39 elements); a stride of 0 is accepted for a dimension of size 1 and replaced by 8.
bool take_strides(const fa_strides& in, int B, int H, Strides* out) {
    long long v[3] = {in.batch, in.head, in.row};
    const int size[3] = {B, H, 2};  // the row dimension always counts
    for (int i = 0; i < 3; ++i) {
        if (v[i] == 0 && size[i] == 1) v[i] = 8;
        if (v[i] <= 0 || (v[i] & 7) != 0 || v[i] >= (1LL << 39)) return false;
    }
    *out = {v[0], v[1], v[2]};
    return true;
}

// Bytes from the first to one past the last element of a strided [B, H, L, D] 16-bit operand.
Range extent(const void* p, const Strides& s, int B, int H, int L, int D) {
    const long long last = (long long)(B - 1) * s.b + (long long)(H - 1) * s.h +
                           (long long)(L - 1) * s.l + D;
    return range(p, (size_t)last * 2u);
}

// Two outputs of the same shape and strides whose extents overlap are still disjoint element by
// element when they are interleaved parts of one packed tensor: the H heads of a row lie
// together (head stride D), the two bases are at least H*D elements apart and the second's heads
// end before the first's next row, and rows of different batches do not interleave.
bool interleaved_disjoint(const void* a, const void* b, const Strides& s, int L, int H, int D) {
    const long long da = reinterpret_cast<intptr_t>(a), db = reinterpret_cast<intptr_t>(b);
    const long long delta = (da > db ? da - db : db - da) / 2;
    const long long span = (long long)H * D;
    return s.h == D && delta >= span && delta + span <= s.l && s.b >= (long long)L * s.l;
}

bool same_strides(const Strides& a, const Strides& b) {
    return a.b == b.b && a.h == b.h && a.l == b.l;
}

// Dropout parameters: p in [0, 1); an entry is dropped iff its Philox word is below
// floor(p * 2^32), and kept ones are scaled by 1 / (1 - p).  p = 0 gives threshold 0 (nothing
// dropped); the caller then runs the kernels without dropout.
bool make_dropout(double p, uint64_t seed, Dropout* d) {
    if (!(p >= 0.0 && p < 1.0)) return false;  // also rejects NaN
    d->threshold = (uint32_t)std::floor(p * 4294967296.0);
    d->seed_lo = (uint32_t)(seed & 0xffffffffu);
    d->seed_hi = (uint32_t)(seed >> 32);
    d->keep_scale = (float)(1.0 / (1.0 - p));
    return true;
}

// Whether the backward reduces dQ inside the dK/dV pass (non-deterministic: fp32 additions in
// arrival order) instead of running the separate dQ pass: only when the caller allows it, at
// D = 64 (TMEM holds the extra accumulators only there) and without dropout.
bool dq_reduce_path(int D, int deterministic, double dropout_p) {
    return deterministic == 0 && D == 64 && !(dropout_p > 0.0);
}

// Backward workspace: -LSE*log2(e) and Delta ([BH, Lqpad] fp32 each), then for dQ by reduction
// the fp32 accumulator [BH, Lqpad, D], then the persistent passes' work counters.
size_t bwd_sched_offset(const Shape& sh, int D, bool dq_reduce) {
    const size_t rows = (size_t)sh.BH * (size_t)sh.Lqpad;
    return 2u * rows * 4u + (dq_reduce ? rows * (size_t)D * 4u : 0u);
}
size_t bwd_workspace_need(const Shape& sh, int D, bool dq_reduce) {
    return bwd_sched_offset(sh, D, dq_reduce) + kSchedBytes;
}

}  // namespace

void trace_disarm() { t_trace_pairs = 0; }

int sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int bwd_check_args(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, const void* dq, const void* dk, const void* dv, int B, int H,
                   int L, int D, float scale, int causal, int dtype, size_t* ws_need) {
    Shape sh;
    *ws_need = 0;
    fa_status st = check_shape(B, H, L, L, D, scale, causal, dtype, &sh);
    if (st != FA_OK) return st;
    if (sh.empty) return FA_OK;
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    *ws_need = bwd_workspace_need(sh, D, false);
    return FA_OK;
}

cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t s);

namespace {
__global__ void fa_wait_selftest_kernel(int* status, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);  // nothing ever arrives on it
        mbar_fence_init();
    }
    __syncthreads();
    const bool ok = wait_bounded(&bar, 0, &abort_flag, timeout_ns);
    if (!ok && threadIdx.x == 0) record_timeout(status, &abort_flag);
}
}  // namespace

cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t s) {
    return launch_kernel(fa_wait_selftest_kernel, 1, 32, 0, s, status, timeout_ns);
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
        default: return "FA_ERR_UNKNOWN";
    }
}

fa_status fa_set_forward_pair(int mode) {
    if (mode != 0 && mode != 1) return FA_ERR_INVALID_ARG;
    g_fwd_pair.store(mode);
    return FA_OK;
}

fa_status fa_set_wait_timeout_ns(uint64_t timeout_ns) {
    g_timeout_ns.store(timeout_ns ? timeout_ns : kDefaultTimeoutNs);
    return FA_OK;
}

fa_status fa_trace_next_call(void* const* events, int n_pairs) {
    if (n_pairs < 0 || n_pairs > kMaxTracePairs || (n_pairs > 0 && !events))
        return FA_ERR_INVALID_ARG;
    for (int i = 0; i < 2 * n_pairs; ++i) {
        if (!events[i]) return FA_ERR_INVALID_ARG;
        t_trace_events[i] = static_cast<cudaEvent_t>(events[i]);
    }
    t_trace_pairs = n_pairs;
    return FA_OK;
}

uint64_t fa_launch_count(void) { return g_launches.load(); }

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                    const fa_strides* strides, int B, int H, int Lq, int Lk, int D, float scale,
                    int causal, double dropout_p, uint64_t seed, int dtype, void* stream) {
    TraceDisarm disarm;
    Shape sh;
    fa_status st = check_shape(B, H, Lq, Lk, D, scale, causal, dtype, &sh);
    if (st != FA_OK) return st;
    Dropout drop;
    if (!make_dropout(dropout_p, seed, &drop)) return FA_ERR_INVALID_ARG;
    if (sh.empty) return FA_OK;
    if (Lk == 0) return FA_ERR_UNSUPPORTED;  // queries but no key at all
    if (!q || !k || !v || !o || !lse || !strides) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID_ARG;
    Strides sq, sk, sv, so;
    if (!take_strides(strides[0], B, H, &sq) || !take_strides(strides[1], B, H, &sk) ||
        !take_strides(strides[2], B, H, &sv) || !take_strides(strides[3], B, H, &so))
        return FA_ERR_INVALID_ARG;
    const Range rq = extent(q, sq, B, H, Lq, D), rk = extent(k, sk, B, H, Lk, D),
                rv = extent(v, sv, B, H, Lk, D), ro = extent(o, so, B, H, Lq, D),
                rl = range(lse, sh.lse_bytes);
    for (Range out : {ro, rl})
        for (Range in : {rq, rk, rv})
            if (overlap(out, in)) return FA_ERR_INVALID_ARG;
    if (overlap(ro, rl)) return FA_ERR_INVALID_ARG;

    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    const bool bf16 = dtype == FA_BF16;
    if (!bind_context()) return FA_ERR_CUDA;
    if (!make_map(&p.tm_q, q, B, H, Lq, D, sq, bf16) || !make_map(&p.tm_k, k, B, H, Lk, D, sk, bf16) ||
        !make_map(&p.tm_v, v, B, H, Lk, D, sv, bf16))
        return FA_ERR_CUDA;
    p.o = o;
    p.so = so;
    p.lse = lse;
    p.Lq = Lq;
    p.Lk = Lk;
    p.H = H;
    p.BH = sh.BH;
    p.n_qtiles = sh.n_qtiles;
    p.n_ktiles = sh.n_ktiles;
    p.group = schedule_group(sh.BH, Lk, D);
    // The softmax takes the row maximum of the stored S, so it must work with a non-negative
    // multiplier: a negative scale is moved into the S contraction as an exact sign flip.  The
    // multiplier is at least the smallest normal float, so that a masked logit (-inf) stays
    // -inf; for scale = 0 every visible logit times it is below 2^-100 in magnitude and exp2
    // returns exactly 1, the uniform softmax that scale 0 defines.
    p.scale_log2 = std::fmax(std::fabs(scale) * 1.4426950408889634f, FLT_MIN);
    p.s_negate = scale < 0.0f ? kIdescNegateA : 0u;
    p.drop = drop;
    p.status = status_ptr();
    p.timeout_ns = g_timeout_ns.load();
    if (!p.status) return FA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool dr = dropout_p > 0.0;
    // The CTA-pair forward: D = 128 without dropout, when selected (fa_set_forward_pair).
    const bool pair = D == 128 && !dr && g_fwd_pair.load() == 1;
    if (pair && !make_map(&p.tm_k_half, k, B, H, Lk, D, sk, bf16, 64)) return FA_ERR_CUDA;
    cudaError_t e = traced_launch(0, s, [&] {
        return pair ? launch_fwd_pair(p, bf16, causal != 0, s)
                    : launch_fwd(p, D, bf16, causal != 0, dr, s);
    });
    if (e != cudaSuccess) return FA_ERR_CUDA;
    // Under the causal mask the first Lq - Lk query rows see no key when Lq > Lk.
    const int empty_rows = (causal && Lq > Lk) ? Lq - Lk : 0;
    if (empty_rows > 0)
        e = traced_launch(1, s, [&] { return launch_fwd_empty_rows(p, D, empty_rows, s); });
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int L, int D, float scale, int causal, int dtype, void* stream) {
    const fa_strides c = {(int64_t)H * L * D, (int64_t)L * D, (int64_t)D};
    const fa_strides all[4] = {c, c, c, c};
    return fa_fwd_ex(q, k, v, o, lse, all, B, H, L, L, D, scale, causal, 0.0, 0, dtype, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int L, int D) {
    return fa_bwd_workspace_bytes_ex(B, H, L, D, 1);
}

size_t fa_bwd_workspace_bytes_ex(int B, int H, int Lq, int D, int deterministic) {
    Shape sh;
    if ((deterministic != 0 && deterministic != 1) ||
        check_shape(B, H, Lq, Lq, D, 1.0f, 0, FA_BF16, &sh) != FA_OK || sh.empty)
        return 0;
    return bwd_workspace_need(sh, D, dq_reduce_path(D, deterministic, 0.0));
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, void* workspace,
                    size_t workspace_bytes, const fa_strides* strides, int B, int H, int Lq,
                    int Lk, int D, float scale, int causal, double dropout_p, uint64_t seed,
                    int deterministic, int dtype, void* stream) {
    TraceDisarm disarm;
    Shape sh;
    fa_status st = check_shape(B, H, Lq, Lk, D, scale, causal, dtype, &sh);
    if (st != FA_OK) return st;
    Dropout drop;
    if (!make_dropout(dropout_p, seed, &drop)) return FA_ERR_INVALID_ARG;
    if (deterministic != 0 && deterministic != 1) return FA_ERR_INVALID_ARG;
    if (sh.BH == 0 || (Lq == 0 && Lk == 0)) return FA_OK;  // nothing to compute
    if (Lq == 0 || Lk == 0) return FA_ERR_UNSUPPORTED;     // queries without keys, or keys
                                                           // without queries
    const bool dqr = dq_reduce_path(D, deterministic, dropout_p);
    const size_t ws_need = bwd_workspace_need(sh, D, dqr);
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace || !strides)
        return FA_ERR_INVALID_ARG;
    if (workspace_bytes < ws_need) return FA_ERR_INVALID_ARG;
    const void* all[] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
    for (const void* ptr : all)
        if (!aligned16(ptr)) return FA_ERR_INVALID_ARG;
    Strides s8[8];
    for (int i = 0; i < 8; ++i)
        if (!take_strides(strides[i], B, H, &s8[i])) return FA_ERR_INVALID_ARG;
    const Strides &sq = s8[0], &sk = s8[1], &sv = s8[2], &so = s8[3], &sdo = s8[4], &sdq = s8[5],
                  &sdk = s8[6], &sdv = s8[7];
    const Range ins[] = {extent(q, sq, B, H, Lq, D),    extent(k, sk, B, H, Lk, D),
                         extent(v, sv, B, H, Lk, D),    extent(o, so, B, H, Lq, D),
                         extent(dout, sdo, B, H, Lq, D), range(lse, sh.lse_bytes)};
    const void* out_ptr[3] = {dq, dk, dv};
    const Strides out_st[3] = {sdq, sdk, sdv};
    const int out_len[3] = {Lq, Lk, Lk};
    Range outs[4];
    for (int i = 0; i < 3; ++i) outs[i] = extent(out_ptr[i], out_st[i], B, H, out_len[i], D);
    outs[3] = range(workspace, ws_need);
    for (int a = 0; a < 4; ++a) {
        for (const Range& b : ins)
            if (overlap(outs[a], b)) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 4; ++b) {
            if (!overlap(outs[a], outs[b])) continue;
            // dQ, dK, dV may be the interleaved parts of one packed gradient tensor.
            const bool packed = a < 3 && b < 3 && Lq == Lk && same_strides(out_st[a], out_st[b]) &&
                                interleaved_disjoint(out_ptr[a], out_ptr[b], out_st[a], Lq, H, D);
            if (!packed) return FA_ERR_INVALID_ARG;
        }
    }

    const bool bf16 = dtype == FA_BF16;
    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    if (!bind_context()) return FA_ERR_CUDA;
    if (!make_map(&p.tm_q, q, B, H, Lq, D, sq, bf16) || !make_map(&p.tm_k, k, B, H, Lk, D, sk, bf16) ||
        !make_map(&p.tm_v, v, B, H, Lk, D, sv, bf16) ||
        !make_map(&p.tm_do, dout, B, H, Lq, D, sdo, bf16))
        return FA_ERR_CUDA;
    float* nlse2_pad = static_cast<float*>(workspace);
    float* delta_pad = nlse2_pad + (size_t)sh.BH * sh.Lqpad;
    p.dout = dout;
    p.sdo = sdo;
    p.nlse2_pad = nlse2_pad;
    p.delta_pad = delta_pad;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.sdq = sdq;
    p.sdk = sdk;
    p.sdv = sdv;
    p.Lq = Lq;
    p.Lk = Lk;
    p.Lqpad = sh.Lqpad;
    p.H = H;
    p.BH = sh.BH;
    p.n_qtiles = sh.n_qtiles;
    p.n_ktiles = sh.n_ktiles;
    p.group = schedule_group(sh.BH, Lq > Lk ? Lq : Lk, D);
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.drop = drop;
    p.dq_acc = dqr ? delta_pad + (size_t)sh.BH * sh.Lqpad : nullptr;
    p.sched = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) +
                                     bwd_sched_offset(sh, D, dqr));
    p.status = status_ptr();
    p.timeout_ns = g_timeout_ns.load();
    if (!p.status) return FA_ERR_CUDA;

    BwdPreParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.o = o;
    pp.dout = dout;
    pp.dq = dq;
    pp.so = so;
    pp.sdo = sdo;
    pp.sdq = sdq;
    pp.lse = lse;
    pp.nlse2_pad = nlse2_pad;
    pp.delta_pad = delta_pad;
    pp.dq_acc = p.dq_acc;
    pp.sched = p.sched;
    pp.Lq = Lq;
    pp.Lqpad = sh.Lqpad;
    pp.H = H;
    pp.BH = sh.BH;
    pp.D = D;
    // Under the causal mask query row i sees key j iff j <= i + Lk - Lq: rows below Lq - Lk
    // see none (their dQ is zero).
    // (With dQ by reduction the conversion writes every row, zeros included.)
    pp.first_seen_row = (causal && Lq > Lk && !dqr) ? Lq - Lk : 0;
    pp.bf16 = bf16 ? 1 : 0;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (traced_launch(0, s, [&] { return launch_bwd_pre(pp, s); }) != cudaSuccess)
        return FA_ERR_CUDA;
    const bool dr = dropout_p > 0.0;
    if (dqr) {
        if (traced_launch(1, s, [&] { return launch_bwd_dkdv_dq_reduce(p, bf16, causal != 0, s); }) !=
            cudaSuccess)
            return FA_ERR_CUDA;
        if (traced_launch(2, s, [&] { return launch_bwd_dq_convert(p, D, bf16, s); }) != cudaSuccess)
            return FA_ERR_CUDA;
        return FA_OK;
    }
    if (traced_launch(1, s, [&] { return launch_bwd_dkdv(p, D, bf16, causal != 0, dr, s); }) !=
        cudaSuccess)
        return FA_ERR_CUDA;
    if (traced_launch(2, s, [&] { return launch_bwd_dq(p, D, bf16, causal != 0, dr, s); }) !=
        cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace,
                 size_t workspace_bytes, int B, int H, int L, int D, float scale, int causal,
                 int dtype, void* stream) {
    const fa_strides c = {(int64_t)H * L * D, (int64_t)L * D, (int64_t)D};
    const fa_strides all[8] = {c, c, c, c, c, c, c, c};
    return fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, all, B, H, L,
                     L, D, scale, causal, 0.0, 0, 1, dtype, stream);
}

size_t fa_decode_workspace_bytes(int B, int H, int D, int max_pages) {
    if (B <= 0 || H <= 0 || (D != 64 && D != 128) || max_pages < 0) return 0;
    const int splits = decode_splits(B, H, max_pages);
    if (splits <= 1) return 0;
    return (size_t)B * H * splits * (size_t)(D + 1) * 4u;
}

fa_status fa_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* seq_lens, void* o,
                          float* lse, void* workspace, size_t workspace_bytes, int B, int H, int D,
                          int num_pages, int max_pages, float scale, int dtype, void* stream) {
    TraceDisarm disarm;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || D <= 0 || num_pages < 0 || max_pages < 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;  // grid dimensions
    if (B == 0 || H == 0) return FA_OK;
    if (!q || !o || !lse || !seq_lens || (num_pages > 0 && (!k_cache || !v_cache)) ||
        (max_pages > 0 && !block_tables))
        return FA_ERR_INVALID_ARG;
    const void* al16[] = {q, o, lse, k_cache, v_cache};
    for (const void* ptr : al16)
        if (ptr && !aligned16(ptr)) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u))
        return FA_ERR_INVALID_ARG;
    const int splits = decode_splits(B, H, max_pages);
    const size_t ws_need = splits > 1 ? (size_t)B * H * splits * (size_t)(D + 1) * 4u : 0;
    if (ws_need > 0 && (!workspace || workspace_bytes < ws_need || !aligned16(workspace)))
        return FA_ERR_INVALID_ARG;
    const size_t rows = (size_t)B * H;
    const size_t cache_bytes = (size_t)num_pages * H * kPageTokens * D * 2u;
    const Range ins[] = {range(q, rows * D * 2u), range(k_cache, cache_bytes),
                         range(v_cache, cache_bytes),
                         range(block_tables, (size_t)B * max_pages * 4u),
                         range(seq_lens, (size_t)B * 4u)};
    const Range outs[] = {range(o, rows * D * 2u), range(lse, rows * 4u),
                          range(workspace, ws_need)};
    for (int a = 0; a < 3; ++a) {
        for (const Range& in : ins)
            if (overlap(outs[a], in)) return FA_ERR_INVALID_ARG;
        for (int b2 = a + 1; b2 < 3; ++b2)
            if (overlap(outs[a], outs[b2])) return FA_ERR_INVALID_ARG;
    }
    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.o = o;
    p.lse = lse;
    p.part_o = static_cast<float*>(workspace);
    p.part_lse = ws_need ? static_cast<float*>(workspace) + rows * splits * D : nullptr;
    p.B = B;
    p.H = H;
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.splits = splits;
    p.pages_per_split = max_pages > 0 ? (max_pages + splits - 1) / splits : 1;
    p.scale_log2 = scale * 1.4426950408889634f;
    if (!bind_context()) return FA_ERR_CUDA;
    p.status = status_ptr();
    p.timeout_ns = g_timeout_ns.load();
    if (!p.status) return FA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = traced_launch(0, s, [&] { return launch_decode(p, D, dtype == FA_BF16, s); });
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_get_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    if (!status_ptr()) return FA_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    if (word == 0) return FA_OK;
    if (word == (int)kDevBadArg) return FA_ERR_INVALID_ARG;
    return word == (int)kDevTimeout ? FA_ERR_TIMEOUT : FA_ERR_CUDA;
}

fa_status fa_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
    int* sp = status_ptr();
    if (!sp) return FA_ERR_CUDA;
    if (launch_wait_selftest(sp, timeout_ns, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

}  // extern "C"
