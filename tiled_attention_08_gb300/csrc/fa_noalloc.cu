// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass for callers that cannot allocate.
//
// fa_bwd needs a device workspace from its caller (two fp32 vectors per head: LSE*log2(e) and
// Delta, padded to whole 128-row tiles).  Some callers have no way to provide one: a plugin
// whose host framework owns every byte of device memory and hands it only inputs and outputs,
// or a latency-critical loop that must not call cudaMalloc (an allocation can synchronise the
// device and its cost is unbounded) once it is running.  This entry point serves them by
// taking its scratch from a fixed array compiled into the library instead.
//
// The array is a file-scope __device__ variable, so its symbol in host code is only a host-side
// stand-in, not a device address.  The device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on the device; that
// first call should therefore come before any stream capture.  The address is then passed to
// the kernels exactly as a caller's workspace would be.  No cudaMalloc, cudaFree or allocating
// library routine is called here.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kScratchBytes = FA_BWD_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device, and it keeps the last call's contents.  Nothing in it has
// to start at zero: the backward's preprocess kernel writes every element the later two
// kernels read (including the zero padding past L) before they run.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (set-up on first use per device).
fa_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
        if (e != cudaSuccess || ptr == nullptr) return FA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

// Consumes a fa_trace_next_call arming on every way out, as fa_bwd itself does.
struct DisarmOnExit {
    ~DisarmOnExit() { fa::trace_disarm(); }
};

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const void* dout, const float* lse, void* dq, void* dk,
                                    void* dv, int B, int H, int L, int D, float scale, int causal,
                                    int dtype, void* stream) {
    DisarmOnExit disarm;
    // fa_bwd's own checks first (sizes, flags, null pointers), so a call that fa_bwd would
    // refuse gets fa_bwd's status whatever its size.
    size_t need = 0;
    const int chk = fa::bwd_check_args(q, k, v, o, dout, lse, dq, dk, dv, B, H, L, D, scale,
                                       causal, dtype, &need);
    if (chk != FA_OK) return static_cast<fa_status>(chk);
    if (need == 0) return FA_OK;                          // empty problem: nothing to do
    if (need > kScratchBytes) return FA_ERR_UNSUPPORTED;  // larger than the fixed scratch
    void* scratch = nullptr;
    const fa_status st = scratch_address(&scratch);
    if (st != FA_OK) return st;
    return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, kScratchBytes, B, H, L, D, scale,
                  causal, dtype, stream);
}
