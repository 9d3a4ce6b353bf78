// qh_noalloc.cu -- qhead_fwd_noalloc: the forward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run the head: a decode loop inside a serving engine whose device memory
// is owned by a pre-sized arena, a plugin loaded into a host framework that
// forbids allocation after start-up, or latency-critical code that must not
// take the allocator's locks or trigger its synchronisation.  Such callers
// still own h and the outputs; this entry point supplies the forward's
// scratch from a fixed, statically allocated device array instead of a
// caller-provided workspace.
//
// The array is a file-scope __device__ object: every GPU that loads this
// library holds it until the process exits.  In host code its name is only a
// host-side stand-in, never a device address, so the address is looked up
// once per device with cudaGetSymbolAddress (with that device current) and
// cached by device ordinal.  The cached address belongs to the device's
// primary context as it was at that first call: after cudaDeviceReset, or
// under another context made current on the same device, it is stale.  All calls share the one array: nothing in it has to start at zero
// (each call writes every scratch byte it later reads), but two calls whose
// kernels overlap on the GPU -- e.g. on two streams -- race on it and must be
// serialised by the caller.
#include <mutex>
#include <string>

#include "../../include/qhead.h"
#include "qh_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)8 << 20;  // 8 MiB per device
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 1024;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up on the first
// call made with that device current).
int scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        qh::set_error(std::string("qhead_fwd_noalloc: cudaGetDevice: ") + cudaGetErrorString(e));
        return QHEAD_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        qh::set_error("qhead_fwd_noalloc: device ordinal out of range");
        return QHEAD_EINVAL;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p) {
            qh::set_error(std::string("qhead_fwd_noalloc: cudaGetSymbolAddress: ") +
                          cudaGetErrorString(e));
            return QHEAD_ECUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return QHEAD_OK;
}

}  // namespace

extern "C" int qhead_fwd_noalloc(const qhead_head* head, const void* h, int64_t M,
                                 const int32_t* targets, const uint8_t* mask, float* logp,
                                 float* lse, int32_t* argmax, void* stream) {
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != QHEAD_OK) return rc;
    // Invalid arguments make qhead_fwd_workspace return (size_t)-1; qhead_fwd
    // below then rejects them with the precise code and launches nothing.
    const size_t need = qhead_fwd_workspace(head, M);
    if (need != (size_t)-1 && need > kScratchBytes) {
        // The call ends here without reaching qhead_fwd: disarm the thread's
        // one-shot hooks as a forward call would, so that they do not fire
        // on its next call instead.
        qhead_time_next_head_kernel(nullptr, nullptr);
        qhead_test_stall_next_call(0);
        qh::set_error("qhead_fwd_noalloc: " + std::to_string(M) + " rows need " +
                      std::to_string(need) + " bytes of scratch, more than the fixed " +
                      std::to_string(kScratchBytes) +
                      " bytes; use qhead_fwd with a caller-allocated workspace");
        return QHEAD_EINVAL;
    }
    return qhead_fwd(head, h, M, targets, mask, logp, lse, argmax, scratch, kScratchBytes, stream);
}
