// Allocation-free variant of the fused expert MLP (r9q_gate_up_swiglu_down).
//
// Some callers cannot allocate device memory at the point where they run the
// MLP: code that runs under a memory-pool or arena owner that hands out no
// scratch, plug-ins that only receive their input and output buffers, and
// code paths that must not call cudaMalloc (which synchronises the device and
// may fail under memory pressure).  The regular entry point needs a workspace
// for the intermediate h = silu(gate) * up whenever the caller does not want
// h itself; this variant keeps h in a fixed scratch array that is part of the
// library instead, so the caller passes only inputs and outputs.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "r9q.h"
#include "r9q_kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)1 << 20;   // 1 MiB: h [M][I] bf16, M * I <= 524288

// The scratch for h.  Every GPU that loads the library holds this array until
// the process exits.  Host code must not pass the symbol itself to a kernel (on
// the host it only names a stand-in): its device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
    std::once_flag once;
    void* ptr = nullptr;
    int status = R9Q_OK;
};
ScratchAddr g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (set up on the
// first call made with that device current).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return R9Q_ERR_DEVICE;
    ScratchAddr& s = g_scratch_addr[dev];
    std::call_once(s.once, [&s]() {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            (void)cudaGetLastError();   // leave no pending error behind for the caller's next CUDA call
            s.status = R9Q_ERR_LAUNCH;
            return;
        }
        s.ptr = p;
    });
    *out = s.ptr;
    return s.status;
}

}  // namespace

extern "C" int r9q_gate_up_swiglu_down_noalloc(const void* x_bf16, const uint8_t* w_gu, const float* s_gu,
                                               const uint8_t* w_dn, const float* s_dn, void* y_bf16, int64_t M,
                                               int64_t H, int64_t I, int64_t H_out, uint8_t* hq_out,
                                               float* hs_out, int flags, void* stream) {
    if (!x_bf16 || !w_gu || !s_gu || !w_dn || !s_dn || !y_bf16) return R9Q_ERR_NULL;
    if (flags & R9Q_MLP_UNFUSED) return R9Q_ERR_ARG;            // the separate-launch chain needs more scratch
    if (M < 1 || I < 1) return R9Q_ERR_DIM;
    if ((size_t)M * (size_t)I * 2 > kNoAllocScratchBytes) return R9Q_ERR_WORKSPACE;   // beyond the fixed scratch
    // The library's device check (an sm_103 GPU) comes before the scratch
    // lookup, so another GPU gets R9Q_ERR_DEVICE and no lookup is attempted.
    int* err_word = nullptr;
    int rc = r9q::device_error_word(&err_word);
    if (rc) return rc;
    void* h = nullptr;
    rc = scratch_address(&h);
    if (rc) return rc;
    // The existing fused path with h in the library's scratch: no workspace.
    return r9q_gate_up_swiglu_down(x_bf16, w_gu, s_gu, w_dn, s_dn, y_bf16, M, H, I, H_out, h, hq_out, hs_out, flags,
                                   nullptr, 0, stream);
}
