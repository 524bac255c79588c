// mtp_draft_head_argmax_static_ws: the bf16 draft head with its scratch in a
// fixed device array owned by this library, for callers that cannot hand the
// library device memory.
//
// Who needs it: code that runs where allocating device memory is not an
// option, e.g. a serving engine's per-step execute hook or plugin interface
// that gives extensions no allocator and no workspace, or a decode loop with
// a fixed, pre-planned memory budget.  cudaMalloc there can synchronise the
// device or fail at an unpredictable point, and a framework allocator may not
// exist on that side of the interface, so the call must bring its own scratch.
//
// Scratch: `vh_static_scratch`, a file-scope __device__ array of
// kStaticScratchBytes (4 KiB) on every device that loads this library, held
// until the process exits.  It serves up to kStaticMaxRows (256) hidden rows
// per call.  Host code only ever sees a host-side stand-in under that name,
// so the device address is looked up with cudaGetSymbolAddress once per
// device (on that device's first call, with the device current) and passed
// to the kernel.  The cached address belongs to the context of that first
// call: after cudaDeviceReset the module is loaded again and the address may
// change, so this entry point does not support a device reset in the process.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "../../include/verifyhead.h"
#include "vh_kernels.h"
#include "vh_verify.h"

namespace {

constexpr int kStaticMaxRows = vh::kMaxDraftB;
constexpr size_t kStaticScratchBytes = 4096;
static_assert(vh::ws_total_bytes(kStaticMaxRows) <= kStaticScratchBytes, "static scratch too small");

static __device__ __align__(256) unsigned char vh_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).  Returns nullptr on failure.
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, vh_static_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" {

vh_status mtp_draft_head_argmax_static_ws(const void* hidden, const void* W_cand, const int32_t* cand_ids, int B,
                                          int H, int Vc, int32_t* ids, float* maxlogit, void* stream) {
    if (!hidden || !W_cand || !cand_ids || !ids || !maxlogit) return VH_ERR_NULL;
    if (B < 1 || H < 16 || H > vh::kMaxH || H % 16 != 0 || Vc < 1) return VH_ERR_SHAPE;
    if (B > kStaticMaxRows) return VH_ERR_WORKSPACE;  // more rows than the fixed scratch holds
    if (!aligned(hidden, 16) || !aligned(W_cand, 32) || !aligned(cand_ids, 4) || !aligned(ids, 4) ||
        !aligned(maxlogit, 4))
        return VH_ERR_ALIGN;
    int dev = -1, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess || major < 10) {
        cudaGetLastError();
        return VH_ERR_DEVICE;
    }
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return VH_ERR_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left; the keys and the
    // ticket must start at zero.
    const size_t used = vh::ws_total_bytes(B);
    if (cudaMemsetAsync(scratch, 0, used, s) != cudaSuccess) {
        cudaGetLastError();
        return VH_ERR_LAUNCH;
    }
    const vh::Workspace w = vh::ws_view(scratch);
    const int grp = vh::draft_launch_rows(H, B);  // the same launch groups and kernels as mtp_draft_head_argmax
    const uint16_t* x = static_cast<const uint16_t*>(hidden);
    for (int b0 = 0; b0 < B; b0 += grp) {
        const int nb = std::min(grp, B - b0);
        cudaError_t e = vh::launch_draft_group(x + (size_t)b0 * H, nb, H, static_cast<const uint16_t*>(W_cand),
                                               cand_ids, Vc, w, ids + b0, maxlogit + b0, vh::AcceptTail{}, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return VH_ERR_LAUNCH;
        }
    }
    return VH_OK;
}

}  // extern "C"
