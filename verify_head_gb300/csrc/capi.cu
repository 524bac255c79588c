// C ABI of libverifyhead.so: host-side argument checks and kernel dispatch.
// Declarations and the contract of every entry point: include/verifyhead.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "../../include/verifyhead.h"
#include "vh_kernels.h"
#include "vh_verify.h"

namespace {

using vh::gemv_group;
using vh::kMaxDraftB;
using vh::kMaxH;
constexpr int kTcRows = 256;   // hidden rows per tensor-core verify launch
constexpr int kMmaRows = 16;   // hidden rows per warp-MMA launch (8 when H > 5120)
constexpr int kTcFp4Rows = 16;  // hidden rows per tensor-core 4-bit draft launch
constexpr int kMmaFp4Rows = 8;  // hidden rows per warp-level-MMA 4-bit launch
constexpr int kPackedRows = 16;  // hidden rows per pass over a tiled 4-bit head
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

vh_status check_device() {
    static std::atomic<int> ok_cache[64] = {};  // 1: device already checked
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return VH_ERR_DEVICE;
    }
    if (dev < 64 && ok_cache[dev].load(std::memory_order_relaxed)) return VH_OK;
    int major = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess || major < 10) {
        cudaGetLastError();
        return VH_ERR_DEVICE;
    }
    if (dev < 64) ok_cache[dev].store(1, std::memory_order_relaxed);
    return VH_OK;
}

vh::Workspace make_ws(void* ws, int /*rows*/) { return vh::ws_view(ws); }

// Shapes the tiled 4-bit kernel takes: H % 256 == 0 and the f16 hidden rows of
// one 16-row pass (H * 32 bytes) within its shared-memory limit (H <= 6144).
inline bool packed_shape_ok(int H) {
    return H >= 256 && H <= kMaxH && H % 256 == 0 && vh::nvfp4_packed_smem(kPackedRows, H) <= vh::nvfp4_packed_max_smem();
}

vh_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return VH_OK;
    cudaGetLastError();  // clear a non-sticky launch error
    return VH_ERR_LAUNCH;
}

}  // namespace

namespace vh {

// Warp-MMA step length.  For 2-16 rows against heads of 768 MiB or more each warp streams 1 KiB of every
// row per step: 4 rows on the 248,320 x 2048 head took 166.9-168.2 against 172.0-173.9 us with 512-byte
// steps.  Below that, and for one row at every size, 512-byte steps are as fast or faster (4 rows on 768
// MiB: 140.1 / 140.3 us; one row on the full head: 160.0 against 161.0 us per chained call).
static bool long_steps(int nb, long long head_bytes) {
    constexpr long long kLongStepBytes = 768ll << 20;
    return nb >= 2 && head_bytes >= kLongStepBytes;
}

int draft_group(int H) { return gemv_mma_supported(16, H) ? 16 : gemv_group(H); }

cudaError_t launch_draft_group(const uint16_t* x, int nb, int H, const uint16_t* W, const int32_t* cand, int n_rows,
                               Workspace ws, int32_t* ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s) {
    // 17-256 rows (H % 64 == 0): one pass of the tcgen05 contraction over the table.
    // 2-16 rows: the warp MMAs (0.85-0.87 of HBM on 65,536 x 2048 at 2-8 rows), where the GEMV slows with
    // every row it holds.  One row: the CUDA-core GEMV on tables under 384 MiB (it starts faster: 128 MiB 22.6 against
    // 26.3 us, 256 MiB 41.2 against 45.3 us per chained call), the warp MMAs from 384 MiB up (65.2 against
    // 65.7 us; 512 MiB 83.8 against 86.7 us; the 248,320 x 2048 head 150.6 against 161.0 us, 0.99 against
    // 0.93 of HBM)
    // One row of 256 or 512 elements: the warp MMAs at every table size, where a 512- or 1024-byte row
    // leaves the GEMV too few bytes in flight per warp (262,144 x 256: 28.6 against 55.3 us; 131,072 x
    // 512: 28.4 against 31.6 us; 1,024 x 256: 6.5 against 7.2 us per chained call).
    constexpr long long kOneRowMmaBytes = 384ll << 20;
    const long long bytes = (long long)n_rows * H * 2;
    if (nb > 16 && H % 64 == 0) return launch_draft_tc(x, nb, H, W, cand, n_rows, ws, ids, maxlogit, s);
    // At H = 512 a one-row draft takes 512-element steps: a row group is then one unit of work, never cut
    // between warps, so a row scores the same bits wherever it sits in the table, as on the GEMV; they are
    // also faster there (131,072 x 512: 28.4 against 28.7 us; 990,000 x 512: 164.6 against 170.0 us).
    if (gemv_mma_supported(nb, H) && (nb >= 2 || H <= 512 || bytes >= kOneRowMmaBytes))
        return launch_gemv_mma_bf16(x, nb, H, W, cand, n_rows, ws, ids, maxlogit, tail, s,
                                    long_steps(nb, bytes) || (nb == 1 && H == 512));
    return launch_gemv_bf16(x, nb, H, W, cand, n_rows, ws, ids, maxlogit, tail, s);
}

}  // namespace vh

extern "C" {

int vh_version(void) { return 10000; }

const char* vh_status_string(int status) {
    switch (status) {
        case VH_OK: return "ok";
        case VH_ERR_NULL: return "a required pointer is NULL";
        case VH_ERR_SHAPE: return "a size is out of range or not a required multiple";
        case VH_ERR_ALIGN: return "a pointer is not aligned as required";
        case VH_ERR_WORKSPACE: return "workspace smaller than vh_workspace_bytes(rows)";
        case VH_ERR_LAUNCH: return "CUDA launch error";
        case VH_ERR_DEVICE: return "no usable CUDA device (sm_100 family required)";
        default: return "unknown status";
    }
}

size_t vh_workspace_bytes(int rows) {
    if (rows < 1) return 0;
    return vh::ws_total_bytes(rows);
}

size_t vh_verify_nvfp4_workspace_bytes(int rows, int H) {
    if (rows < 1 || H < 1) return 0;
    // argmax workspace, then the f16 hidden rows and one float per row
    return vh::ws_total_bytes(rows) + vh::round16((size_t)rows * (size_t)H * 2) + vh::round16((size_t)rows * 4);
}

vh_status mtp_draft_head_argmax(const void* hidden, const void* W_cand, const int32_t* cand_ids, int B, int H,
                                int Vc, int32_t* ids, float* maxlogit, void* ws, size_t ws_bytes, void* stream) {
    if (!hidden || !W_cand || !cand_ids || !ids || !maxlogit || !ws) return VH_ERR_NULL;
    if (B < 1 || B > kMaxDraftB || H < 16 || H > kMaxH || H % 16 != 0 || Vc < 1) return VH_ERR_SHAPE;
    if (!aligned(hidden, 16) || !aligned(W_cand, 32) || !aligned(cand_ids, 4) || !aligned(ids, 4) ||
        !aligned(maxlogit, 4) || !aligned(ws, 16))
        return VH_ERR_ALIGN;
    if (ws_bytes < vh_workspace_bytes(B)) return VH_ERR_WORKSPACE;
    vh_status st = check_device();
    if (st != VH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const vh::Workspace w = make_ws(ws, B);
    const uint16_t* x = static_cast<const uint16_t*>(hidden);
    const int grp = vh::draft_launch_rows(H, B);
    for (int b0 = 0; b0 < B; b0 += grp) {
        const int nb = std::min(grp, B - b0);
        cudaError_t e = vh::launch_draft_group(x + (size_t)b0 * H, nb, H, static_cast<const uint16_t*>(W_cand),
                                               cand_ids, Vc, w, ids + b0, maxlogit + b0, vh::AcceptTail{}, s);
        if (e != cudaSuccess) return launch_status(e);
    }
    return VH_OK;
}

vh_status mtp_draft_head_argmax_gather(const void* hidden, const void* W_full, const int32_t* row_ids, int B, int H,
                                       int n_ids, int V, int32_t* ids, float* maxlogit, void* ws, size_t ws_bytes,
                                       void* stream) {
    if (!hidden || !W_full || !row_ids || !ids || !maxlogit || !ws) return VH_ERR_NULL;
    if (B < 1 || B > kMaxDraftB || H < 16 || H > kMaxH || H % 16 != 0 || n_ids < 1 || V < 1) return VH_ERR_SHAPE;
    if (!aligned(hidden, 16) || !aligned(W_full, 32) || !aligned(row_ids, 4) || !aligned(ids, 4) ||
        !aligned(maxlogit, 4) || !aligned(ws, 16))
        return VH_ERR_ALIGN;
    if (ws_bytes < vh_workspace_bytes(B)) return VH_ERR_WORKSPACE;
    vh_status st = check_device();
    if (st != VH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const vh::Workspace w = make_ws(ws, B);
    const uint16_t* x = static_cast<const uint16_t*>(hidden);
    const int grp = gemv_group(H);
    for (int b0 = 0; b0 < B; b0 += grp) {
        const int nb = std::min(grp, B - b0);
        cudaError_t e = vh::launch_gemv_bf16(x + (size_t)b0 * H, nb, H, static_cast<const uint16_t*>(W_full), row_ids,
                                             n_ids, w, ids + b0, maxlogit + b0, vh::AcceptTail{}, s, V);
        if (e != cudaSuccess) return launch_status(e);
    }
    return VH_OK;
}

vh_status mtp_draft_head_argmax_nvfp4_path(const void* hidden, const uint8_t* Wq, const uint8_t* scales,
                                           float tensor_scale, const int32_t* cand_ids, int B, int H, int Vc,
                                           int32_t* ids, float* maxlogit, void* ws, size_t ws_bytes, void* stream,
                                           int path) {
    if (!hidden || !Wq || !scales || !cand_ids || !ids || !maxlogit || !ws) return VH_ERR_NULL;
    if (B < 1 || B > kMaxDraftB || H < 64 || H > kMaxH || H % 64 != 0 || Vc < 1) return VH_ERR_SHAPE;
    if (!(tensor_scale > 0.0f) || !(tensor_scale < 3.0e38f)) return VH_ERR_SHAPE;
    if (path != VH_PATH_AUTO && path != VH_PATH_CUDA_CORE && path != VH_PATH_TENSOR) return VH_ERR_SHAPE;
    const bool mma_ok = vh::nvfp4_mma_supported(kMmaFp4Rows, H);
    if (path == VH_PATH_TENSOR && !mma_ok && H % 512 != 0) return VH_ERR_SHAPE;
    if (!aligned(hidden, 16) || !aligned(Wq, 32) || !aligned(scales, 16) || !aligned(cand_ids, 4) ||
        !aligned(ids, 4) || !aligned(maxlogit, 4) || !aligned(ws, 16))
        return VH_ERR_ALIGN;
    if (ws_bytes < vh_workspace_bytes(B)) return VH_ERR_WORKSPACE;
    vh_status st = check_device();
    if (st != VH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const vh::Workspace w = make_ws(ws, B);
    const uint16_t* x = static_cast<const uint16_t*>(hidden);
    // one hidden row: CUDA-core streaming GEMV.  2..8 rows: warp-level MMAs
    // (H = 256 * 2^i <= 4096).  More rows: tcgen05 in groups of 16 when H is a
    // multiple of the 512-element raw stage (one pass over the head for 16
    // rows beats two 8-row MMA passes), else MMA groups of 8, else CUDA cores.
    // VH_PATH_TENSOR takes the same tensor-core kernels for any B;
    // VH_PATH_CUDA_CORE the GEMV for any B.
    const bool tensor = path == VH_PATH_TENSOR || (path == VH_PATH_AUTO && B > 1 && (mma_ok || H % 512 == 0));
    const bool tc = tensor && H % 512 == 0 && !(B <= kMmaFp4Rows && mma_ok);
    const bool mma = tensor && !tc && mma_ok;
    const int grp = mma ? kMmaFp4Rows : tc ? kTcFp4Rows : gemv_group(H);
    for (int b0 = 0; b0 < B; b0 += grp) {
        const int nb = std::min(grp, B - b0);
        const uint16_t* xb = x + (size_t)b0 * H;
        cudaError_t e =
            mma  ? vh::launch_nvfp4_mma(xb, nb, H, Wq, scales, tensor_scale, cand_ids, Vc, w, ids + b0, maxlogit + b0, s)
            : tc ? vh::launch_nvfp4_tc(xb, nb, H, Wq, scales, tensor_scale, cand_ids, Vc, w, ids + b0, maxlogit + b0, s)
                 : vh::launch_gemv_nvfp4(xb, nb, H, Wq, scales, tensor_scale, cand_ids, Vc, w, ids + b0, maxlogit + b0,
                                         s);
        if (e != cudaSuccess) return launch_status(e);
    }
    return VH_OK;
}

vh_status mtp_draft_head_argmax_nvfp4(const void* hidden, const uint8_t* Wq, const uint8_t* scales,
                                      float tensor_scale, const int32_t* cand_ids, int B, int H, int Vc,
                                      int32_t* ids, float* maxlogit, void* ws, size_t ws_bytes, void* stream) {
    return mtp_draft_head_argmax_nvfp4_path(hidden, Wq, scales, tensor_scale, cand_ids, B, H, Vc, ids, maxlogit, ws,
                                            ws_bytes, stream, VH_PATH_AUTO);
}

vh_status spec_verify_greedy_path(const void* hidden, const void* W_full, const int32_t* draft_ids, int B, int k,
                                  int H, int V, int32_t* accept_len, int32_t* next_ids, float* row_maxlogit,
                                  void* ws, size_t ws_bytes, void* stream, int path) {
    if (!hidden || !W_full || !draft_ids || !accept_len || !next_ids || !ws) return VH_ERR_NULL;
    if (B < 1 || k < 1 || k > 15 || H < 16 || H > kMaxH || H % 16 != 0 || V < 1) return VH_ERR_SHAPE;
    if ((long long)B * (k + 1) > 65536) return VH_ERR_SHAPE;
    if (path != VH_PATH_AUTO && path != VH_PATH_CUDA_CORE && path != VH_PATH_TENSOR && path != VH_PATH_WARP_MMA)
        return VH_ERR_SHAPE;
    if (path == VH_PATH_TENSOR && H % 64 != 0) return VH_ERR_SHAPE;
    if (path == VH_PATH_WARP_MMA && !vh::gemv_mma_supported(1, H)) return VH_ERR_SHAPE;
    if (!aligned(hidden, 16) || !aligned(W_full, 32) || !aligned(draft_ids, 4) || !aligned(accept_len, 4) ||
        !aligned(next_ids, 4) || !aligned(row_maxlogit, 4) || !aligned(ws, 16))
        return VH_ERR_ALIGN;
    const int R = B * (k + 1);
    if (ws_bytes < vh_workspace_bytes(R)) return VH_ERR_WORKSPACE;
    vh_status st = check_device();
    if (st != VH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const vh::Workspace w = make_ws(ws, R);
    const uint16_t* X = static_cast<const uint16_t*>(hidden);
    const uint16_t* W = static_cast<const uint16_t*>(W_full);

    // The one-CTA tensor kernel streams the head at the same rate for 2 rows as for 128, while the
    // CUDA-core GEMV slows with every row it holds (2 / 4 / 8 rows: 257 / 360 / 602 us against 177 us
    // on the 248,320 x 2048 head), so AUTO takes the tensor cores whenever the width allows.  On heads
    // under 384 MiB up to 16 rows (8 above H = 5120) take the warp-level MMAs fed from the weight stream
    // instead (H % 256 == 0): they start faster than the tcgen05 kernel (no TMEM, barrier or tensor-map
    // set-up).  4 rows on 2 MiB: 10.5 against 12.3 us; on 128 / 256 MiB: 32.8 / 53.5 against 34.6 /
    // 55.4 us.  From 512 MiB the eight-stage tcgen05 ring streams faster (512 MiB: 90.1 against 98.5
    // us; the 248,320 x 2048 head, 16 rows: 153.9 against 158.8 us), and with dependent launch a
    // batch-1 MTP3 round (three one-row drafts on 65,536 x 2048, then this verify) takes 269.5 against
    // 274.0 us.
    constexpr long long kMmaVerifyMaxBytes = 384ll << 20;
    const bool wmma = (path == VH_PATH_WARP_MMA) ||
                      (path == VH_PATH_AUTO && R <= kMmaRows && vh::gemv_mma_supported(R, H) &&
                       (long long)V * H * 2 < kMmaVerifyMaxBytes);
    const bool tensor = !wmma && ((path == VH_PATH_TENSOR) || (path == VH_PATH_AUTO && H % 64 == 0));
    const int mma_group = vh::gemv_mma_supported(kMmaRows, H) ? kMmaRows : 8;  // 16 rows need H <= 5120
    const int group = wmma ? mma_group : tensor ? kTcRows : gemv_group(H);
    for (int r0 = 0; r0 < R; r0 += group) {
        const int nr = std::min(group, R - r0);
        vh::AcceptTail tail;
        if (r0 + nr == R) {  // the final group also runs the acceptance scan
            tail.draft = draft_ids;
            tail.next_ids = next_ids;
            tail.accept_len = accept_len;
            tail.B = B;
            tail.k = k;
        }
        float* ml = row_maxlogit ? row_maxlogit + r0 : nullptr;
        cudaError_t e;
        if (wmma) {
            e = vh::launch_gemv_mma_bf16(X + (size_t)r0 * H, nr, H, W, nullptr, V, w, next_ids + r0, ml, tail, s,
                                         vh::long_steps(nr, (long long)V * H * 2));
        } else if (tensor) {
            e = vh::launch_verify_tc(X + (size_t)r0 * H, nr, H, W, V, w, next_ids + r0, ml, tail, s);
        } else {
            e = vh::launch_gemv_bf16(X + (size_t)r0 * H, nr, H, W, nullptr, V, w, next_ids + r0, ml, tail, s);
        }
        if (e != cudaSuccess) return launch_status(e);
    }
    return VH_OK;
}

vh_status spec_verify_greedy_nvfp4(const void* hidden, const uint8_t* Wq, const uint8_t* scales, float tensor_scale,
                                   const int32_t* draft_ids, int B, int k, int H, int V, int32_t* accept_len,
                                   int32_t* next_ids, float* row_maxlogit, void* ws, size_t ws_bytes, void* stream) {
    if (!hidden || !Wq || !scales || !draft_ids || !accept_len || !next_ids || !ws) return VH_ERR_NULL;
    if (B < 1 || k < 1 || k > 15 || H < 64 || H > kMaxH || H % 64 != 0 || V < 1) return VH_ERR_SHAPE;
    if ((long long)B * (k + 1) > 65536) return VH_ERR_SHAPE;
    if (!(tensor_scale > 0.0f) || !(tensor_scale < 3.0e38f)) return VH_ERR_SHAPE;
    if (!aligned(hidden, 16) || !aligned(Wq, 32) || !aligned(scales, 16) || !aligned(draft_ids, 4) ||
        !aligned(accept_len, 4) || !aligned(next_ids, 4) || !aligned(row_maxlogit, 4) || !aligned(ws, 16))
        return VH_ERR_ALIGN;
    const int R = B * (k + 1);
    if (ws_bytes < vh_verify_nvfp4_workspace_bytes(R, H)) return VH_ERR_WORKSPACE;
    vh_status st = check_device();
    if (st != VH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const vh::Workspace w = make_ws(ws, R);
    const uint16_t* x = static_cast<const uint16_t*>(hidden);
    const bool tc = (H % 512 == 0);
    if (tc && R > kTcFp4Rows) {
        // CTA-pair kernel over f16 copies of the hidden rows (workspace), up to
        // 256 rows per pass over the head
        uint16_t* xh = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + vh::ws_total_bytes(R));
        float* colscale = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xh) + vh::round16((size_t)R * H * 2));
        cudaError_t e = vh::launch_hidden_f16(x, R, H, tensor_scale, xh, colscale, s);
        if (e != cudaSuccess) return launch_status(e);
        for (int r0 = 0; r0 < R && e == cudaSuccess; r0 += kTcRows) {
            const int nr = std::min(kTcRows, R - r0);
            vh::AcceptTail tail;
            if (r0 + nr == R) {
                tail.draft = draft_ids;
                tail.next_ids = next_ids;
                tail.accept_len = accept_len;
                tail.B = B;
                tail.k = k;
            }
            float* ml = row_maxlogit ? row_maxlogit + r0 : nullptr;
            e = vh::launch_verify_fp4_pair(xh + (size_t)r0 * H, colscale + r0, nr, H, Wq, scales, V, w,
                                           next_ids + r0, ml, tail, s);
            if (e == cudaErrorNotSupported && r0 == 0) break;  // no cluster fits: row groups of 16 below
        }
        if (e != cudaErrorNotSupported) return e == cudaSuccess ? VH_OK : launch_status(e);
        cudaGetLastError();
    }
    // up to 16 rows (or H off the pair kernel's grid): warp-level MMAs for up
    // to 8 rows (H = 256 * 2^i <= 4096), tcgen05 groups of 16 for more (or
    // MMA groups of 8 where H % 512 != 0), else CUDA cores
    const bool mma = vh::nvfp4_mma_supported(kMmaFp4Rows, H) && (R <= kMmaFp4Rows || !tc);
    const int grp = mma ? kMmaFp4Rows : tc ? kTcFp4Rows : gemv_group(H);
    for (int r0 = 0; r0 < R; r0 += grp) {
        const int nr = std::min(grp, R - r0);
        vh::AcceptTail tail;
        if (r0 + nr == R) {  // the final group also runs the acceptance scan
            tail.draft = draft_ids;
            tail.next_ids = next_ids;
            tail.accept_len = accept_len;
            tail.B = B;
            tail.k = k;
        }
        float* ml = row_maxlogit ? row_maxlogit + r0 : nullptr;
        const uint16_t* xr = x + (size_t)r0 * H;
        cudaError_t e =
            mma  ? vh::launch_nvfp4_mma(xr, nr, H, Wq, scales, tensor_scale, nullptr, V, w, next_ids + r0, ml, s, tail)
            : tc ? vh::launch_nvfp4_tc(xr, nr, H, Wq, scales, tensor_scale, nullptr, V, w, next_ids + r0, ml, s, tail)
                 : vh::launch_gemv_nvfp4(xr, nr, H, Wq, scales, tensor_scale, nullptr, V, w, next_ids + r0, ml, s,
                                         tail);
        if (e != cudaSuccess) return launch_status(e);
    }
    return VH_OK;
}

size_t vh_nvfp4_packed_bytes(int V, int H) { return vh::nvfp4_packed_bytes(V, H); }

vh_status vh_nvfp4_pack(const uint8_t* Wq, const uint8_t* scales, int V, int H, void* packed, size_t packed_bytes,
                        void* stream) {
    if (!Wq || !scales || !packed) return VH_ERR_NULL;
    if (V < 1 || H < 256 || H > kMaxH || H % 256 != 0) return VH_ERR_SHAPE;
    if (!aligned(Wq, 16) || !aligned(scales, 16) || !aligned(packed, 16)) return VH_ERR_ALIGN;
    if (packed_bytes < vh::nvfp4_packed_bytes(V, H)) return VH_ERR_WORKSPACE;
    vh_status st = check_device();
    if (st != VH_OK) return st;
    return launch_status(vh::launch_nvfp4_pack(Wq, scales, V, H, static_cast<uint8_t*>(packed),
                                               static_cast<cudaStream_t>(stream)));
}

vh_status mtp_draft_head_argmax_nvfp4_packed(const void* hidden, const void* packed, float tensor_scale,
                                             const int32_t* cand_ids, int B, int H, int Vc, int32_t* ids,
                                             float* maxlogit, void* ws, size_t ws_bytes, void* stream) {
    if (!hidden || !packed || !cand_ids || !ids || !maxlogit || !ws) return VH_ERR_NULL;
    if (B < 1 || B > kMaxDraftB || !packed_shape_ok(H) || Vc < 1) return VH_ERR_SHAPE;
    if (!(tensor_scale > 0.0f) || !(tensor_scale < 3.0e38f)) return VH_ERR_SHAPE;
    if (!aligned(hidden, 16) || !aligned(packed, 32) || !aligned(cand_ids, 4) || !aligned(ids, 4) ||
        !aligned(maxlogit, 4) || !aligned(ws, 16))
        return VH_ERR_ALIGN;
    if (ws_bytes < vh_workspace_bytes(B)) return VH_ERR_WORKSPACE;
    vh_status st = check_device();
    if (st != VH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const vh::Workspace w = make_ws(ws, B);
    const uint16_t* x = static_cast<const uint16_t*>(hidden);
    const uint8_t* P = static_cast<const uint8_t*>(packed);
    for (int b0 = 0; b0 < B; b0 += kPackedRows) {
        const int nb = std::min(kPackedRows, B - b0);
        cudaError_t e = vh::launch_nvfp4_packed(x + (size_t)b0 * H, nb, H, P, tensor_scale, cand_ids, Vc, w, ids + b0,
                                                maxlogit + b0, s);
        if (e != cudaSuccess) return launch_status(e);
    }
    return VH_OK;
}

vh_status spec_verify_greedy_nvfp4_packed(const void* hidden, const void* packed, float tensor_scale,
                                          const int32_t* draft_ids, int B, int k, int H, int V, int32_t* accept_len,
                                          int32_t* next_ids, float* row_maxlogit, void* ws, size_t ws_bytes,
                                          void* stream) {
    if (!hidden || !packed || !draft_ids || !accept_len || !next_ids || !ws) return VH_ERR_NULL;
    if (B < 1 || k < 1 || k > 15 || !packed_shape_ok(H) || V < 1) return VH_ERR_SHAPE;
    if ((long long)B * (k + 1) > 65536) return VH_ERR_SHAPE;
    if (!(tensor_scale > 0.0f) || !(tensor_scale < 3.0e38f)) return VH_ERR_SHAPE;
    if (!aligned(hidden, 16) || !aligned(packed, 32) || !aligned(draft_ids, 4) || !aligned(accept_len, 4) ||
        !aligned(next_ids, 4) || !aligned(row_maxlogit, 4) || !aligned(ws, 16))
        return VH_ERR_ALIGN;
    const int R = B * (k + 1);
    if (ws_bytes < vh_workspace_bytes(R)) return VH_ERR_WORKSPACE;
    vh_status st = check_device();
    if (st != VH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const vh::Workspace w = make_ws(ws, R);
    const uint16_t* x = static_cast<const uint16_t*>(hidden);
    const uint8_t* P = static_cast<const uint8_t*>(packed);
    for (int r0 = 0; r0 < R; r0 += kPackedRows) {
        const int nr = std::min(kPackedRows, R - r0);
        vh::AcceptTail tail;
        if (r0 + nr == R) {  // the final group also runs the acceptance scan
            tail.draft = draft_ids;
            tail.next_ids = next_ids;
            tail.accept_len = accept_len;
            tail.B = B;
            tail.k = k;
        }
        float* ml = row_maxlogit ? row_maxlogit + r0 : nullptr;
        cudaError_t e = vh::launch_nvfp4_packed(x + (size_t)r0 * H, nr, H, P, tensor_scale, nullptr, V, w,
                                                next_ids + r0, ml, s, tail);
        if (e != cudaSuccess) return launch_status(e);
    }
    return VH_OK;
}

vh_status spec_verify_greedy(const void* hidden, const void* W_full, const int32_t* draft_ids, int B, int k, int H,
                             int V, int32_t* accept_len, int32_t* next_ids, float* row_maxlogit, void* ws,
                             size_t ws_bytes, void* stream) {
    return spec_verify_greedy_path(hidden, W_full, draft_ids, B, k, H, V, accept_len, next_ids, row_maxlogit, ws,
                                   ws_bytes, stream, VH_PATH_AUTO);
}

}  // extern "C"
