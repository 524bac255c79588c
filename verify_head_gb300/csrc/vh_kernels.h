// Internal launchers behind the C ABI (not part of the public interface).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "vh_common.cuh"

namespace vh {

// Limits of the C ABI shared by every entry point.
constexpr int kMaxDraftB = 256;  // hidden rows per draft call
constexpr int kMaxH = 65536;     // hidden width
constexpr int kGemvRows = 8;     // hidden rows per CUDA-core launch

// Hidden rows per CUDA-core launch for width H: up to kGemvRows, fewer when
// the staged hidden rows (rows x H bf16 in shared memory) would exceed 128 KiB.
inline int gemv_group(int H) {
    int g = kGemvRows;
    while (g > 1 && (size_t)g * H * 2 > 131072) g /= 2;
    return g;
}

// Optional acceptance scan run by the last CTA of a launch, after the group's
// argmax ids are written: accept_len[b] = leading j < k with
// next_ids[b*(k+1)+j] == draft[b*k+j], over all B sequences.
struct AcceptTail {
    const int32_t* draft = nullptr;  // [B][k]; nullptr = no scan
    const int32_t* next_ids = nullptr;  // [B*(k+1)], complete once this launch ends
    int32_t* accept_len = nullptr;   // [B]
    int B = 0;
    int k = 0;
};

// bf16 streaming GEMV + argmax over rows [0, n_rows) of W for nb <= 8 hidden
// rows.  gid of row r is cand[r] (cand != nullptr) or r.  With gather_V > 0
// the scan reads W row cand[r] of a [gather_V][H] head instead of row r (ids
// outside [0, gather_V) are skipped).
cudaError_t launch_gemv_bf16(const uint16_t* x, int nb, int H, const uint16_t* W, const int32_t* cand, int n_rows,
                             Workspace ws, int32_t* ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s,
                             int gather_V = 0);

// bf16 head for 1-16 hidden rows on warp-level MMAs fed straight from the
// weight stream (mma.m16n8k16, hidden rows as A, 8 head rows as B) + argmax.
// gemv_mma_supported: H % 256 == 0 and the hidden rows in fragment order
// (16*H bytes for up to 8 rows, 32*H for 9-16) fit 160 KiB of shared memory.
// Returns cudaErrorNotSupported otherwise.
bool gemv_mma_supported(int nb, int H);
// long_steps: 512-element steps (1 KiB of each head row per load step, one
// step in registers) when H % 512 == 0, else 256-element steps, two in flight.
cudaError_t launch_gemv_mma_bf16(const uint16_t* x, int nb, int H, const uint16_t* W, const int32_t* cand, int n_rows,
                                 Workspace ws, int32_t* ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s,
                                 bool long_steps = false);
// Hidden rows per launch group of the bf16 draft head: 16 where the warp-MMA
// kernel takes 16 rows (H % 256 == 0, H <= 5120), else gemv_group(H).
int draft_group(int H);
// One launch group (nb <= draft_group(H) hidden rows) of the bf16 draft head:
// the kernel both draft entry points use for that group size.
cudaError_t launch_draft_group(const uint16_t* x, int nb, int H, const uint16_t* W, const int32_t* cand, int n_rows,
                               Workspace ws, int32_t* ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s);

// Block-scaled 4-bit (E2M1 codes, E4M3 block scales, fp32 tensor scale)
// GEMV + argmax on CUDA cores, nb <= 8.
cudaError_t launch_gemv_nvfp4(const uint16_t* x, int nb, int H, const uint8_t* Wq, const uint8_t* scales, float g,
                              const int32_t* cand, int n_rows, Workspace ws, int32_t* ids, float* maxlogit,
                              cudaStream_t s, const AcceptTail& tail = AcceptTail{});

// Block-scaled 4-bit head on the tensor cores (exact f16 dequantisation,
// tcgen05 kind::f16), nb <= 16 hidden rows, H % 512 == 0.  Returns
// cudaErrorNotSupported for other shapes.
cudaError_t launch_nvfp4_tc(const uint16_t* x, int nb, int H, const uint8_t* Wq, const uint8_t* scales, float g,
                            const int32_t* cand, int Vc, Workspace ws, int32_t* ids, float* maxlogit, cudaStream_t s,
                            const AcceptTail& tail = AcceptTail{});

// Block-scaled 4-bit head on warp-level MMAs fed from registers (codes
// streamed per warp with cp.async, exact f16 dequantisation, fp32
// accumulation), nb <= 8 hidden rows, H = 256 * 2^i <= 4096.  Returns
// cudaErrorNotSupported for other shapes.
bool nvfp4_mma_supported(int nb, int H);
cudaError_t launch_nvfp4_mma(const uint16_t* x, int nb, int H, const uint8_t* Wq, const uint8_t* scales, float g,
                             const int32_t* cand, int Vc, Workspace ws, int32_t* ids, float* maxlogit, cudaStream_t s,
                             const AcceptTail& tail = AcceptTail{});

// Tiled ("packed") layout of a block-scaled 4-bit head: records of 16 rows x
// 256 elements (2,048 code bytes in MMA-fragment order + 256 scale bytes).
// nvfp4_packed_bytes: size for V rows of width H (0 unless H % 256 == 0).
size_t nvfp4_packed_bytes(long long V, int H);
// Shared memory of launch_nvfp4_packed for nb rows of width H, and its limit.
size_t nvfp4_packed_smem(int nb, int H);
size_t nvfp4_packed_max_smem();
// Row-major codes [V][H/2] + scales [V][H/16] -> the tiled layout.
cudaError_t launch_nvfp4_pack(const uint8_t* Wq, const uint8_t* scales, int V, int H, uint8_t* packed, cudaStream_t s);
// Block-scaled 4-bit head in the tiled layout, nb <= 16 hidden rows on
// warp-level MMAs, one pass over the table.  Returns cudaErrorNotSupported
// for other shapes.
cudaError_t launch_nvfp4_packed(const uint16_t* x, int nb, int H, const uint8_t* packed, float g, const int32_t* cand,
                                int Vc, Workspace ws, int32_t* ids, float* maxlogit, cudaStream_t s,
                                const AcceptTail& tail = AcceptTail{});

// tcgen05 skinny GEMM + per-row argmax + acceptance scan for R <= 256 hidden
// rows (H % 64 == 0).  Returns cudaErrorNotSupported when the shape does not
// fit the kernel.
cudaError_t launch_verify_tc(const uint16_t* X, int R, int H, const uint16_t* W, int V, Workspace ws,
                             int32_t* next_ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s);

// bf16 hidden rows [R][H] -> f16 rows prescaled by 2^k_r (largest |x| into
// [2^14, 2^15)) and colscale[r] = g * 2^-k_r, for launch_verify_fp4_pair.
cudaError_t launch_hidden_f16(const uint16_t* X, int R, int H, float g, uint16_t* Xh, float* colscale, cudaStream_t s);

// Block-scaled 4-bit full head on a CTA pair (exact f16 dequantisation in
// shared memory, tcgen05 cta_group::2, M = 256 W rows x N = 128 or 256 hidden
// rows) + per-row argmax + acceptance scan over the f16 rows of
// launch_hidden_f16, R <= 256, H % 512 == 0.  Returns cudaErrorNotSupported
// for other shapes or when no cluster fits.
cudaError_t launch_verify_fp4_pair(const uint16_t* Xh, const float* colscale, int R, int H, const uint8_t* Wq,
                                   const uint8_t* scales, int V, Workspace ws, int32_t* next_ids, float* maxlogit,
                                   const AcceptTail& tail, cudaStream_t s);

int sm_count();

}  // namespace vh
