/*
 * verifyhead — restricted-vocabulary MTP draft head and greedy speculative
 * verification on one GPU (GB300, sm_103a).  C ABI of libverifyhead.so.
 *
 * Source of the method: "少读一张大表，草稿路径才真正快起来" in the Qwen3.8
 * Flash dual-Spark tuning log (cnblogs): the MTP draft path scores a smaller
 * candidate table (65,536 rows) instead of the 248,320-row full output head,
 * takes the argmax and maps it to the global token id; the target model keeps
 * the full head and verifies the draft.  "长上下文推理优化" §5 gives the
 * speculative loop (MTP proposal -> target verification -> accept several
 * tokens; acceptance rate and mean accepted tokens per step).  "为什么生产推理我
 * 默认 vLLM" §3 names the NVFP4 4-bit weight format used for the 4-bit head.
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must be device memory (or managed
 *    memory) owned by the caller; the library never allocates, frees or
 *    synchronises.  Work is enqueued on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and outputs are valid in stream order.
 *  - Arguments are checked on the host before anything is launched; a failed
 *    check returns a negative status and launches nothing.  VH_ERR_LAUNCH
 *    reports a CUDA launch error (the workspace must then be re-zeroed).
 *  - Argmax rule: the largest fp32 score wins; equal scores go to the lowest
 *    global token id (for the draft heads given their precondition of
 *    ascending candidate ids; see mtp_draft_head_argmax).  NaN scores count
 *    as -inf; -0 equals +0.
 *  - bf16 tensors are passed as raw 16-bit patterns, row-major.
 *  - Workspace: `ws` is a caller-owned device buffer of at least
 *    vh_workspace_bytes(rows) bytes, 16-byte aligned, zeroed ONCE by the
 *    caller after allocation.  Every call leaves it zeroed again, so
 *    consecutive calls in one stream (or a captured CUDA graph) can reuse it
 *    with no memset.  Calls that may overlap in time (different streams)
 *    need different workspaces.
 *  - No global state beyond thread-safe caches of per-device launch facts
 *    (SM count, occupancy): calls are thread-safe given distinct workspaces.
 *  - Kernels launch as programmatic dependents of the previous kernel in the
 *    stream and may begin reading their weight table (W_cand, W_full, the
 *    4-bit tables) before that kernel has finished; everything else is read
 *    only after it has.  A kernel lets its dependent start early only if it
 *    signals so (griddepcontrol.launch_dependents): this library's kernels
 *    do and never write a weight table.  A table written by a copy, or by a
 *    kernel that does not signal early, is seen complete; do not write a
 *    weight table from a kernel that signals early right before a call.
 *  - The same sources also build as libverifyhead_debug.so (-DVH_DEBUG): an
 *    identical ABI whose kernels check their row indices on the device and
 *    report a failed check in the workspace error word (bit 2) instead of
 *    touching memory out of range.
 */
#ifndef VERIFYHEAD_H
#define VERIFYHEAD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VH_API __attribute__((visibility("default")))
#else
#define VH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VH_OK = 0,
    VH_ERR_NULL = -1,      /* a required pointer is NULL */
    VH_ERR_SHAPE = -2,     /* a size is out of range or not a required multiple */
    VH_ERR_ALIGN = -3,     /* a pointer is not aligned as documented */
    VH_ERR_WORKSPACE = -4, /* ws_bytes < vh_workspace_bytes(rows) */
    VH_ERR_LAUNCH = -5,    /* CUDA reported an error when launching */
    VH_ERR_DEVICE = -6     /* no usable CUDA device / unsupported architecture */
} vh_status;

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
VH_API int vh_version(void);

/* Human-readable name of a status code (static string, never NULL). */
VH_API const char* vh_status_string(int status);

/* Bytes of workspace needed by calls that produce `rows` argmax rows
 * (rows = B for the draft heads, B*(k+1) for verification).  0 if rows < 1. */
VH_API size_t vh_workspace_bytes(int rows);

/*
 * Restricted-vocabulary draft head, bf16 weights.
 *
 * For each hidden row b < B:
 *     s[b,c]      = sum_h hidden[b,h] * W_cand[c,h]      (fp32 accumulation)
 *     ids[b]      = cand_ids[argmax_c s[b,c]]            (lowest id on ties)
 *     maxlogit[b] = max_c s[b,c]
 * Scores are never written to memory.  ("少读一张大表": only the small
 * candidate table is read; the winner is returned as a global token id.)
 *
 *  hidden    device, bf16 [B][H], 16-byte aligned
 *  W_cand    device, bf16 [Vc][H] row-major, 32-byte aligned (a separate copy
 *            of the candidate rows, not a view of the full head)
 *  cand_ids  device, int32 [Vc], ascending and distinct (precondition, not
 *            checked; up to 16 hidden rows per call, ties are broken by id
 *            either way, above that by position in cand_ids), values in
 *            [0, 2^31)
 *  B         1 <= B <= 256.  B > 16 with H % 64 == 0: all rows in one pass of
 *            the tcgen05 contraction over W_cand.  Otherwise groups of 16
 *            hidden rows when H % 256 == 0 and H <= 5120, else of 8, each
 *            reading W_cand once: 2-16 rows on warp-level MMAs when H % 256
 *            == 0, one row on the streaming GEMV, or on the warp-level MMAs
 *            when H is 256 or 512 or the table is 384 MiB or more
 *  H         16 <= H <= 65536, H % 16 == 0
 *  Vc        1 <= Vc <= 2^31 - 1
 *  ids       device, int32 [B] (out)
 *  maxlogit  device, fp32 [B] (out)
 *  ws        device workspace, ws_bytes >= vh_workspace_bytes(B)
 */
VH_API vh_status mtp_draft_head_argmax(const void* hidden, const void* W_cand, const int32_t* cand_ids, int B, int H,
                                int Vc, int32_t* ids, float* maxlogit, void* ws, size_t ws_bytes, void* stream);

/*
 * Draft head over candidate rows gathered from the full head (dynamic
 * candidate rows): no copy of the candidate table is made.
 *
 * "少读一张大表，草稿路径才真正快起来" reports upstream work (vLLM #59740) that
 * scores 32K fixed plus 16K per-step dynamic candidate rows; the fixed rows
 * can live in a separate table (mtp_draft_head_argmax), while a per-step set
 * is best read in place.  For each hidden row b < B:
 *     s[b,i]      = sum_h hidden[b,h] * W_full[row_ids[i],h]   (fp32 accumulation)
 *     ids[b]      = row_ids[argmax_i s[b,i]]     (ties: the lowest row id)
 *     maxlogit[b] = max_i s[b,i]
 *
 *  hidden    device, bf16 [B][H], 16-byte aligned
 *  W_full    device, bf16 [V][H] row-major, 32-byte aligned
 *  row_ids   device, int32 [n_ids], any order, repeats allowed; entries
 *            outside [0, V) are ignored (never read).  At least one entry
 *            must lie in [0, V), otherwise ids/maxlogit are unspecified.
 *  B         1 <= B <= 256;  H: 16 <= H <= 65536, H % 16 == 0
 *  n_ids     >= 1;  V >= 1
 *  ids, maxlogit, ws: as for mtp_draft_head_argmax
 */
VH_API vh_status mtp_draft_head_argmax_gather(const void* hidden, const void* W_full, const int32_t* row_ids, int B,
                                              int H, int n_ids, int V, int32_t* ids, float* maxlogit, void* ws,
                                              size_t ws_bytes, void* stream);

/*
 * Restricted-vocabulary draft head, block-scaled 4-bit weights (NVFP4).
 *
 * Source: "为什么生产推理我默认 vLLM" §3 (NVFP4: 4-bit weights with scale
 * factors) and "少读一张大表，草稿路径才真正快起来" (the upstream candidate
 * head keeps its candidate rows in NVFP4; the draft returns a global id from
 * the candidate table).
 *
 * Weight (c, h) = e2m1(code) * e4m3(scales[c][h/16]) * tensor_scale, where
 * code is the low nibble of Wq[c][h/2] for even h and the high nibble for
 * odd h; E2M1 = sign, 2 exponent bits (bias 1), 1 mantissa bit (magnitudes
 * 0 0.5 1 1.5 2 3 4 6); E4M3 = OCP FP8 e4m3fn (bias 7, max 448).  Scores,
 * ids and maxlogit are as for mtp_draft_head_argmax.  The tensor scale is
 * applied after accumulation (the result equals the per-weight rule up to
 * fp32 rounding).
 *
 * Kernels: one hidden row on CUDA cores; 2..8 rows with H = 256 * 2^i <=
 * 4096 in one pass of warp-level MMAs fed from registers; otherwise tcgen05
 * passes of 16 rows when H % 512 == 0, warp-level MMA passes of 8 rows when
 * H == 256, else CUDA-core passes of 8 rows.  Every pass reads the whole
 * table once.  (A head converted once with vh_nvfp4_pack is scored faster by
 * mtp_draft_head_argmax_nvfp4_packed, below.)
 *
 *  hidden        device, bf16 [B][H], 16-byte aligned
 *  Wq            device, uint8 [Vc][H/2], 32-byte aligned
 *  scales        device, uint8 [Vc][H/16], 16-byte aligned
 *  tensor_scale  finite, > 0
 *  cand_ids      as above
 *  B             1 <= B <= 256;  H: 64 <= H <= 65536, H % 64 == 0
 *  ids, maxlogit, ws: as above
 */
VH_API vh_status mtp_draft_head_argmax_nvfp4(const void* hidden, const uint8_t* Wq, const uint8_t* scales,
                                      float tensor_scale, const int32_t* cand_ids, int B, int H, int Vc,
                                      int32_t* ids, float* maxlogit, void* ws, size_t ws_bytes, void* stream);

/*
 * Greedy speculative verification over the full output head.
 *
 * Source: "少读一张大表，草稿路径才真正快起来" (the draft path scores a small
 * candidate table while the target model keeps the full 248,320-row head and
 * verifies the draft tokens) and "长上下文推理优化" §5 (the MTP loop: draft
 * proposals, target verification, several tokens accepted per step;
 * acceptance rate and mean accepted length as its metrics).  The greedy rule
 * below is the plainest reading of "the target verifies": a draft token is
 * accepted while it equals the target's own argmax at that position.
 *
 * Row r = b*(k+1) + j of `hidden` is the target model's hidden state for
 * sequence b after its context plus draft tokens 0..j-1 (j = 0 is the
 * position right after the last verified token).  Then
 *     next_ids[r]     = argmax_v sum_h hidden[r,h] * W_full[v,h]   (lowest v on ties)
 *     row_maxlogit[r] = the maximum score                          (optional)
 *     accept_len[b]   = number of leading j < k with next_ids[b*(k+1)+j] == draft_ids[b*k+j]
 * so sequence b emits draft_ids[b, 0..a-1] followed by next_ids[b*(k+1)+a]
 * (the correction token, or the bonus token when a == k).
 *
 *  hidden        device, bf16 [B*(k+1)][H], 16-byte aligned
 *  W_full        device, bf16 [V][H] row-major, 32-byte aligned
 *  draft_ids     device, int32 [B][k]
 *  B, k          B >= 1, 1 <= k <= 15, B*(k+1) <= 65536
 *  H             16 <= H <= 65536, H % 16 == 0
 *  V             1 <= V < 2^31
 *  accept_len    device, int32 [B] (out), values in 0..k
 *  next_ids      device, int32 [B*(k+1)] (out)
 *  row_maxlogit  device, fp32 [B*(k+1)] (out) or NULL
 *  ws            device workspace, ws_bytes >= vh_workspace_bytes(B*(k+1))
 *
 * Rows are processed in groups of at most 256 on the tensor cores (H % 64
 * == 0; against a head under 384 MiB up to 16 rows on warp-level MMAs when
 * H % 256 == 0 and H <= 5120, up to 8 when 5120 < H <= 10240) or 8 on CUDA
 * cores (other H); each group reads W_full once.
 */
VH_API vh_status spec_verify_greedy(const void* hidden, const void* W_full, const int32_t* draft_ids, int B, int k, int H,
                             int V, int32_t* accept_len, int32_t* next_ids, float* row_maxlogit, void* ws,
                             size_t ws_bytes, void* stream);

/*
 * mtp_draft_head_argmax without a caller workspace (no counterpart in the
 * source pages; an interface addition).
 *
 * For callers that cannot allocate device memory or pass a workspace: e.g.
 * an engine's per-step execute hook or plugin interface that gives extensions
 * no allocator, or a decode loop with a fixed memory plan, where cudaMalloc
 * may synchronise the device or fail mid-step.  Results are those of
 * mtp_draft_head_argmax with the same arguments.
 *
 * Scratch is a fixed 4 KiB device array inside this library, on every device
 * that loads it, kept until the process exits.  Limit: B <= 256 hidden rows
 * per call; a larger B returns VH_ERR_WORKSPACE and launches nothing.  The
 * call allocates and frees nothing.  It clears the part of the array it uses
 * (cudaMemsetAsync on `stream`) before the kernel, because the array keeps
 * whatever the previous call left.
 *
 * All calls on one device share that single array: calls that can overlap
 * on the GPU (different streams without ordering, several host threads)
 * race and may return wrong ids.  Keep such calls in one stream.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  The cached address belongs to that
 * device's context: after cudaDeviceReset it may be stale, so a device reset
 * in the process is not supported for this entry point.
 *
 * Arguments as for mtp_draft_head_argmax, without ws / ws_bytes.
 */
VH_API vh_status mtp_draft_head_argmax_static_ws(const void* hidden, const void* W_cand, const int32_t* cand_ids,
                                                 int B, int H, int Vc, int32_t* ids, float* maxlogit,
                                                 void* stream);

/*
 * Error word of the workspace: a 32-bit value at byte offset
 * vh_workspace_error_offset() of `ws` (the same offset for every workspace
 * size).  Bit 1: a bounded internal wait of a tensor-core kernel expired
 * (about 2 s; e.g. the GPU is oversubscribed or another process holds its
 * tensor memory) and the kernel stopped early.  Bit 2 (debug build only): a
 * device-side index check failed and the access was skipped.  Either way the
 * outputs of that call are invalid.  The library never clears this word: the
 * caller may read it (one 4-byte copy) and reset it.
 */
VH_API size_t vh_workspace_error_offset(void);

/*
 * Self-test of that bounded-wait path: launches one CTA that waits on a
 * barrier nothing completes, gives up after `timeout_us` microseconds
 * (1..1,000,000), sets *flag |= 1 (device memory, 4-byte aligned) and
 * returns.  The context stays usable.  No counterpart in the source pages.
 */
VH_API vh_status vh_selftest_bounded_wait(unsigned int* flag, unsigned int timeout_us, void* stream);

/*
 * Workspace size for spec_verify_greedy_nvfp4 with `rows` = B*(k+1) hidden
 * rows of width H: the argmax workspace of vh_workspace_bytes(rows) followed
 * by scratch for f16 copies of the hidden rows (rows*H*2 bytes) and one
 * float per row, each rounded up to 16 bytes.  0 for rows < 1 or H < 1.
 */
VH_API size_t vh_verify_nvfp4_workspace_bytes(int rows, int H);

/*
 * Greedy speculative verification over a block-scaled 4-bit full head (the
 * NVFP4 format of mtp_draft_head_argmax_nvfp4, rows = the V vocabulary
 * entries).  Rows, next_ids, row_maxlogit and accept_len are defined as for
 * spec_verify_greedy, with W_full replaced by the decoded 4-bit head.
 * Source: the verification of "少读一张大表，草稿路径才真正快起来" and
 * "长上下文推理优化" §5 (as for spec_verify_greedy) over the NVFP4 weights of
 * "为什么生产推理我默认 vLLM" §3.
 *
 * Kernels: up to 8 rows in one pass of warp-level MMAs fed from registers
 * (H = 256 * 2^i <= 4096); up to 16 rows in one tcgen05 pass with N = 16
 * (H % 512 == 0); more rows (H % 512 == 0) on a CTA pair (tcgen05
 * cta_group::2) with N = 128 or 256, up to 256 rows per pass over the head,
 * after converting the hidden rows to f16 with a per-row power-of-two
 * prescale into the workspace scratch (exact for every element within 2^31
 * of its row's largest magnitude).  Other H: CUDA cores, groups of 8 rows.
 *
 *  hidden        device, bf16 [B*(k+1)][H], 16-byte aligned
 *  Wq, scales    device, uint8 [V][H/2] (32-byte aligned), uint8 [V][H/16] (16-byte aligned)
 *  tensor_scale  finite, > 0
 *  B, k, V       as for spec_verify_greedy;  H: 64 <= H <= 65536, H % 64 == 0
 *  draft_ids, accept_len, next_ids, row_maxlogit: as for spec_verify_greedy
 *  ws, ws_bytes  device, 16-byte aligned, zeroed once, at least
 *                vh_verify_nvfp4_workspace_bytes(B*(k+1), H) bytes
 *                (VH_ERR_WORKSPACE otherwise); the argmax part is left zeroed,
 *                the scratch holds the last call's f16 rows
 */
VH_API vh_status spec_verify_greedy_nvfp4(const void* hidden, const uint8_t* Wq, const uint8_t* scales,
                                          float tensor_scale, const int32_t* draft_ids, int B, int k, int H, int V,
                                          int32_t* accept_len, int32_t* next_ids, float* row_maxlogit, void* ws,
                                          size_t ws_bytes, void* stream);

/* Kernel selection for spec_verify_greedy_path. */
typedef enum {
    VH_PATH_AUTO = 0,      /* 1-16 rows, H % 256 == 0, H <= 5120 (1-8 rows up to H = 10240) and a
                              head under 384 MiB: VH_PATH_WARP_MMA; else tcgen05 when H % 64 == 0,
                              else CUDA cores */
    VH_PATH_CUDA_CORE = 1, /* streaming GEMV, groups of 8 rows */
    VH_PATH_TENSOR = 2,    /* tcgen05 skinny GEMM, groups of 256 rows; VH_ERR_SHAPE if H % 64 != 0 */
    VH_PATH_WARP_MMA = 3   /* warp-level MMAs fed from the weight stream, groups of 16 rows (8 when
                              H > 5120); VH_ERR_SHAPE unless H % 256 == 0 and H <= 10240 */
} vh_path;

/* spec_verify_greedy with an explicit kernel choice (same results up to fp32
 * summation order); the same passages define it. */
VH_API vh_status spec_verify_greedy_path(const void* hidden, const void* W_full, const int32_t* draft_ids, int B, int k,
                                  int H, int V, int32_t* accept_len, int32_t* next_ids, float* row_maxlogit,
                                  void* ws, size_t ws_bytes, void* stream, int path);

/* mtp_draft_head_argmax_nvfp4 with an explicit kernel choice (same results
 * up to fp32 summation order; the same passages define it).  VH_PATH_TENSOR:
 * the tensor-core kernels that mtp_draft_head_argmax_nvfp4 takes for B > 1,
 * for any B (warp-level MMAs in passes of 8 rows for H = 256 * 2^i <= 4096
 * and B <= 8, else tcgen05 passes of 16 rows when H % 512 == 0, else
 * warp-level MMA passes of 8 rows; VH_ERR_SHAPE when neither applies).
 * VH_PATH_CUDA_CORE: the streaming GEMV on CUDA cores (one pass per 8 rows,
 * fewer for wide H).  VH_PATH_AUTO: the kernel mtp_draft_head_argmax_nvfp4
 * runs. */
VH_API vh_status mtp_draft_head_argmax_nvfp4_path(const void* hidden, const uint8_t* Wq, const uint8_t* scales,
                                                  float tensor_scale, const int32_t* cand_ids, int B, int H, int Vc,
                                                  int32_t* ids, float* maxlogit, void* ws, size_t ws_bytes,
                                                  void* stream, int path);

/*
 * Tiled layout of a block-scaled 4-bit head (same NVFP4 format as
 * mtp_draft_head_argmax_nvfp4, "为什么生产推理我默认 vLLM" §3; NVFP4 candidate
 * rows in "少读一张大表，草稿路径才真正快起来").  The weights are static, so a
 * caller converts them once (at load time) with vh_nvfp4_pack and then scores
 * the tiled copy with the *_nvfp4_packed calls, which read the same bytes per
 * call as the row-major calls but stream them front to back in the order the
 * tensor-core fragments need them.
 *
 * Layout: rows in blocks of 16 and K in tiles of 256 elements; tile (block
 * b, tile t) is the 2,304-byte record at byte ((b * H/256) + t) * 2304:
 *   [h*1024 + L*32, +32) for h = 0, 1 and L = 0..31: the 32 code bytes of row
 *       16b + L/4 + 8h, elements 256t + 64*(L%4) + [0, 64) (nibble order as in
 *       the row-major codes);
 *   [2048 + L*8 + h*4, +4): the 4 E4M3 scales of those elements.
 * Rows past V are zero.  Size: vh_nvfp4_packed_bytes(V, H) =
 * ceil(V/16) * 9*H bytes; 0 unless H % 256 == 0.
 */
VH_API size_t vh_nvfp4_packed_bytes(int V, int H);

/* Row-major codes Wq [V][H/2] and scales [V][H/16] (device, 16-byte aligned)
 * -> `packed` (device, 16-byte aligned, at least vh_nvfp4_packed_bytes(V, H)
 * bytes, else VH_ERR_WORKSPACE).  V >= 1; 256 <= H <= 65536, H % 256 == 0.
 * Enqueued on `stream`; allocates nothing. */
VH_API vh_status vh_nvfp4_pack(const uint8_t* Wq, const uint8_t* scales, int V, int H, void* packed,
                               size_t packed_bytes, void* stream);

/* mtp_draft_head_argmax_nvfp4 over the tiled copy made by vh_nvfp4_pack (the
 * same ids and max logits up to fp32 summation order).  One pass over the
 * table per 16 hidden rows on warp-level tensor-core MMAs, the codes streamed
 * straight into registers.  packed: device, 32-byte aligned.  H % 256 == 0
 * and H <= 6144 (the f16 copy of 16 hidden rows fits in shared memory), else
 * VH_ERR_SHAPE.  Other arguments as for mtp_draft_head_argmax_nvfp4. */
VH_API vh_status mtp_draft_head_argmax_nvfp4_packed(const void* hidden, const void* packed, float tensor_scale,
                                                    const int32_t* cand_ids, int B, int H, int Vc, int32_t* ids,
                                                    float* maxlogit, void* ws, size_t ws_bytes, void* stream);

/* spec_verify_greedy_nvfp4 over the tiled copy of the full 4-bit head (V
 * rows): one pass over the head per 16 hidden rows, the acceptance scan in
 * the last pass.  Workspace: vh_workspace_bytes(B*(k+1)) (no f16 scratch).
 * Shapes as for mtp_draft_head_argmax_nvfp4_packed; B, k, V, outputs as for
 * spec_verify_greedy. */
VH_API vh_status spec_verify_greedy_nvfp4_packed(const void* hidden, const void* packed, float tensor_scale,
                                                 const int32_t* draft_ids, int B, int k, int H, int V,
                                                 int32_t* accept_len, int32_t* next_ids, float* row_maxlogit,
                                                 void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFYHEAD_H */
