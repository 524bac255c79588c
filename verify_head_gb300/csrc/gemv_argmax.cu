// Split-V streaming GEMV with a fused two-level argmax and candidate-id
// mapping, on CUDA cores.
//
// Draft head ("少读一张大表，草稿路径才真正快起来", Qwen3.8 Flash dual-Spark log):
// the draft path scores a small candidate table (65,536 rows instead of the
// 248,320-row full head), takes the maximum and returns the global token id
// of the winning candidate.  There each rank took a local argmax and the
// ranks exchanged (max score, global id); here the whole head sits on one GPU
// and the exchange becomes a 64-bit atomicMax on packed (score, id) keys.
//
// Layout: every warp owns a contiguous range of rows and streams each row
// once with 256-bit loads (a warp reads 1 KiB per instruction, two rows in
// flight); x is staged in shared memory.  A row's dot
// product is a lane-strided partial sum reduced with warp shuffles.  The
// per-warp best keys are merged in shared memory, then one atomicMax per
// (CTA, hidden row); the last CTA (ticket counter) decodes the keys, writes
// ids / max logits, optionally runs the acceptance scan, and re-zeroes the
// workspace.  No CTA ever waits on another.
#include <cuda_fp16.h>

#include <algorithm>

#include "vh_kernels.h"

namespace vh {

struct GemvArgs {
    const uint16_t* x;  // [nb][H] bf16
    const void* W;      // bf16 [n_rows][H], or 4-bit codes [n_rows][H/2]
    const uint8_t* scales;  // [n_rows][H/16] E4M3 (4-bit head only)
    float g;                // tensor scale (4-bit head only)
    const int32_t* cand;    // [n_rows] or nullptr
    int nb;
    int H;
    int n_rows;
    int rows_per_warp;
    Workspace ws;
    int32_t* ids;
    float* maxlogit;
    AcceptTail tail;
};

__device__ __forceinline__ U32x8 ld_x32(const uint16_t* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    uint4 a = q[0], b = q[1];
    U32x8 r;
    r.v[0] = a.x; r.v[1] = a.y; r.v[2] = a.z; r.v[3] = a.w;
    r.v[4] = b.x; r.v[5] = b.y; r.v[6] = b.z; r.v[7] = b.w;
    return r;
}

// 16-element bf16 dot product into two accumulators (even / odd elements).
__device__ __forceinline__ void dot16(const U32x8& w, const U32x8& x, float& a0, float& a1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a0 = fmaf(bf_lo(w.v[j]), bf_lo(x.v[j]), a0);
        a1 = fmaf(bf_hi(w.v[j]), bf_hi(x.v[j]), a1);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Merge per-warp best keys, publish with atomicMax, and let the last CTA
// decode, run the optional acceptance scan and reset the workspace.
template <int NB>
__device__ __forceinline__ void finish_argmax(const unsigned long long (&best)[NB], const GemvArgs& a) {
    __shared__ unsigned long long red[kWarps][NB];
    __shared__ unsigned int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
#pragma unroll
        for (int b = 0; b < NB; ++b) red[warp][b] = best[b];
    }
    __syncthreads();
    if (threadIdx.x < a.nb) {
        unsigned long long k = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) k = red[w][threadIdx.x] > k ? red[w][threadIdx.x] : k;
        if (k != 0) atomicMax(a.ws.keys + threadIdx.x, k);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(a.ws.ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x < a.nb) {
        unsigned long long k = atomicExch(a.ws.keys + threadIdx.x, 0ull);
        a.ids[threadIdx.x] = (int32_t)key_gid(k);
        if (a.maxlogit != nullptr) a.maxlogit[threadIdx.x] = key_score(k);
    }
    if (threadIdx.x == 0) atomicExch(a.ws.ticket, 0u);
    if (a.tail.draft != nullptr) {
        __threadfence();
        __syncthreads();
        const int k = a.tail.k;
        for (int b = threadIdx.x; b < a.tail.B; b += blockDim.x) {
            const volatile int32_t* nid = a.tail.next_ids + (size_t)b * (k + 1);
            const int32_t* d = a.tail.draft + (size_t)b * k;
            int acc = 0;
            while (acc < k && nid[acc] == d[acc]) ++acc;
            a.tail.accept_len[b] = acc;
        }
    }
}

// ---------------------------------------------------------------------------
// bf16 head.  x is staged in shared memory as bf16 (read once per chunk and
// shared by the two rows in flight); the row is walked in segments of 2048
// elements (four 32-byte chunks per lane).

template <int NB>
__global__ void __launch_bounds__(kThreads, (NB == 1 ? 2 : 1)) k_gemv_bf16(const GemvArgs a) {
    extern __shared__ __align__(16) uint16_t xs[];  // [NB][H]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = a.H, nch = H >> 4;  // 32-byte chunks per row
    const uint16_t* __restrict__ W = static_cast<const uint16_t*>(a.W);

    {
        const int n16 = NB * H / 8;
        for (int i = threadIdx.x; i < n16; i += blockDim.x) {
            const int b = i / (H / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (b < a.nb) v = reinterpret_cast<const uint4*>(a.x)[i];
            reinterpret_cast<uint4*>(xs)[i] = v;
        }
        __syncthreads();
    }

    unsigned long long best[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) best[b] = 0ull;

    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const long long r0 = gw * a.rows_per_warp;
    const long long r1 = min(r0 + (long long)a.rows_per_warp, (long long)a.n_rows);

    for (long long r = r0; r < r1; r += 2) {
        const bool two = (r + 1 < r1);
        const uint16_t* w0p = W + (size_t)r * H;
        const uint16_t* w1p = w0p + H;
        float p0[NB][2], p1[NB][2];
#pragma unroll
        for (int b = 0; b < NB; ++b) p0[b][0] = p0[b][1] = p1[b][0] = p1[b][1] = 0.f;
        for (int seg = 0; seg < nch; seg += 128) {
            U32x8 w0[4], w1[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = seg + lane + 32 * i;
                if (c < nch) {
                    w0[i] = ld_stream32(w0p + c * 16);
                    if (two) w1[i] = ld_stream32(w1p + c * 16);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = seg + lane + 32 * i;
                if (c < nch) {
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const U32x8 xv = ld_x32(xs + (size_t)b * H + c * 16);
                        dot16(w0[i], xv, p0[b][0], p0[b][1]);
                        if (two) dot16(w1[i], xv, p1[b][0], p1[b][1]);
                    }
                }
            }
        }
        const uint32_t g0 = a.cand ? (uint32_t)__ldg(a.cand + r) : (uint32_t)r;
        const uint32_t g1 = two ? (a.cand ? (uint32_t)__ldg(a.cand + r + 1) : (uint32_t)(r + 1)) : 0u;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float s0 = warp_sum(p0[b][0] + p0[b][1]);
            const unsigned long long k0 = make_key(s0, g0);
            best[b] = k0 > best[b] ? k0 : best[b];
            if (two) {
                const float s1 = warp_sum(p1[b][0] + p1[b][1]);
                const unsigned long long k1 = make_key(s1, g1);
                best[b] = k1 > best[b] ? k1 : best[b];
            }
        }
    }
    finish_argmax<NB>(best, a);
}

// ---------------------------------------------------------------------------
// Block-scaled 4-bit head on CUDA cores.  A lane chunk is 32 code bytes = 64
// elements = 4 scale blocks.  Each 16-element block is summed unscaled, then
// multiplied by its E4M3 scale; the tensor scale g multiplies the total.

__device__ __forceinline__ float2 e2m1x2_to_f2(uint32_t byte) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two_bytes) {
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(two_bytes));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

template <int NB>
__global__ void __launch_bounds__(kThreads) k_gemv_nvfp4(const GemvArgs a) {
    extern __shared__ __align__(16) uint16_t xs[];  // [NB][H]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = a.H, nch = H >> 6;  // 64-element (32-byte) chunks per row
    const uint8_t* __restrict__ Wq = static_cast<const uint8_t*>(a.W);

    {
        const int n16 = NB * H / 8;
        for (int i = threadIdx.x; i < n16; i += blockDim.x) {
            const int b = i / (H / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (b < a.nb) v = reinterpret_cast<const uint4*>(a.x)[i];
            reinterpret_cast<uint4*>(xs)[i] = v;
        }
        __syncthreads();
    }

    unsigned long long best[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) best[b] = 0ull;

    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const long long r0 = gw * a.rows_per_warp;
    const long long r1 = min(r0 + (long long)a.rows_per_warp, (long long)a.n_rows);

    for (long long r = r0; r < r1; ++r) {
        const uint8_t* qrow = Wq + (size_t)r * (H / 2);
        const uint8_t* srow = a.scales + (size_t)r * (H / 16);
        float acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = 0.f;
        for (int seg = 0; seg < nch; seg += 64) {
            U32x8 q[2];
            uint32_t sc[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int c = seg + lane + 32 * i;
                if (c < nch) {
                    q[i] = ld_stream32(qrow + c * 32);
                    sc[i] = __ldg(reinterpret_cast<const uint32_t*>(srow) + c);
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int c = seg + lane + 32 * i;
                if (c >= nch) continue;
                const float2 s01 = e4m3x2_to_f2(sc[i] & 0xFFFFu);
                const float2 s23 = e4m3x2_to_f2(sc[i] >> 16);
                const float sblk[4] = {s01.x, s01.y, s23.x, s23.y};
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    float w[16];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t word = q[i].v[blk * 2 + (j >> 2)];
                        const float2 f = e2m1x2_to_f2((word >> (8 * (j & 3))) & 0xFFu);
                        w[2 * j] = f.x;
                        w[2 * j + 1] = f.y;
                    }
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const U32x8 xv = ld_x32(xs + (size_t)b * H + c * 64 + blk * 16);
                        float p0 = 0.f, p1 = 0.f;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            p0 = fmaf(w[2 * j], bf_lo(xv.v[j]), p0);
                            p1 = fmaf(w[2 * j + 1], bf_hi(xv.v[j]), p1);
                        }
                        acc[b] = fmaf(p0 + p1, sblk[blk], acc[b]);
                    }
                }
            }
        }
        const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + r) : (uint32_t)r;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float s = warp_sum(acc[b]) * a.g;
            const unsigned long long k = make_key(s, gid);
            best[b] = k > best[b] ? k : best[b];
        }
    }
    finish_argmax<NB>(best, a);
}

// ---------------------------------------------------------------------------
// Host launchers.

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

template <typename K>
static cudaError_t launch_split_v(K kernel, size_t smem, int n_rows, GemvArgs& a, cudaStream_t s) {
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (per_sm < 1 || sms < 1) return cudaErrorInvalidConfiguration;
    // one resident wave; each warp gets a contiguous, equal share of rows
    long long grid = (long long)sms * per_sm;
    const long long min_rows_per_warp = 2;
    const long long max_grid = ((long long)n_rows + kWarps * min_rows_per_warp - 1) / (kWarps * min_rows_per_warp);
    grid = std::max(1LL, std::min(grid, max_grid));
    const long long warps = grid * kWarps;
    a.rows_per_warp = (int)(((long long)n_rows + warps - 1) / warps);
    grid = ((long long)n_rows + (long long)a.rows_per_warp * kWarps - 1) / ((long long)a.rows_per_warp * kWarps);
    kernel<<<(unsigned)grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gemv_bf16(const uint16_t* x, int nb, int H, const uint16_t* W, const int32_t* cand, int n_rows,
                             Workspace ws, int32_t* ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s) {
    GemvArgs a{};
    a.x = x; a.W = W; a.scales = nullptr; a.g = 1.f; a.cand = cand;
    a.nb = nb; a.H = H; a.n_rows = n_rows; a.ws = ws; a.ids = ids; a.maxlogit = maxlogit; a.tail = tail;
#define VH_GEMV_CASE(NBV) \
    if (nb <= NBV) return launch_split_v(k_gemv_bf16<NBV>, (size_t)NBV * H * 2, n_rows, a, s);
    VH_GEMV_CASE(1)
    VH_GEMV_CASE(2)
    VH_GEMV_CASE(4)
    VH_GEMV_CASE(8)
#undef VH_GEMV_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemv_nvfp4(const uint16_t* x, int nb, int H, const uint8_t* Wq, const uint8_t* scales, float g,
                              const int32_t* cand, int n_rows, Workspace ws, int32_t* ids, float* maxlogit,
                              cudaStream_t s) {
    GemvArgs a{};
    a.x = x; a.W = Wq; a.scales = scales; a.g = g; a.cand = cand;
    a.nb = nb; a.H = H; a.n_rows = n_rows; a.ws = ws; a.ids = ids; a.maxlogit = maxlogit;
#define VH_NVFP4_CASE(NBV) \
    if (nb <= NBV) return launch_split_v(k_gemv_nvfp4<NBV>, (size_t)NBV * H * 2, n_rows, a, s);
    VH_NVFP4_CASE(1)
    VH_NVFP4_CASE(2)
    VH_NVFP4_CASE(4)
    VH_NVFP4_CASE(8)
#undef VH_NVFP4_CASE
    return cudaErrorInvalidValue;
}

}  // namespace vh
