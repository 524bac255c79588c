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
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "vh_kernels.h"
#include "vh_ptx.cuh"

namespace vh {

struct GemvArgs {
    const uint16_t* x;  // [nb][H] bf16
    const void* W;      // bf16 [n_rows][H], or 4-bit codes [n_rows][H/2]
    const uint8_t* scales;  // [n_rows][H/16] E4M3 (4-bit head only)
    float g;                // tensor scale (4-bit head only)
    const int32_t* cand;    // [n_rows] or nullptr
    int gather;             // 1: row r of the scan is W row cand[r] (rows outside [0, V) are skipped)
    int V;                  // rows of W when gathering
    int nb;
    int H;
    int n_rows;
    int rows_per_warp;
    unsigned int* err;
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
template <int NB, int NW = kWarps, typename Args>
__device__ __forceinline__ void finish_argmax(const unsigned long long (&best)[NB], const Args& a) {
    __shared__ unsigned long long red[NW][NB];
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
        for (int w = 0; w < NW; ++w) k = red[w][threadIdx.x] > k ? red[w][threadIdx.x] : k;
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
        vh_guard(k != 0ull || a.gather, a.err);  // every row of a candidate table has a winner
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
// shared by the rows in flight); the row is walked in segments of 2048
// elements (four 32-byte chunks per lane).  RPI rows per warp iteration.
//
// Programmatic dependent launch: the kernel lets the next kernel in the
// stream launch at once, prefetches its first rows into L2 (read-only
// weights), and only then waits for the previous kernel to finish, before
// it touches x or the workspace.

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Rows (per warp) whose lines are prefetched into L2 ahead of the row being
// loaded: more bytes in flight per SM without more registers.  Every 128-byte
// line of the row is prefetched (lane L takes the lines at L*128 + k*4096):
// one line per 256 bytes left half the row to demand misses and measured
// 0.8-2.8% slower.
constexpr int kPrefetchRows = 1;
constexpr int kGatherPrefetchRows = 1;  // gathering: rows listed next, prefetched from the id cache (2 was slower)

template <int NB, int RPI, bool GATHER>
__global__ void __launch_bounds__(kThreads, (NB == 1 ? 4 : 1)) k_gemv_bf16(const GemvArgs a) {
    extern __shared__ __align__(16) uint16_t xs[];  // [NB][H]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = a.H, nch = H >> 4;  // 32-byte chunks per row
    const uint16_t* __restrict__ W = static_cast<const uint16_t*>(a.W);

    // even split of the rows over every warp of the resident wave (13 or 14
    // rows each for 65,536 rows): every SM streams the same share
    const long long gw = (long long)blockIdx.x * kWarps + warp, nw = (long long)gridDim.x * kWarps;
    const long long r0 = gw * a.n_rows / nw;
    const long long r1 = (gw + 1) * a.n_rows / nw;

    // physical W row of scan position r (the identity unless gathering)
    auto wrow = [&](long long r) -> long long { return GATHER ? (long long)__ldg(a.cand + r) : r; };
    auto in_range = [&](long long pr) -> bool { return !GATHER || (pr >= 0 && pr < a.V); };

    pdl_launch_dependents();
    for (long long r = r0; r < min(r1, r0 + RPI); ++r) {
        const long long pr = wrow(r);
        if (in_range(pr))
            for (int c = lane; c < min(nch, 128); c += 32) prefetch_l2(W + (size_t)pr * H + c * 16);
    }
    pdl_wait();

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

    int idx_cache = 0;  // gathering: row ids of the next 32 scan positions, one per lane
    for (long long r = r0; r < r1; r += RPI) {
        if (GATHER && ((r - r0) & 31) == 0) {
            const long long rr = r + lane;
            idx_cache = rr < r1 ? __ldg(a.cand + rr) : -1;
        }
        if constexpr (kPrefetchRows > 0 && !GATHER) {  // keep rows ahead of the loads in flight to L2
            const long long rp = r + kPrefetchRows * RPI;
            for (int rr = 0; rr < RPI; ++rr)
                if (rp + rr < r1)
                    for (int c = lane * 4; c < nch; c += 128) prefetch_l2(W + (size_t)(rp + rr) * H + c * 16);
        } else if constexpr (kPrefetchRows > 0) {
            // gathering: the next positions' row ids come from the warp's id cache (a shuffle, no load);
            // a position in the next 32-id block is not prefetched
#pragma unroll
            for (int rr = 0; rr < kGatherPrefetchRows * RPI; ++rr) {
                const long long rp = r + RPI + rr;
                const int slot = (int)((rp - r0) & 31);
                if (rp < r1 && rp - r0 < (((r - r0) >> 5) + 1) * 32) {
                    const int pid = __shfl_sync(0xFFFFFFFFu, idx_cache, slot);
                    if (pid >= 0 && pid < a.V)
                        for (int c = lane * 4; c < nch; c += 128) prefetch_l2(W + (size_t)pid * H + c * 16);
                }
            }
        }
        const long long pr0 = GATHER ? (long long)__shfl_sync(0xFFFFFFFFu, idx_cache, (int)((r - r0) & 31)) : r;
        const long long pr1 =
            (RPI > 1 && r + 1 < r1)
                ? (GATHER ? (long long)__shfl_sync(0xFFFFFFFFu, idx_cache, (int)((r + 1 - r0) & 31)) : r + 1)
                : 0;
        const bool ok0 = in_range(pr0) && vh_guard(GATHER || pr0 < a.n_rows, a.err);
        const bool two = RPI > 1 && (r + 1 < r1) && in_range(pr1);
        const uint16_t* w0p = W + (size_t)(ok0 ? pr0 : 0) * H;
        const uint16_t* w1p = W + (size_t)(two ? pr1 : 0) * H;
        float p0[NB][2], p1[NB][2];
#pragma unroll
        for (int b = 0; b < NB; ++b) p0[b][0] = p0[b][1] = p1[b][0] = p1[b][1] = 0.f;
        for (int seg = 0; seg < nch; seg += 128) {
            U32x8 w0[4], w1[RPI > 1 ? 4 : 1];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = seg + lane + 32 * i;
                if (c < nch) {
                    if (ok0) w0[i] = ld_stream32(w0p + c * 16);
                    if (two) w1[RPI > 1 ? i : 0] = ld_stream32(w1p + c * 16);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = seg + lane + 32 * i;
                if (c < nch && ok0) {
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const U32x8 xv = ld_x32(xs + (size_t)b * H + c * 16);
                        dot16(w0[i], xv, p0[b][0], p0[b][1]);
                        if (two) dot16(w1[RPI > 1 ? i : 0], xv, p1[b][0], p1[b][1]);
                    }
                }
            }
        }
        const uint32_t g0 = GATHER ? (uint32_t)pr0 : (a.cand ? (uint32_t)__ldg(a.cand + r) : (uint32_t)r);
        const uint32_t g1 =
            two ? (GATHER ? (uint32_t)pr1 : (a.cand ? (uint32_t)__ldg(a.cand + r + 1) : (uint32_t)(r + 1))) : 0u;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float s0 = warp_sum(p0[b][0] + p0[b][1]);
            const unsigned long long k0 = ok0 ? make_key(s0, g0) : 0ull;
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
// Block-scaled 4-bit decoding helpers.  E2M1 pairs and E4M3 scale pairs go
// through the hardware conversions to f16x2 (exact: every E2M1 and E4M3
// value is an f16 value).

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

// ---------------------------------------------------------------------------
// Block-scaled 4-bit decode helpers.  Weights decode with one
// cvt.rn.f16x2.e2m1x2 per byte (exact); the hidden row is held as f16,
// prescaled by a power of two 2^k so that its largest magnitude lies in
// [2^14, 2^15) (exact for every element within 2^31 of the largest);
// products accumulate in fp32 with the mixed-precision fma.rn.f32.f16.  Each
// 16-element block sum is multiplied by its E4M3 scale; the total by g*2^-k.

__device__ __forceinline__ void split_h2(uint32_t w, unsigned short& lo, unsigned short& hi) {
    asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(w));
}

__device__ __forceinline__ float fma_f16_f32(unsigned short a, unsigned short b, float c) {
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}

// 16-element block: codes in (q0, q1) (element 2i in the low nibble of byte
// i), hidden row as 8 f16x2 words.  Unscaled fp32 sum.
// E2M1 pair in byte J of `word` -> f16x2, the byte taken through a .b8
// register view of the word (no shift / mask).
template <int J>
__device__ __forceinline__ uint32_t e2m1_byte_h2(uint32_t word) {
    uint32_t h2;
    if (J == 0)
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
            : "=r"(h2) : "r"(word));
    else if (J == 1)
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b1;\n\t}"
            : "=r"(h2) : "r"(word));
    else if (J == 2)
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b2;\n\t}"
            : "=r"(h2) : "r"(word));
    else
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b3;\n\t}"
            : "=r"(h2) : "r"(word));
    return h2;
}

template <int J>
__device__ __forceinline__ void nvfp4_pair_fma(uint32_t word, uint32_t xh, float& a0, float& a1) {
    const uint32_t w2 = e2m1_byte_h2<J>(word);
    unsigned short wl, wh, xl, xhh;
    split_h2(w2, wl, wh);
    split_h2(xh, xl, xhh);
    a0 = fma_f16_f32(wl, xl, a0);
    a1 = fma_f16_f32(wh, xhh, a1);
}

__device__ __forceinline__ float nvfp4_block16(uint32_t q0, uint32_t q1, const uint32_t* xh) {
    float a0 = 0.f, a1 = 0.f;
    nvfp4_pair_fma<0>(q0, xh[0], a0, a1);
    nvfp4_pair_fma<1>(q0, xh[1], a0, a1);
    nvfp4_pair_fma<2>(q0, xh[2], a0, a1);
    nvfp4_pair_fma<3>(q0, xh[3], a0, a1);
    nvfp4_pair_fma<0>(q1, xh[4], a0, a1);
    nvfp4_pair_fma<1>(q1, xh[5], a0, a1);
    nvfp4_pair_fma<2>(q1, xh[6], a0, a1);
    nvfp4_pair_fma<3>(q1, xh[7], a0, a1);
    return a0 + a1;
}


__device__ __forceinline__ uint32_t f32x2_to_h2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}

// ---------------------------------------------------------------------------
// Block-scaled 4-bit head, B = 1, H % 64 == 0, H <= 8192: direct streaming.
// Each warp owns a contiguous run of rows and reads every code row with
// 256-bit loads (one 64-element chunk = 32 code bytes + 4 scale bytes per
// lane), two rows in flight.  The hidden row is held in registers as f16,
// prescaled by 2^k so that its largest magnitude lies in [2^14, 2^15)
// (exact for every element within 2^31 of the largest); weights decode with
// cvt.rn.f16x2.e2m1x2 and accumulate in fp32 with fma.rn.f32.f16; each
// 16-element block sum is multiplied by its E4M3 scale, the row by g*2^-k.

template <int CPL>
__global__ void __launch_bounds__(kThreads, (CPL >= 4 ? 1 : 2)) k_gemv_nvfp4_direct(const GemvArgs a) {
    __shared__ float s_xmax[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = a.H, nch = H >> 6;
    const size_t qrow = (size_t)H / 2, srow = (size_t)H / 16;
    const uint8_t* __restrict__ Wq = static_cast<const uint8_t*>(a.W);

    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const long long r0 = gw * a.rows_per_warp;
    const long long r1 = min(r0 + (long long)a.rows_per_warp, (long long)a.n_rows);

    pdl_launch_dependents();
    for (long long r = r0; r < min(r1, r0 + 2); ++r)
        for (int c = lane; c < nch; c += 32) prefetch_l2(Wq + (size_t)r * qrow + c * 32);
    pdl_wait();

    // power-of-two prescale from the largest |x| (identical in every CTA)
    float m = 0.f;
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf_lo(v.x)), fabsf(bf_hi(v.x))), fmaxf(fabsf(bf_lo(v.y)), fabsf(bf_hi(v.y)))));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf_lo(v.z)), fabsf(bf_hi(v.z))), fmaxf(fabsf(bf_lo(v.w)), fabsf(bf_hi(v.w)))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) s_xmax[warp] = m;
    __syncthreads();
    float xmax = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) xmax = fmaxf(xmax, s_xmax[w]);
    const int k = xmax > 0.f ? min(127, 141 - (int)((__float_as_uint(xmax) >> 23) & 0xFF)) : 0;
    const float up = ldexpf(1.f, k), out_scale = a.g * ldexpf(1.f, -k);

    uint32_t xh[CPL][32];  // lane's chunks of x as f16x2 (element 2i in the low half)
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const int c = lane + 32 * j;
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            if (c < nch) {
                const uint32_t pr = reinterpret_cast<const uint32_t*>(a.x)[c * 32 + t];
                xh[j][t] = f32x2_to_h2(bf_lo(pr) * up, bf_hi(pr) * up);
            } else {
                xh[j][t] = 0u;
            }
        }
    }

    unsigned long long best = 0ull;
    for (long long r = r0; r < r1 && vh_guard(r1 <= a.n_rows, a.err); r += 2) {
        const bool two = (r + 1 < r1);
        U32x8 q0[CPL], q1[CPL];
        uint32_t s0[CPL], s1[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = lane + 32 * j;
            if (c < nch) {
                q0[j] = ld_stream32(Wq + (size_t)r * qrow + c * 32);
                s0[j] = __ldg(reinterpret_cast<const uint32_t*>(a.scales + (size_t)r * srow) + c);
                if (two) {
                    q1[j] = ld_stream32(Wq + (size_t)(r + 1) * qrow + c * 32);
                    s1[j] = __ldg(reinterpret_cast<const uint32_t*>(a.scales + (size_t)(r + 1) * srow) + c);
                }
            }
        }
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = lane + 32 * j;
            if (c < nch) {
                const float2 a01 = e4m3x2_to_f2(s0[j] & 0xFFFFu), a23 = e4m3x2_to_f2(s0[j] >> 16);
                acc0 = fmaf(nvfp4_block16(q0[j].v[0], q0[j].v[1], &xh[j][0]), a01.x, acc0);
                acc0 = fmaf(nvfp4_block16(q0[j].v[2], q0[j].v[3], &xh[j][8]), a01.y, acc0);
                acc0 = fmaf(nvfp4_block16(q0[j].v[4], q0[j].v[5], &xh[j][16]), a23.x, acc0);
                acc0 = fmaf(nvfp4_block16(q0[j].v[6], q0[j].v[7], &xh[j][24]), a23.y, acc0);
                if (two) {
                    const float2 b01 = e4m3x2_to_f2(s1[j] & 0xFFFFu), b23 = e4m3x2_to_f2(s1[j] >> 16);
                    acc1 = fmaf(nvfp4_block16(q1[j].v[0], q1[j].v[1], &xh[j][0]), b01.x, acc1);
                    acc1 = fmaf(nvfp4_block16(q1[j].v[2], q1[j].v[3], &xh[j][8]), b01.y, acc1);
                    acc1 = fmaf(nvfp4_block16(q1[j].v[4], q1[j].v[5], &xh[j][16]), b23.x, acc1);
                    acc1 = fmaf(nvfp4_block16(q1[j].v[6], q1[j].v[7], &xh[j][24]), b23.y, acc1);
                }
            }
        }
        {
            const float sc = warp_sum(acc0) * out_scale;
            const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + r) : (uint32_t)r;
            const unsigned long long kk = make_key(sc, gid);
            best = kk > best ? kk : best;
        }
        if (two) {
            const float sc = warp_sum(acc1) * out_scale;
            const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + r + 1) : (uint32_t)(r + 1);
            const unsigned long long kk = make_key(sc, gid);
            best = kk > best ? kk : best;
        }
    }
    unsigned long long b1[1] = {best};
    finish_argmax<1>(b1, a);
}


// Same as k_gemv_nvfp4_direct with the prescaled f16 hidden row in shared
// memory instead of registers (fewer registers -> more warps and more bytes
// in flight).  Chunk c (64 elements = 8 pieces of 16 bytes) is stored with its
// pieces XOR-swizzled by c % 8, so the 32 lanes of a warp (chunks c .. c+31)
// read a block's two pieces without bank conflicts.
__device__ __forceinline__ void lds128(uint32_t addr, uint32_t* r) {
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// Three CTAs per SM (80 registers): at four the compiler has 64 registers and
// spills the two rows' code words, which cost ~14% of the kernel's time.
__global__ void __launch_bounds__(kThreads, 3) k_gemv_nvfp4_xs(const GemvArgs a) {
    extern __shared__ __align__(16) uint32_t xsh[];  // [nch][8 pieces][4 words], swizzled
    __shared__ float s_xmax[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = a.H, nch = H >> 6;
    const size_t qrow = (size_t)H / 2, srow = (size_t)H / 16;
    const uint8_t* __restrict__ Wq = static_cast<const uint8_t*>(a.W);

    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const long long r0 = gw * a.rows_per_warp;
    const long long r1 = min(r0 + (long long)a.rows_per_warp, (long long)a.n_rows);

    pdl_launch_dependents();
    for (long long r = r0; r < min(r1, r0 + 2); ++r)
        for (int c = lane; c < nch; c += 32) prefetch_l2(Wq + (size_t)r * qrow + c * 32);
    pdl_wait();

    // largest |x| over 16-byte pieces (H / 8 of them, one or two per thread)
    float m = 0.f;
    const uint4* xv = reinterpret_cast<const uint4*>(a.x);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) {
        const uint4 v = __ldg(xv + i);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf_lo(v.x)), fabsf(bf_hi(v.x))), fmaxf(fabsf(bf_lo(v.y)), fabsf(bf_hi(v.y)))));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf_lo(v.z)), fabsf(bf_hi(v.z))), fmaxf(fabsf(bf_lo(v.w)), fabsf(bf_hi(v.w)))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) s_xmax[warp] = m;
    __syncthreads();
    float xmax = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) xmax = fmaxf(xmax, s_xmax[w]);
    const int k = xmax > 0.f ? min(127, 141 - (int)((__float_as_uint(xmax) >> 23) & 0xFF)) : 0;
    const float up = ldexpf(1.f, k), out_scale = a.g * ldexpf(1.f, -k);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) {  // piece i = elements 8i .. 8i+7
        const uint4 v = __ldg(xv + i);
        const int c = i >> 3, piece = i & 7;
        uint4 h;
        h.x = f32x2_to_h2(bf_lo(v.x) * up, bf_hi(v.x) * up);
        h.y = f32x2_to_h2(bf_lo(v.y) * up, bf_hi(v.y) * up);
        h.z = f32x2_to_h2(bf_lo(v.z) * up, bf_hi(v.z) * up);
        h.w = f32x2_to_h2(bf_lo(v.w) * up, bf_hi(v.w) * up);
        *reinterpret_cast<uint4*>(xsh + c * 32 + ((piece ^ (c & 7)) << 2)) = h;
    }
    __syncthreads();
    const uint32_t xbase = ptx::smem_u32(xsh);

    unsigned long long best = 0ull;
    for (long long r = r0; r < r1 && vh_guard(r1 <= a.n_rows, a.err); r += 2) {
        const bool two = (r + 1 < r1);
        U32x8 q0[2], q1[2];
        uint32_t s0[2], s1[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = lane + 32 * j;
            if (c < nch) {
                q0[j] = ld_stream32(Wq + (size_t)r * qrow + c * 32);
                s0[j] = __ldg(reinterpret_cast<const uint32_t*>(a.scales + (size_t)r * srow) + c);
                if (two) {
                    q1[j] = ld_stream32(Wq + (size_t)(r + 1) * qrow + c * 32);
                    s1[j] = __ldg(reinterpret_cast<const uint32_t*>(a.scales + (size_t)(r + 1) * srow) + c);
                }
            }
        }
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // H <= 4096: at most two 64-element chunks per lane
            const int c = lane + 32 * j;
            if (c < nch) {
                const float2 a01 = e4m3x2_to_f2(s0[j] & 0xFFFFu), a23 = e4m3x2_to_f2(s0[j] >> 16);
                const float2 b01 = two ? e4m3x2_to_f2(s1[j] & 0xFFFFu) : make_float2(0.f, 0.f);
                const float2 b23 = two ? e4m3x2_to_f2(s1[j] >> 16) : make_float2(0.f, 0.f);
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    uint32_t xv[8];
                    lds128(xbase + (uint32_t)(c * 128 + (((2 * blk) ^ (c & 7)) << 4)), xv);
                    lds128(xbase + (uint32_t)(c * 128 + (((2 * blk + 1) ^ (c & 7)) << 4)), xv + 4);
                    const float sa = blk == 0 ? a01.x : blk == 1 ? a01.y : blk == 2 ? a23.x : a23.y;
                    acc0 = fmaf(nvfp4_block16(q0[j].v[2 * blk], q0[j].v[2 * blk + 1], xv), sa, acc0);
                    if (two) {
                        const float sb = blk == 0 ? b01.x : blk == 1 ? b01.y : blk == 2 ? b23.x : b23.y;
                        acc1 = fmaf(nvfp4_block16(q1[j].v[2 * blk], q1[j].v[2 * blk + 1], xv), sb, acc1);
                    }
                }
            }
        }
        {
            const float sc = warp_sum(acc0) * out_scale;
            const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + r) : (uint32_t)r;
            const unsigned long long kk = make_key(sc, gid);
            best = kk > best ? kk : best;
        }
        if (two) {
            const float sc = warp_sum(acc1) * out_scale;
            const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + r + 1) : (uint32_t)(r + 1);
            const unsigned long long kk = make_key(sc, gid);
            best = kk > best ? kk : best;
        }
    }
    unsigned long long b1[1] = {best};
    finish_argmax<1>(b1, a);
}

// ---------------------------------------------------------------------------
// Block-scaled 4-bit head on CUDA cores, any B <= 8.  A lane chunk is 32 code
// bytes = 64 elements = 4 scale blocks.  Each 16-element block is summed
// unscaled, then multiplied by its E4M3 scale; g multiplies the total.

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

// Per-device launch facts, looked up once (device ordinals below kMaxDev).
constexpr int kMaxDev = 64;

int sm_count() {
    static std::atomic<int> cache[kMaxDev] = {};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDev) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDev) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Resident CTAs per SM of `kernel` at `smem` bytes of dynamic shared memory on
// the current device, queried once per (kernel, smem, device).
static cudaError_t occupancy(const void* kernel, size_t smem, int& per_sm) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, size_t, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const auto key = std::make_tuple(kernel, smem, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        const auto it = cache.find(key);
        if (it != cache.end()) {
            per_sm = it->second;
            return cudaSuccess;
        }
    }
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = per_sm;
    return cudaSuccess;
}

template <typename K>
static cudaError_t launch_split_v(K kernel, size_t smem, int n_rows, GemvArgs& a, cudaStream_t s, bool pdl,
                                  bool even_rows = false) {
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    cudaError_t oe = occupancy(reinterpret_cast<const void*>(kernel), smem, per_sm);
    if (oe != cudaSuccess) return oe;
    const int sms = sm_count();
    if (per_sm < 1 || sms < 1) return cudaErrorInvalidConfiguration;
    // one resident wave; each warp gets a contiguous share of rows: with
    // even_rows the kernel splits n_rows over all grid * kWarps warps (shares
    // differ by at most one row), else every warp takes rows_per_warp rows
    // and the grid shrinks to the warps needed
    long long grid = (long long)sms * per_sm;
    const long long min_rows_per_warp = 2;
    const long long max_grid = ((long long)n_rows + kWarps * min_rows_per_warp - 1) / (kWarps * min_rows_per_warp);
    grid = std::max(1LL, std::min(grid, max_grid));
    const long long warps = grid * kWarps;
    a.rows_per_warp = (int)(((long long)n_rows + warps - 1) / warps);
    if (!even_rows)
        grid = ((long long)n_rows + (long long)a.rows_per_warp * kWarps - 1) / ((long long)a.rows_per_warp * kWarps);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

cudaError_t launch_gemv_bf16(const uint16_t* x, int nb, int H, const uint16_t* W, const int32_t* cand, int n_rows,
                             Workspace ws, int32_t* ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s,
                             int gather_V) {
    GemvArgs a{};
    a.x = x; a.W = W; a.scales = nullptr; a.g = 1.f; a.cand = cand;
    a.gather = gather_V > 0 ? 1 : 0;
    a.V = gather_V;
    a.nb = nb; a.H = H; a.n_rows = n_rows; a.ws = ws; a.ids = ids; a.maxlogit = maxlogit; a.tail = tail;
    a.err = ws.ticket + 1;
    if (nb == 1)
        return a.gather ? launch_split_v(k_gemv_bf16<1, 1, true>, (size_t)H * 2, n_rows, a, s, true, true)
                        : launch_split_v(k_gemv_bf16<1, 1, false>, (size_t)H * 2, n_rows, a, s, true, true);
#define VH_GEMV_CASE(NBV)                                                                                          \
    if (nb <= NBV)                                                                                                 \
        return a.gather ? launch_split_v(k_gemv_bf16<NBV, 2, true>, (size_t)NBV * H * 2, n_rows, a, s, true, true) \
                        : launch_split_v(k_gemv_bf16<NBV, 2, false>, (size_t)NBV * H * 2, n_rows, a, s, true, true);
    VH_GEMV_CASE(2)
    VH_GEMV_CASE(4)
    VH_GEMV_CASE(8)
#undef VH_GEMV_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemv_nvfp4(const uint16_t* x, int nb, int H, const uint8_t* Wq, const uint8_t* scales, float g,
                              const int32_t* cand, int n_rows, Workspace ws, int32_t* ids, float* maxlogit,
                              cudaStream_t s, const AcceptTail& tail) {
    GemvArgs a{};
    a.x = x; a.W = Wq; a.scales = scales; a.g = g; a.cand = cand;
    a.nb = nb; a.H = H; a.n_rows = n_rows; a.ws = ws; a.ids = ids; a.maxlogit = maxlogit; a.tail = tail;
    a.err = ws.ticket + 1;
    if (nb == 1 && H <= 4096) return launch_split_v(k_gemv_nvfp4_xs, (size_t)H * 2, n_rows, a, s, true);
    if (nb == 1 && H <= 8192) {
        const int cpl = (H / 64 + 31) / 32;
        if (cpl <= 1) return launch_split_v(k_gemv_nvfp4_direct<1>, 0, n_rows, a, s, true);
        if (cpl <= 2) return launch_split_v(k_gemv_nvfp4_direct<2>, 0, n_rows, a, s, true);
        return launch_split_v(k_gemv_nvfp4_direct<4>, 0, n_rows, a, s, true);
    }
#define VH_NVFP4_CASE(NBV) \
    if (nb <= NBV) return launch_split_v(k_gemv_nvfp4<NBV>, (size_t)NBV * H * 2, n_rows, a, s, false);
    VH_NVFP4_CASE(1)
    VH_NVFP4_CASE(2)
    VH_NVFP4_CASE(4)
    VH_NVFP4_CASE(8)
#undef VH_NVFP4_CASE
    return cudaErrorInvalidValue;
}

}  // namespace vh
