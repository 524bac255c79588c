// bf16 head scored for 1-8 hidden rows on warp-level tensor-core MMAs fed
// straight from the weight stream, fused with the argmax, the candidate-id
// mapping and (for verify) the acceptance scan.  Serves the draft head
// ("少读一张大表，草稿路径才真正快起来": a candidate table, the winning
// candidate's global id) for small batches and the batch-1 MTP verify rows
// (the target scores k+1 rows against the full head).
//
// MMA roles.  mma.m16n8k16 with A = the hidden rows (M = 16: up to 8 real
// rows with the upper 8 zero, or up to 16 in the 16-row instance), B = 8 head
// rows (N = 8), fp32 accumulation.
// Lane L (g = L/4, t = L%4) supplies B for head row g of the group, so a warp
// streams 8 head rows at once, STEP contiguous elements of each per step: load
// i (i < STEP/64) of lane t reads the row's bytes 128i + 32t .. +31, so the
// four lanes of a row read one whole 128-byte line per instruction.  A step is
// 256 elements (512 bytes of each row, two steps in flight per warp) or 512
// elements (1 KiB of each row, one step in flight).
//
// K order.  Within a step, MMA j = 4i + m (i < STEP/64, m = 0..3) gives lane
// (g, t) the physical elements 64i + 16t + 4m + {0,1} for its K slots {2t,
// 2t+1} and 64i + 16t + 4m + {2,3} for {2t+8, 2t+9}, on A and B alike: each
// MMA sums the same products as the plain order, and a lane's B registers for
// MMA j are registers 2m and 2m+1 of its load i.  The hidden rows sit in
// shared memory in that fragment order: lane L's 8 bytes for (step s, MMA j)
// are row g's elements STEP*s + 64i + 16t + 4m .. +3, and a warp reads 256
// consecutive bytes per MMA.  The 16-row instance also holds hidden row g+8's
// 4 elements: 16 bytes per lane per MMA, {row g, row g+8, row g, row g+8} as
// the A registers a0..a3 want them, 512 consecutive bytes per warp.
//
// Output.  Accumulator registers c0 / c1 of lane (g, t) are hidden row g's
// scores of head rows 2t and 2t+1 of the group; c2 / c3 are hidden row g+8's
// (zero rows in the 8-row instance).  Each lane keeps one packed (score, id)
// key per hidden row it holds; the four lanes of a row, the warps of a CTA
// and the CTAs merge by max, and the
// last CTA (ticket counter) writes ids / max logits, runs the optional
// acceptance scan and re-zeroes the workspace.
//
// Work split.  Each CTA owns whole 8-row groups; inside a CTA the (group,
// step) units are split evenly over the warps, and a group cut between two
// warps is summed in shared memory in warp order (with one step per group,
// no group is ever cut: a row then scores the same bits wherever it sits).
#include <algorithm>
#include <climits>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "vh_kernels.h"
#include "vh_ptx.cuh"

namespace vh {
namespace gmma {

constexpr int kWarpsG = 8;
constexpr int kThreadsG = kWarpsG * 32;
constexpr int kStepK = 256;   // elements of K per step, short steps (512 bytes of each head row)
constexpr int kStepLong = 512;  // long steps (1 KiB of each head row), single-buffered
constexpr int kRowsG = 8;     // head rows per warp group (MMA N)
constexpr int kMaxRows = 16;  // hidden rows per launch (the 16-row instance)

struct Args {
    const uint16_t* x;  // bf16 [nb][H]
    const uint16_t* W;  // bf16 [n_rows][H]
    const int32_t* cand;
    int nb, H, n_rows, n_groups;
    Workspace ws;
    unsigned int* err;
    int32_t* ids;
    float* maxlogit;
    AcceptTail tail;
};

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// D += A (16 x 16 bf16: a0 / a2 row g, a1 / a3 row g+8) * B (16 x 8 bf16), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int STEP>
struct Seg {  // this lane's part of one head row's step: elements 64i + 16t .. +15, i < STEP/64
    U32x8 v[STEP / 64];
};

template <int STEP>
__device__ __forceinline__ void load_seg(Seg<STEP>& s, const uint16_t* p) {  // p: the step's element 16t of the row
#pragma unroll
    for (int i = 0; i < STEP / 64; ++i) s.v[i] = ld_stream32(p + i * 64);
}

// The STEP/16 MMAs of one step: B from the lane's registers, A from shared
// memory (8 bytes per lane per MMA with NR = 8 hidden rows, 16 with NR = 16).
template <int STEP, int NR>
__device__ __forceinline__ void step_mma(const Seg<STEP>& w, uint32_t afrag, float (&c0)[4], float (&c1)[4]) {
#pragma unroll
    for (int j = 0; j < STEP / 16; ++j) {
        const uint32_t b0 = w.v[j >> 2].v[2 * (j & 3)], b1 = w.v[j >> 2].v[2 * (j & 3) + 1];
        if constexpr (NR == 8) {
            const uint2 a = lds64(afrag + (uint32_t)(j * 256));
            mma_bf16_16816((j & 1) ? c1 : c0, a.x, 0u, a.y, 0u, b0, b1);
        } else {
            const uint4 a = lds128(afrag + (uint32_t)(j * 512));
            mma_bf16_16816((j & 1) ? c1 : c0, a.x, a.y, a.z, a.w, b0, b1);
        }
    }
}

// STEP: K elements per step (256 or 512); NBUF: steps in registers per warp (2 or 1);
// NR: hidden rows the instance holds (8 or 16).
template <int STEP, int NBUF, int NR>
__global__ void __launch_bounds__(kThreadsG, 2) k_gemv_mma_bf16(const Args a) {
    constexpr int kMmaStep = STEP / 16;                  // MMAs per step
    constexpr int kFragB = NR == 16 ? 16 : 8;            // bytes per lane per MMA
    constexpr int KB = NR == 16 ? 2 : 1;                 // keys (hidden rows) per lane
    extern __shared__ __align__(16) uint8_t xfrag[];  // [H/STEP steps][STEP/16 MMAs][32 lanes][kFragB B]
    using Cut = std::conditional_t<NR == 16, float4, float2>;
    __shared__ Cut cut[kWarpsG][2][32];                // partial scores of groups cut between warps
    __shared__ unsigned long long merge[kMaxRows];
    __shared__ unsigned int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int H = a.H, n_steps = H / STEP;

    // CTA c owns the 8-row groups [G0, G1); its (group, step) units are split
    // evenly into contiguous ranges, one per warp.  A group cut by a range
    // boundary is finished after all warps are done: each warp leaves its
    // partial scores of its first and last group in shared memory and the
    // warp that holds the group's first step adds the pieces in warp order.
    const int G0 = (int)((long long)blockIdx.x * a.n_groups / gridDim.x);
    const int G1 = (int)((long long)(blockIdx.x + 1) * a.n_groups / gridDim.x);
    const int CU = (G1 - G0) * n_steps;
    auto u_begin = [&](int w) { return (int)((long long)w * CU / kWarpsG); };
    const int v_lo = u_begin(warp), v_hi = u_begin(warp + 1);

    auto unit_ptr = [&](int v) -> const uint16_t* {  // this lane's 64 elements of unit v
        const int r = (G0 + v / n_steps) * kRowsG + g;
        return a.W + (size_t)(r < a.n_rows ? r : 0) * H + (size_t)(v % n_steps) * STEP + (size_t)t * 16;
    };
    // the 128-byte lines of a group's eight rows head for L2 (lane L: row L/4, lines L%4, L%4 + 4, ...).
    // Done once, for the warp's first group, while the kernel waits for the previous one; prefetching
    // the next group from inside the loop competed with the demand loads (0.74 against 0.91 of HBM on
    // the 248,320-row head).
    auto prefetch_group = [&](int grp) {
        const int r = (G0 + grp) * kRowsG + g;
        if (r < a.n_rows)
            for (int c = t * 64; c < H; c += 256) prefetch_l2(a.W + (size_t)r * H + c);
    };
    // keys of one finished group (this lane: hidden rows g and, with NR = 16, g+8; head rows 2t and 2t+1)
    unsigned long long best[KB];
#pragma unroll
    for (int q = 0; q < KB; ++q) best[q] = 0ull;
    auto finish_group = [&](int grp, float4 s) {
        if (g >= a.nb) return;  // (then g + 8 >= nb too)
        const int r0 = (G0 + grp) * kRowsG + 2 * t;
        const float sc[2][2] = {{s.x, s.y}, {s.z, s.w}};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = r0 + h;
            if (r < a.n_rows) {
                const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + r) : (uint32_t)r;
#pragma unroll
                for (int q = 0; q < KB; ++q)
                    if (g + 8 * q < a.nb) {
                        const unsigned long long k = make_key(sc[q][h], gid);
                        best[q] = k > best[q] ? k : best[q];
                    }
            }
        }
    };

    pdl_launch_dependents();
    if (v_lo < v_hi) prefetch_group(v_lo / n_steps);  // the head never changes: before the dependency wait
    if (threadIdx.x < kMaxRows) merge[threadIdx.x] = 0ull;
    pdl_wait();  // the hidden rows and the workspace may come from the previous kernel

    // hidden rows -> fragment order (rows >= nb are zero)
    for (int e = threadIdx.x; e < n_steps * kMmaStep * 32; e += blockDim.x) {
        const int L = e & 31, j = (e >> 5) % kMmaStep, st = (e >> 5) / kMmaStep;
        const int gg = L >> 2, tt = L & 3;
        const size_t off = (size_t)st * STEP + (j >> 2) * 64 + tt * 16 + (j & 3) * 4;
        uint2 v = make_uint2(0u, 0u);
        if (gg < a.nb) v = *reinterpret_cast<const uint2*>(a.x + (size_t)gg * H + off);
        if constexpr (NR == 8) {
            reinterpret_cast<uint2*>(xfrag)[e] = v;
        } else {
            uint2 u = make_uint2(0u, 0u);
            if (gg + 8 < a.nb) u = *reinterpret_cast<const uint2*>(a.x + (size_t)(gg + 8) * H + off);
            reinterpret_cast<uint4*>(xfrag)[e] = make_uint4(v.x, u.x, v.y, u.y);
        }
    }
    __syncthreads();

    const uint32_t afrag0 = ptx::smem_u32(xfrag) + (uint32_t)lane * (uint32_t)kFragB;
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    bool first = true;
    const bool starts_cut = v_lo % n_steps != 0;
    Seg<STEP> w[NBUF];
    if (NBUF == 2 && v_lo < v_hi) load_seg<STEP>(w[0], unit_ptr(v_lo));
    for (int v0 = v_lo; v0 < v_hi; v0 += NBUF) {
#pragma unroll
        for (int d = 0; d < NBUF; ++d) {
            const int v = v0 + d;
            if (v < v_hi) {
                if (NBUF == 1)
                    load_seg<STEP>(w[0], unit_ptr(v));  // one step at a time: the other warps cover its latency
                else if (v + 1 < v_hi)
                    load_seg<STEP>(w[d ^ 1], unit_ptr(v + 1));
                const int grp = v / n_steps, st = v % n_steps;
                step_mma<STEP, NR>(w[d], afrag0 + (uint32_t)(st * kMmaStep * 32 * kFragB), c0, c1);
                const bool grp_end = st + 1 == n_steps, range_end = v + 1 == v_hi;
                if (grp_end || range_end) {
                    const float4 sg = make_float4(c0[0] + c1[0], c0[1] + c1[1], c0[2] + c1[2], c0[3] + c1[3]);
                    if (!(first && starts_cut) && grp_end)
                        finish_group(grp, sg);
                    else if constexpr (NR == 16)  // a piece of a cut group: slot 0 = this warp's first group, 1 = its last
                        cut[warp][first ? 0 : 1][lane] = sg;
                    else
                        cut[warp][first ? 0 : 1][lane] = make_float2(sg.x, sg.y);
#pragma unroll
                    for (int i = 0; i < 4; ++i) c0[i] = c1[i] = 0.f;
                    first = false;
                }
            }
        }
    }
    __syncthreads();
    // finish the cut group that starts in this warp's range (its last group, cut at the range end)
    if (v_lo < v_hi && v_hi % n_steps != 0) {
        const int jg = (v_hi - 1) / n_steps;  // CTA-local group
        if (jg * n_steps >= v_lo) {          // its first step is ours: add the pieces in warp order
            float4 sg = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int ww = warp; ww < kWarpsG; ++ww) {
                const int wl = u_begin(ww), wh = u_begin(ww + 1);
                if (wl >= (jg + 1) * n_steps) break;
                if (wh <= wl) continue;  // a warp without units
                const Cut p = cut[ww][(wl / n_steps == jg) ? 0 : 1][lane];
                sg.x += p.x;
                sg.y += p.y;
                if constexpr (NR == 16) {
                    sg.z += p.z;
                    sg.w += p.w;
                }
            }
            finish_group(jg, sg);
        }
    }

    // the four lanes of a hidden row, then the warps, then the CTAs
#pragma unroll
    for (int q = 0; q < KB; ++q) {
#pragma unroll
        for (int m = 1; m <= 2; m <<= 1) {
            const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best[q], m);
            best[q] = o > best[q] ? o : best[q];
        }
        if (t == 0 && g + 8 * q < a.nb && best[q] != 0ull) atomicMax(&merge[g + 8 * q], best[q]);
    }
    __syncthreads();
    if (threadIdx.x < a.nb && merge[threadIdx.x] != 0ull) atomicMax(a.ws.keys + threadIdx.x, merge[threadIdx.x]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(a.ws.ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x < a.nb) {
        const unsigned long long k = atomicExch(a.ws.keys + threadIdx.x, 0ull);
        vh_guard(k != 0ull, a.err);  // every hidden row has a winner
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

template <int STEP, int NBUF, int NR>
static cudaError_t launch_steps(const Args& a, cudaStream_t s) {
    auto kernel = k_gemv_mma_bf16<STEP, NBUF, NR>;
    const size_t smem = (size_t)a.H * (NR == 16 ? 32 : 16);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    static std::mutex mu;
    static std::map<std::tuple<size_t, int>, int> cache;  // (shared memory, device) -> resident CTAs per SM
    int dev = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        const auto key = std::make_tuple(smem, dev);
        const auto it = cache.find(key);
        if (it != cache.end()) {
            per_sm = it->second;
        } else {
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreadsG, smem);
            if (e != cudaSuccess) return e;
            cache[key] = per_sm;
        }
    }
    if (per_sm < 1) return cudaErrorNotSupported;
    // one resident wave, at least one 8-row group per CTA
    const long long grid = std::max(1LL, std::min((long long)sm_count() * per_sm, (long long)a.n_groups));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreadsG);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace gmma

bool gemv_mma_supported(int nb, int H) {  // 1-16 hidden rows, H % 256 == 0, hidden rows fit shared memory
    return nb >= 1 && nb <= gmma::kMaxRows && H >= gmma::kStepK && H % gmma::kStepK == 0 &&
           (size_t)H * (nb > 8 ? 32 : 16) <= 160 * 1024;
}

cudaError_t launch_gemv_mma_bf16(const uint16_t* x, int nb, int H, const uint16_t* W, const int32_t* cand, int n_rows,
                                 Workspace ws, int32_t* ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s,
                                 bool long_steps) {
    using namespace gmma;
    if (!gemv_mma_supported(nb, H) || n_rows < 1 || n_rows > INT_MAX - kRowsG) return cudaErrorNotSupported;
    Args a{};
    a.x = x;
    a.W = W;
    a.cand = cand;
    a.nb = nb;
    a.H = H;
    a.n_rows = n_rows;
    a.n_groups = (n_rows + kRowsG - 1) / kRowsG;
    a.ws = ws;
    a.err = ws.ticket + 1;
    a.ids = ids;
    a.maxlogit = maxlogit;
    a.tail = tail;
    const bool l = long_steps && H % kStepLong == 0;
    if (nb > 8) return l ? launch_steps<kStepLong, 1, 16>(a, s) : launch_steps<kStepK, 2, 16>(a, s);
    return l ? launch_steps<kStepLong, 1, 8>(a, s) : launch_steps<kStepK, 2, 8>(a, s);
}

}  // namespace vh

