// Block-scaled 4-bit head for up to 8 hidden rows on warp-level tensor-core
// MMAs (mma.sync m16n8k16, f16 operands, fp32 accumulation) fed straight
// from registers, fused with the argmax and the candidate-id mapping.
//
// Format (NVFP4 weights, "为什么生产推理我默认 vLLM" §3; NVFP4 candidate rows in
// "少读一张大表，草稿路径才真正快起来"): E2M1 codes, element 2i in the low nibble,
// one E4M3 scale per 16 elements along H, one fp32 tensor scale g.
//
// Why warp-level MMAs: with at most 8 hidden rows the contraction is a few
// flops per weight and the tensor pipe idles on any design; the cost is
// turning codes into f16 operands and getting them to the tensor core.  Here
// a warp loads its own codes, decodes them into A fragments in registers and
// issues the MMA itself: no decoded tile goes through shared memory or TMEM
// and no other warp waits for it.
//
// Exactness: every E2M1 x E4M3 product has at most 6 significant bits and
// lies in [2^-10, 2688], so the decoded weight is an f16 value.  The hidden
// rows are converted to f16 with a per-row power-of-two prescale 2^k_b
// (largest |x| into [2^14, 2^15)).  The score of hidden row b is
// acc * g * 2^-k_b.
//
// Work layout (one CTA of 16 warps per SM):
//   block   16 weight rows (the MMA's M); each CTA owns a contiguous range.
//   slice   256 elements of K (128 code bytes + 16 scales per row).  With
//           KS = H/256 slices, the CTA's warps form 16/KS groups of KS warps;
//           warp w of a group always takes slice w, so its B fragments (the
//           prescaled hidden rows over that slice) stay in registers for the
//           whole launch.  Groups take alternate blocks of the CTA's range.
//   stream  each warp copies its slice of its next blocks from HBM into a
//           private 4-stage shared-memory ring with cp.async (16-byte pieces,
//           L1 bypassed, 16-byte chunks XOR-swizzled by row so that the
//           fragment reads are bank-conflict free).
//   MMA j   (j = 0..15 within a slice) gives thread (row group r, lane in
//           group g) the physical elements g*64 + 4j + {0,1 | 2,3} for its
//           logical k slots {2g, 2g+1 | 2g+8, 2g+9}, for A and B alike: the
//           sum is over the same products, and a thread's codes for a slice
//           are 32 contiguous bytes per row.
//   merge   K-slice partials (16 x 8 fp32 per warp) meet in an 8-slot shared
//           ring; one warp per block (rotating through the group) adds them
//           in slice order, takes the per-column argmax over the block's rows
//           (lowest row on ties) and folds it into its running best.  Running
//           bests leave the CTA as packed-key atomicMax; the last CTA decodes.
// Waits on the ring barriers are bounded (see vh_ptx.cuh).
#include <algorithm>
#include <climits>

#include "vh_kernels.h"
#include "vh_ptx.cuh"

namespace vh {
namespace fp4mma {

using namespace ptx;

constexpr int kWarpsM = 16;
constexpr int kThreadsM = kWarpsM * 32;
constexpr int kSlice = 256;                   // K elements per warp slice
constexpr int kSliceCodes = kSlice / 2;       // 128 code bytes per row
constexpr int kSliceScales = kSlice / 16;     // 16 scale bytes per row
constexpr int kBlkRows = 16;                  // weight rows per block (MMA M)
constexpr int kN = 8;                         // hidden rows (MMA N)
constexpr int kStages = 4;                    // cp.async ring depth per warp
constexpr int kStageBytes = kBlkRows * (kSliceCodes + kSliceScales);  // 2,304
constexpr int kSlots = 8;                     // partial-sum ring depth per group
constexpr size_t kRingBytes = (size_t)kWarpsM * kStages * kStageBytes;     // 147,456
constexpr size_t kPartBytes = (size_t)kSlots * kWarpsM * 32 * 16;          // 65,536
constexpr size_t kSmem = kRingBytes + kPartBytes;

struct Args {
    const uint16_t* x;  // bf16 [nb][H]
    const uint8_t* q;   // codes [Vc][H/2]
    const uint8_t* sc;  // E4M3 scales [Vc][H/16]
    const int32_t* cand;
    int nb, H, Vc, n_blk;
    float g;
    Workspace ws;
    unsigned int* err;
    int32_t* ids;
    float* maxlogit;
    AcceptTail tail;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, unsigned long long pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// Four E2M1 pairs (the bytes of `w`, low byte first) -> four f16x2 words.
__device__ __forceinline__ void e2m1x8_h2(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}

// Two E4M3 scales (low 16 bits, low byte first) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_h2(uint32_t two) {
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(two));
    return h2;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t f32x2_h2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}

// D += A (16 x 16, rows r / r+8) * B (16 x 8), f16 in, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// cp.async of one block's slice into a ring stage: codes [16 rows][128 B]
// with 16-byte chunk c of row r at chunk c ^ (r & 7), then scales [16][16 B].
// Rows past Vc repeat row Vc - 1 (their scores are masked).
__device__ __forceinline__ void issue_block(const Args& a, int blk, int wk, int lane, uint32_t stage,
                                            unsigned long long pol) {
    const int row0 = blk * kBlkRows;
    const size_t qrow = (size_t)a.H / 2, srow = (size_t)a.H / 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = (lane >> 3) + 4 * i, c = lane & 7;
        const int row = min(row0 + r, a.Vc - 1);
        cp_async16(stage + (uint32_t)(r * kSliceCodes + ((c ^ (r & 7)) << 4)),
                   a.q + (size_t)row * qrow + (size_t)wk * kSliceCodes + c * 16, pol);
    }
    if (lane < kBlkRows) {
        const int row = min(row0 + lane, a.Vc - 1);
        cp_async16(stage + (uint32_t)(kBlkRows * kSliceCodes + lane * 16),
                   a.sc + (size_t)row * srow + (size_t)wk * kSliceScales, pol);
    }
}

__global__ void __launch_bounds__(kThreadsM, 1) k_nvfp4_mma(const Args a) {
    extern __shared__ __align__(16) uint8_t smem[];
    float4* part = reinterpret_cast<float4*>(smem + kRingBytes);  // [group][slot][slice warp][lane]
    __shared__ unsigned long long bar_full[kWarpsM * kSlots], bar_empty[kWarpsM * kSlots];
    __shared__ unsigned long long merge[kN];
    __shared__ float s_up[kN], s_down[kN];
    __shared__ unsigned int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, KS = H / kSlice, G = kWarpsM / KS;
    const int grp = warp / KS, wk = warp % KS;
    const int g4 = lane & 3, r8 = lane >> 2;
    const int b_lo = (int)((long long)blockIdx.x * a.n_blk / gridDim.x);
    const int b_hi = (int)((long long)(blockIdx.x + 1) * a.n_blk / gridDim.x);
    const int n_t = (b_hi - b_lo - grp + G - 1) / G;  // blocks of this warp's group (may be <= 0)

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < G * kSlots; ++i) {
            mbar_init(&bar_full[i], (uint32_t)KS * 32u);
            mbar_init(&bar_empty[i], 32u);
        }
        fence_barrier_init();
    }
    if (threadIdx.x < kN) merge[threadIdx.x] = 0ull;
    // the first blocks' code lines into L2 while the previous kernel finishes
    if (lane < kBlkRows) {
        for (int p = 0; p < kStages - 1 && p < n_t; ++p) {
            const int row = min((b_lo + grp + p * G) * kBlkRows + lane, a.Vc - 1);
            prefetch_l2(a.q + (size_t)row * (H / 2) + (size_t)wk * kSliceCodes);
        }
    }
    pdl_wait();  // the hidden rows and the workspace may come from the previous kernel

    // per-row power-of-two prescale of the hidden rows (identical in every CTA)
    if (warp < kN) {
        const int b = warp;
        float m = 0.f;
        if (b < a.nb) {
            const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)b * H);
            for (int i = lane; i < H / 8; i += 32) {
                const uint4 v = __ldg(xr + i);
                m = fmaxf(m, fmaxf(fmaxf(fabsf(bf_lo(v.x)), fabsf(bf_hi(v.x))), fmaxf(fabsf(bf_lo(v.y)), fabsf(bf_hi(v.y)))));
                m = fmaxf(m, fmaxf(fmaxf(fabsf(bf_lo(v.z)), fabsf(bf_hi(v.z))), fmaxf(fabsf(bf_lo(v.w)), fabsf(bf_hi(v.w)))));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) {
            int k = 0;
            if (m > 0.f) k = min(127, 141 - (int)((__float_as_uint(m) >> 23) & 0xFF));
            s_up[b] = b < a.nb ? ldexpf(1.f, k) : 0.f;
            s_down[b] = b < a.nb ? a.g * ldexpf(1.f, -k) : 0.f;
        }
    }
    __syncthreads();

    // B fragments of this warp's slice: hidden row r8, elements
    // wk*256 + g4*64 + [0, 64); MMA j takes elements 4j..4j+3
    uint32_t xf[16][2];
    {
        const float up = s_up[r8];  // 0 for rows >= nb
        const uint4* src =
            reinterpret_cast<const uint4*>(a.x + (size_t)min(r8, a.nb - 1) * H + (size_t)wk * kSlice + g4 * 64);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = __ldg(src + i);
            xf[2 * i][0] = f32x2_h2(bf_lo(v.x) * up, bf_hi(v.x) * up);
            xf[2 * i][1] = f32x2_h2(bf_lo(v.y) * up, bf_hi(v.y) * up);
            xf[2 * i + 1][0] = f32x2_h2(bf_lo(v.z) * up, bf_hi(v.z) * up);
            xf[2 * i + 1][1] = f32x2_h2(bf_lo(v.w) * up, bf_hi(v.w) * up);
        }
    }

    const unsigned long long pol = policy_evict_first();
    const uint32_t ring = smem_u32(smem) + (uint32_t)(warp * kStages * kStageBytes);
#pragma unroll
    for (int p = 0; p < kStages - 1; ++p) {
        if (p < n_t) issue_block(a, b_lo + grp + p * G, wk, lane, ring + p * kStageBytes, pol);
        cp_async_commit();
    }

    const float ninf = -__int_as_float(0x7f800000);
    float best_v0 = ninf, best_v1 = ninf;  // columns 2*g4, 2*g4+1 (valid in lanes 0..3)
    int best_r0 = -1, best_r1 = -1;
    bool ok = true;
    for (int t = 0; t < n_t && ok; ++t) {
        const int pn = t + kStages - 1;
        if (pn < n_t) issue_block(a, b_lo + grp + pn * G, wk, lane, ring + (pn % kStages) * kStageBytes, pol);
        cp_async_commit();
        cp_async_wait<kStages - 1>();  // block t's copies (this lane's) have landed
        __syncwarp();                  // ... and every other lane's

        const uint32_t st = ring + (uint32_t)((t % kStages) * kStageBytes);
        const uint32_t ra_off = st + (uint32_t)(r8 * kSliceCodes), rb_off = ra_off + 8u * kSliceCodes;
        const uint32_t c0 = (uint32_t)(((2 * g4) ^ r8) << 4), c1 = (uint32_t)(((2 * g4 + 1) ^ r8) << 4);
        const uint4 qa0 = lds128(ra_off + c0), qa1 = lds128(ra_off + c1);
        const uint4 qb0 = lds128(rb_off + c0), qb1 = lds128(rb_off + c1);
        const uint32_t sa = lds32(st + (uint32_t)(kBlkRows * kSliceCodes + r8 * 16 + g4 * 4));
        const uint32_t sb = lds32(st + (uint32_t)(kBlkRows * kSliceCodes + (r8 + 8) * 16 + g4 * 4));
        __syncwarp();  // the stage may be refilled from here on
        const uint32_t qa[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qa1.x, qa1.y, qa1.z, qa1.w};
        const uint32_t qb[8] = {qb0.x, qb0.y, qb0.z, qb0.w, qb1.x, qb1.y, qb1.z, qb1.w};
        // scale of 16-element block q (= MMA j / 4) in both halves of an f16x2
        const uint32_t sa01 = e4m3x2_h2(sa & 0xFFFFu), sa23 = e4m3x2_h2(sa >> 16);
        const uint32_t sb01 = e4m3x2_h2(sb & 0xFFFFu), sb23 = e4m3x2_h2(sb >> 16);
        const uint32_t sA[4] = {__byte_perm(sa01, 0, 0x1010), __byte_perm(sa01, 0, 0x3232),
                                __byte_perm(sa23, 0, 0x1010), __byte_perm(sa23, 0, 0x3232)};
        const uint32_t sB[4] = {__byte_perm(sb01, 0, 0x1010), __byte_perm(sb01, 0, 0x3232),
                                __byte_perm(sb23, 0, 0x1010), __byte_perm(sb23, 0, 0x3232)};
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // code word i holds MMAs 2i (bytes 0, 1) and 2i + 1 (bytes 2, 3)
            uint32_t ha[4], hb[4];
            e2m1x8_h2(qa[i], ha);
            e2m1x8_h2(qb[i], hb);
            const uint32_t s_a = sA[i >> 1], s_b = sB[i >> 1];
            mma16816(acc0, hmul2(ha[0], s_a), hmul2(hb[0], s_b), hmul2(ha[1], s_a), hmul2(hb[1], s_b), xf[2 * i][0],
                     xf[2 * i][1]);
            mma16816(acc1, hmul2(ha[2], s_a), hmul2(hb[2], s_b), hmul2(ha[3], s_a), hmul2(hb[3], s_b),
                     xf[2 * i + 1][0], xf[2 * i + 1][1]);
        }

        // partial of this slice -> ring slot; the block's reducer adds the slices
        const int slot = t % kSlots;
        const uint32_t ph = (uint32_t)(t / kSlots) & 1u;
        const int bi = grp * kSlots + slot;
        if (!mbar_wait(&bar_empty[bi], ph ^ 1u, a.err)) { ok = false; break; }
        part[(bi * KS + wk) * 32 + lane] =
            make_float4(acc0[0] + acc1[0], acc0[1] + acc1[1], acc0[2] + acc1[2], acc0[3] + acc1[3]);
        mbar_arrive(&bar_full[bi]);
        if (t % KS != wk) continue;
        if (!mbar_wait(&bar_full[bi], ph, a.err)) { ok = false; break; }
        float4 s = part[(bi * KS) * 32 + lane];
        for (int w = 1; w < KS; ++w) {
            const float4 p = part[(bi * KS + w) * 32 + lane];
            s.x += p.x;
            s.y += p.y;
            s.z += p.z;
            s.w += p.w;
        }
        mbar_arrive(&bar_empty[bi]);
        // per-column argmax over the block's 16 rows (lowest row on ties):
        // s.x / s.y = row r8, columns 2*g4 / 2*g4+1; s.z / s.w = row r8 + 8
        const int ra = (b_lo + grp + t * G) * kBlkRows + r8, rb = ra + 8;
        const float d0 = s_down[2 * g4], d1 = s_down[2 * g4 + 1];
        float v0 = ra < a.Vc ? s.x * d0 : ninf, v1 = ra < a.Vc ? s.y * d1 : ninf;
        float v2 = rb < a.Vc ? s.z * d0 : ninf, v3 = rb < a.Vc ? s.w * d1 : ninf;
        v0 = v0 != v0 ? ninf : v0;
        v1 = v1 != v1 ? ninf : v1;
        v2 = v2 != v2 ? ninf : v2;
        v3 = v3 != v3 ? ninf : v3;
        float bv0 = v0, bv1 = v1;
        int br0 = ra, br1 = ra;
        if (v2 > bv0) { bv0 = v2; br0 = rb; }
        if (v3 > bv1) { bv1 = v3; br1 = rb; }
#pragma unroll
        for (int m = 4; m <= 16; m <<= 1) {  // across the 8 row groups
            const float o0 = __shfl_xor_sync(0xFFFFFFFFu, bv0, m), o1 = __shfl_xor_sync(0xFFFFFFFFu, bv1, m);
            const int p0 = __shfl_xor_sync(0xFFFFFFFFu, br0, m), p1 = __shfl_xor_sync(0xFFFFFFFFu, br1, m);
            if (o0 > bv0 || (o0 == bv0 && p0 < br0)) { bv0 = o0; br0 = p0; }
            if (o1 > bv1 || (o1 == bv1 && p1 < br1)) { bv1 = o1; br1 = p1; }
        }
        // blocks come in increasing row order: an equal score keeps the earlier row
        if (best_r0 < 0 || bv0 > best_v0) { best_v0 = bv0; best_r0 = br0; }
        if (best_r1 < 0 || bv1 > best_v1) { best_v1 = bv1; best_r1 = br1; }
    }
    cp_async_wait<0>();

    // ---------------- CTA merge, publish, last-CTA decode ----------------
    if (r8 == 0) {  // lanes 0..3: columns 2*lane, 2*lane + 1
        const int col0 = 2 * g4, col1 = col0 + 1;
        if (best_r0 >= 0 && col0 < a.nb && vh_guard(best_r0 < a.Vc, a.err)) {
            const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + best_r0) : (uint32_t)best_r0;
            atomicMax(&merge[col0], make_key(best_v0, gid));
        }
        if (best_r1 >= 0 && col1 < a.nb && vh_guard(best_r1 < a.Vc, a.err)) {
            const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + best_r1) : (uint32_t)best_r1;
            atomicMax(&merge[col1], make_key(best_v1, gid));
        }
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

}  // namespace fp4mma

bool nvfp4_mma_supported(int nb, int H) {
    const int ks = H / fp4mma::kSlice;
    return nb >= 1 && nb <= fp4mma::kN && H % fp4mma::kSlice == 0 && ks >= 1 && ks <= fp4mma::kWarpsM &&
           (ks & (ks - 1)) == 0;
}

cudaError_t launch_nvfp4_mma(const uint16_t* x, int nb, int H, const uint8_t* Wq, const uint8_t* scales, float g,
                             const int32_t* cand, int Vc, Workspace ws, int32_t* ids, float* maxlogit, cudaStream_t s,
                             const AcceptTail& tail) {
    using namespace fp4mma;
    if (!nvfp4_mma_supported(nb, H) || Vc < 1 || Vc > INT_MAX - kBlkRows) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(k_nvfp4_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    Args a{};
    a.x = x;
    a.q = Wq;
    a.sc = scales;
    a.cand = cand;
    a.nb = nb;
    a.H = H;
    a.Vc = Vc;
    a.n_blk = (Vc + kBlkRows - 1) / kBlkRows;
    a.g = g;
    a.ws = ws;
    a.err = ws.ticket + 1;
    a.ids = ids;
    a.maxlogit = maxlogit;
    a.tail = tail;
    const int grid = std::max(1, std::min(sm_count(), a.n_blk));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreadsM);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_nvfp4_mma, a);
}

}  // namespace vh
