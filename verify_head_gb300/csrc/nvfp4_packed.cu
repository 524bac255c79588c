// Block-scaled 4-bit head (NVFP4 weights, "为什么生产推理我默认 vLLM" §3; NVFP4
// candidate rows in "少读一张大表，草稿路径才真正快起来") in a tiled layout
// made once from the row-major codes and scales, scored for up to 16 hidden
// rows per pass on warp-level tensor-core MMAs, fused with the argmax, the
// candidate-id mapping and (for verify) the acceptance scan.
//
// Tiled layout.  Head rows are grouped in blocks of 16 (the MMA's M) and K in
// tiles of 256 elements.  Tile (block b, tile t) is one contiguous 2,304-byte
// record at ((b * H/256) + t) * 2304:
//   bytes [h*1024 + L*32, +32), h = 0/1, L = 0..31: the 32 code bytes of row
//     16b + L/4 + 8h, elements 256t + 64*(L%4) + [0, 64) (row-major nibble
//     order: element 2i in the low nibble);
//   bytes [2048 + L*8 + h*4, +4): the 4 E4M3 scales of that row for those 64
//     elements.
// Rows past the head are zero.  A block's tiles follow each other, so a block
// is 9*H contiguous bytes and the whole table is read front to back.
//
// Why: lane L of a warp is exactly the MMA thread (row group L/4, k group L%4)
// whose A fragments these bytes are, so a warp streams a tile with two
// 256-bit loads and one 64-bit load per lane (each warp instruction reads 1 KiB
// of consecutive bytes) straight into the registers it decodes: no shared
// memory staging of the codes, and each warp accumulates its own blocks over
// all of K, so no partial sums move between warps.  The hidden rows (the MMA's
// B operand, f16 under a per-row power-of-two prescale) sit in shared memory
// in fragment order: a warp's B fragment for one MMA is 256 consecutive bytes.
//
// MMA j (j = 0..15) of tile t gives thread (row group r, k group g) the
// physical elements 256t + 64g + 4j + {0,1 | 2,3} for its logical k slots
// {2g, 2g+1 | 2g+8, 2g+9}, for A and B alike: the sum runs over the same
// products.  E2M1 codes decode exactly with cvt.rn.f16x2.e2m1x2 and the E4M3
// scale multiplies exactly in f16 (a product has at most 6 significant bits
// and lies in [2^-10, 2688]); fp32 accumulation; the score of hidden row n is
// acc * g * 2^-k_n.
#include <algorithm>
#include <climits>
#include <map>
#include <mutex>
#include <tuple>

#include "vh_kernels.h"
#include "vh_ptx.cuh"

namespace vh {
namespace fp4p {

constexpr int kWarpsNT1 = 16;    // warps per CTA with one n8 tile (up to 8 hidden rows)
constexpr int kWarpsNT2 = 16;    // warps per CTA with two n8 tiles (9..16 hidden rows)
constexpr int kTileK = 256;      // elements of K per tile
constexpr int kTileBytes = 2304;  // 2,048 code bytes + 256 scale bytes
constexpr int kBlkRows = 16;     // head rows per block (MMA M)
// tiles in flight per warp in registers, and tiles prefetched into L2 beyond them, by n8 tile count
// (the two-tile kernel holds twice the B fragments and accumulators, so fewer tiles in registers)
constexpr int kDepthNT1 = 3;
constexpr int kPrefetchNT1 = 1;
constexpr int kDepthNT2 = 1;
constexpr int kPrefetchNT2 = 2;
// dynamic shared memory (the f16 hidden rows) at most: with the static arrays
// (up to 33 KB) within the 227 KB a CTA may use
constexpr size_t kMaxDynSmem = 192 * 1024;

struct Args {
    const uint16_t* x;       // bf16 [nb][H]
    const uint8_t* packed;   // tiled codes + scales
    const int32_t* cand;
    int nb, H, KS, Vc, n_blk;
    float g;
    Workspace ws;
    unsigned int* err;
    int32_t* ids;
    float* maxlogit;
    AcceptTail tail;
};

struct Tile {
    U32x8 lo, hi;  // code words of rows r and r + 8
    uint2 sc;      // their scales
};

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void load_tile(Tile& t, const uint8_t* rec, int lane) {
    t.lo = ld_stream32(rec + lane * 32);
    t.hi = ld_stream32(rec + 1024 + lane * 32);
    t.sc = ld_stream8(rec + 2048 + lane * 8);
}

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
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

// The 16 MMAs of one tile: A decoded from the tile's registers, B fragments
// from shared memory at `frag` (this lane's 8 bytes of tile t's first MMA).
template <int NT, int CH>
__device__ __forceinline__ void tile_mma(const Tile& tl, uint32_t frag, float (&acc)[NT][CH][4]) {
    const uint32_t sa01 = e4m3x2_h2(tl.sc.x & 0xFFFFu), sa23 = e4m3x2_h2(tl.sc.x >> 16);
    const uint32_t sb01 = e4m3x2_h2(tl.sc.y & 0xFFFFu), sb23 = e4m3x2_h2(tl.sc.y >> 16);
    const uint32_t sA[4] = {__byte_perm(sa01, 0, 0x1010), __byte_perm(sa01, 0, 0x3232), __byte_perm(sa23, 0, 0x1010),
                            __byte_perm(sa23, 0, 0x3232)};
    const uint32_t sB[4] = {__byte_perm(sb01, 0, 0x1010), __byte_perm(sb01, 0, 0x3232), __byte_perm(sb23, 0, 0x1010),
                            __byte_perm(sb23, 0, 0x3232)};
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // code word i holds MMAs 2i (bytes 0, 1) and 2i + 1 (bytes 2, 3)
        uint32_t ha[4], hb[4];
        e2m1x8_h2(tl.lo.v[i], ha);
        e2m1x8_h2(tl.hi.v[i], hb);
        const uint32_t s_a = sA[i >> 1], s_b = sB[i >> 1];
        const uint32_t a0 = hmul2(ha[0], s_a), a1 = hmul2(hb[0], s_b), a2 = hmul2(ha[1], s_a), a3 = hmul2(hb[1], s_b);
        const uint32_t c0 = hmul2(ha[2], s_a), c1 = hmul2(hb[2], s_b), c2 = hmul2(ha[3], s_a), c3 = hmul2(hb[3], s_b);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint2 b0 = lds64(frag + (uint32_t)(((2 * i) * NT + nt) * 256));
            const uint2 b1 = lds64(frag + (uint32_t)(((2 * i + 1) * NT + nt) * 256));
            mma16816(acc[nt][0], a0, a1, a2, a3, b0.x, b0.y);
            mma16816(acc[nt][CH - 1], c0, c1, c2, c3, b1.x, b1.y);
        }
    }
}

// Per-column argmax over one finished block of 16 rows (lowest row on ties),
// folded into the running best; blocks reach a warp in increasing row order,
// so an equal score keeps the earlier row.  s[nt] = .x/.y: row r8, columns
// 8nt + 2g4 (+1); .z/.w: row r8 + 8.
template <int NT>
__device__ __forceinline__ void block_argmax(const float4 (&s)[NT], int row0, int r8, int g4, const float* s_down,
                                             int Vc, float (&best_v)[NT][2], int (&best_r)[NT][2]) {
    const float ninf = -__int_as_float(0x7f800000);
    const int ra = row0 + r8, rb = ra + 8;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float d0 = s_down[8 * nt + 2 * g4], d1 = s_down[8 * nt + 2 * g4 + 1];
        float v0 = ra < Vc ? s[nt].x * d0 : ninf, v1 = ra < Vc ? s[nt].y * d1 : ninf;
        float v2 = rb < Vc ? s[nt].z * d0 : ninf, v3 = rb < Vc ? s[nt].w * d1 : ninf;
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
        if (row0 < Vc) {  // a block wholly past the head (never streamed) has no candidate
            if (best_r[nt][0] < 0 || bv0 > best_v[nt][0]) { best_v[nt][0] = bv0; best_r[nt][0] = br0; }
            if (best_r[nt][1] < 0 || bv1 > best_v[nt][1]) { best_v[nt][1] = bv1; best_r[nt][1] = br1; }
        }
    }
}

// Work split: CTA c owns blocks [c*n/grid, (c+1)*n/grid); its (block, tile)
// units are split evenly into contiguous ranges, one per warp.  A block
// cut by a range boundary is finished after all warps are done: each warp
// leaves its partial sums of its first and last block in shared memory, and
// the warp that holds the block's first tile adds the pieces in warp order.
template <int NT, int kWarpsP>
__global__ void __launch_bounds__(kWarpsP * 32, 1) k_nvfp4_packed(const Args a) {
    constexpr int kThreadsP = kWarpsP * 32;
    constexpr int N = 8 * NT;
    constexpr int CH = 2;  // independent accumulation chains per n8 tile (even / odd MMAs)
    constexpr int D = NT == 1 ? kDepthNT1 : kDepthNT2;
    constexpr int kPrefetch = NT == 1 ? kPrefetchNT1 : kPrefetchNT2;
    extern __shared__ __align__(16) uint8_t xfrag[];  // [H/16 MMAs][NT][32 lanes][8 B]
    __shared__ float4 cut[kWarpsP][2][NT][32];         // partial sums of cut blocks
    __shared__ unsigned long long merge[N];
    __shared__ float s_up[N], s_down[N];
    __shared__ unsigned int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g4 = lane & 3, r8 = lane >> 2;
    const int H = a.H, KS = a.KS;
    const int b_lo = (int)((long long)blockIdx.x * a.n_blk / gridDim.x);
    const int b_hi = (int)((long long)(blockIdx.x + 1) * a.n_blk / gridDim.x);
    const int U = (b_hi - b_lo) * KS;  // units of this CTA
    auto u_begin = [&](int w) { return (int)((long long)w * U / kWarpsP); };
    const int u_lo = u_begin(warp), u_hi = u_begin(warp + 1);
    const int n_units = u_hi - u_lo;
    const uint8_t* base = a.packed + ((size_t)b_lo * KS + u_lo) * kTileBytes;  // units are consecutive records

    pdl_launch_dependents();
    // the head never changes: its first tiles head for L2 before the dependency
    // wait and the hidden-row set-up, and are loaded into registers after it
    if (lane == 0)
        for (int u = 0; u < D + kPrefetch && u < n_units; ++u) prefetch_l2_bulk(base + (size_t)u * kTileBytes, kTileBytes);
    if (threadIdx.x < N) merge[threadIdx.x] = 0ull;
    pdl_wait();  // the hidden rows and the workspace may come from the previous kernel

    // B fragments in fragment order: entry (MMA m = 16t + j, tile nt, lane L)
    // holds hidden row L/4 + 8nt, elements 256t + 64(L%4) + 4j + [0, 4).  A
    // thread fills the entries of MMAs m and m + 1 (j even) from one 16-byte
    // load of the bf16 row (pair p: lane p % 32, MMA pair (p / 32) / NT, tile
    // (p / 32) % NT).  Its loads are all issued first; the per-row
    // power-of-two prescale (largest |x| into [2^14, 2^15)) is reduced from the
    // same registers, then the f16 entries are written.  Widths whose pairs do
    // not fit one round of registers read the rows a second time.
    {
        constexpr int kPairs = 16;                    // pairs per thread per round
        const int n_pairs = H * NT;                   // H/32 MMA pairs x NT x 32 lanes
        const bool one_round = n_pairs <= kPairs * kThreadsP;
        if (threadIdx.x < N) s_up[threadIdx.x] = 0.f;  // row maxima, as the bits of non-negative floats
        __syncthreads();
        float m[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) m[nt] = 0.f;
        uint4 v[kPairs];
        auto pair_src = [&](int p, int& nt, int& mp) -> const uint4* {
            const int f = p >> 5;
            nt = f % NT;
            mp = f / NT;
            const int n = r8 + 8 * nt;
            if (p >= n_pairs || n >= a.nb) return nullptr;
            return reinterpret_cast<const uint4*>(a.x + (size_t)n * H + (mp >> 3) * kTileK + g4 * 64 + (mp & 7) * 8);
        };
        for (int base = 0; base < n_pairs; base += kPairs * kThreadsP) {
#pragma unroll
            for (int i = 0; i < kPairs; ++i) {
                int nt, mp;
                const uint4* src = pair_src(base + threadIdx.x + i * kThreadsP, nt, mp);
                v[i] = src ? __ldg(src) : make_uint4(0u, 0u, 0u, 0u);
                const float mm = fmaxf(fmaxf(fmaxf(fabsf(bf_lo(v[i].x)), fabsf(bf_hi(v[i].x))),
                                             fmaxf(fabsf(bf_lo(v[i].y)), fabsf(bf_hi(v[i].y)))),
                                       fmaxf(fmaxf(fabsf(bf_lo(v[i].z)), fabsf(bf_hi(v[i].z))),
                                             fmaxf(fabsf(bf_lo(v[i].w)), fabsf(bf_hi(v[i].w)))));
#pragma unroll
                for (int q = 0; q < NT; ++q)
                    if (q == nt) m[q] = fmaxf(m[q], mm);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {  // lanes with equal L/4 hold the same row
            float mx = fmaxf(m[nt], __shfl_xor_sync(0xFFFFFFFFu, m[nt], 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            if (g4 == 0) atomicMax(reinterpret_cast<unsigned int*>(&s_up[r8 + 8 * nt]), __float_as_uint(mx));
        }
        __syncthreads();
        if (threadIdx.x < N) {
            const float mx = s_up[threadIdx.x];
            int k = 0;
            if (mx > 0.f) k = min(127, 141 - (int)((__float_as_uint(mx) >> 23) & 0xFF));
            s_down[threadIdx.x] = (int)threadIdx.x < a.nb ? a.g * ldexpf(1.f, -k) : 0.f;
            s_up[threadIdx.x] = (int)threadIdx.x < a.nb ? ldexpf(1.f, k) : 0.f;
        }
        __syncthreads();
        for (int base = 0; base < n_pairs; base += kPairs * kThreadsP) {
#pragma unroll
            for (int i = 0; i < kPairs; ++i) {
                int nt, mp;
                const int p = base + threadIdx.x + i * kThreadsP;
                const uint4* src = pair_src(p, nt, mp);
                if (!one_round) v[i] = src ? __ldg(src) : make_uint4(0u, 0u, 0u, 0u);
                if (p < n_pairs) {
                    const float up = s_up[r8 + 8 * nt];  // 0 for rows >= nb
                    const uint2 lo = make_uint2(f32x2_h2(bf_lo(v[i].x) * up, bf_hi(v[i].x) * up),
                                                f32x2_h2(bf_lo(v[i].y) * up, bf_hi(v[i].y) * up));
                    const uint2 hi = make_uint2(f32x2_h2(bf_lo(v[i].z) * up, bf_hi(v[i].z) * up),
                                                f32x2_h2(bf_lo(v[i].w) * up, bf_hi(v[i].w) * up));
                    *reinterpret_cast<uint2*>(xfrag + ((size_t)((2 * mp) * NT + nt) * 32 + lane) * 8) = lo;
                    *reinterpret_cast<uint2*>(xfrag + ((size_t)((2 * mp + 1) * NT + nt) * 32 + lane) * 8) = hi;
                }
            }
        }
    }
    __syncthreads();

    Tile buf[D];
#pragma unroll
    for (int d = 0; d < D; ++d)
        if (d < n_units) load_tile(buf[d], base + (size_t)d * kTileBytes, lane);

    const float ninf = -__int_as_float(0x7f800000);
    float best_v[NT][2];
    int best_r[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        best_v[nt][0] = best_v[nt][1] = ninf;
        best_r[nt][0] = best_r[nt][1] = -1;
    }
    float acc[NT][CH][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < CH; ++c) acc[nt][c][0] = acc[nt][c][1] = acc[nt][c][2] = acc[nt][c][3] = 0.f;
    const uint32_t frag0 = ptx::smem_u32(xfrag) + (uint32_t)lane * 8u;
    const uint32_t frag_tile = (uint32_t)(16 * NT * 256);  // bytes of B fragments per tile

    int t = u_lo % KS, blk = u_lo / KS;  // tile and CTA-local block of the current unit
    bool first = true;                     // the current block is this warp's first
    const bool starts_cut = t != 0;
    for (int u0 = 0; u0 < n_units; u0 += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int u = u0 + d;
            if (u < n_units) {
                tile_mma<NT, CH>(buf[d], frag0 + (uint32_t)t * frag_tile, acc);
                if (u + D < n_units) load_tile(buf[d], base + (size_t)(u + D) * kTileBytes, lane);
                if (lane == 0 && u + D + kPrefetch < n_units)
                    prefetch_l2_bulk(base + (size_t)(u + D + kPrefetch) * kTileBytes, kTileBytes);
                const bool blk_end = ++t == KS, range_end = u + 1 == n_units;
                if (blk_end || range_end) {
                    float4 sum[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        sum[nt] = make_float4(acc[nt][0][0], acc[nt][0][1], acc[nt][0][2], acc[nt][0][3]);
                        if (CH == 2) {
                            sum[nt].x += acc[nt][CH - 1][0];
                            sum[nt].y += acc[nt][CH - 1][1];
                            sum[nt].z += acc[nt][CH - 1][2];
                            sum[nt].w += acc[nt][CH - 1][3];
                        }
#pragma unroll
                        for (int c = 0; c < CH; ++c) acc[nt][c][0] = acc[nt][c][1] = acc[nt][c][2] = acc[nt][c][3] = 0.f;
                    }
                    if (!(first && starts_cut) && blk_end) {
                        block_argmax<NT>(sum, (b_lo + blk) * kBlkRows, r8, g4, s_down, a.Vc, best_v, best_r);
                    } else {  // a piece of a cut block: slot 0 = this warp's first block, 1 = its last
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) cut[warp][first ? 0 : 1][nt][lane] = sum[nt];
                    }
                    first = false;
                    t = 0;
                    ++blk;
                }
            }
        }
    }
    __syncthreads();
    // finish the cut block that starts in this warp's range (its last block, cut at the range end)
    if (n_units > 0 && u_hi % KS != 0) {
        const int jb = (u_hi - 1) / KS;  // CTA-local block
        if (jb * KS >= u_lo) {           // its first tile is ours: add the pieces in warp order
            float4 sum[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) sum[nt] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w = warp; w < kWarpsP; ++w) {
                const int wl = u_begin(w), wh = u_begin(w + 1);
                if (wl >= (jb + 1) * KS) break;
                if (wh <= wl) continue;  // a warp without units (fewer units than warps)
                const int slot = (wl / KS == jb) ? 0 : 1;  // block jb is the first or the last block of warp w
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float4 p = cut[w][slot][nt][lane];
                    sum[nt].x += p.x;
                    sum[nt].y += p.y;
                    sum[nt].z += p.z;
                    sum[nt].w += p.w;
                }
            }
            block_argmax<NT>(sum, (b_lo + jb) * kBlkRows, r8, g4, s_down, a.Vc, best_v, best_r);
        }
    }

    if (r8 == 0) {  // lanes 0..3: columns 8*tile + 2*lane, + 1
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int col = 8 * nt + 2 * g4 + h, r = best_r[nt][h];
                if (r >= 0 && col < a.nb && vh_guard(r < a.Vc, a.err)) {
                    const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + r) : (uint32_t)r;
                    atomicMax(&merge[col], make_key(best_v[nt][h], gid));
                }
            }
        }
    }

    // ---------------- CTA merge, publish, last-CTA decode ----------------
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
            int acc2 = 0;
            while (acc2 < k && nid[acc2] == d[acc2]) ++acc2;
            a.tail.accept_len[b] = acc2;
        }
    }
}

// Row-major codes [V][H/2] and scales [V][H/16] -> tiled records.  One thread
// per (record, half, lane): 32 code bytes and 4 scale bytes.
__global__ void k_nvfp4_pack(const uint8_t* __restrict__ Wq, const uint8_t* __restrict__ sc, int V, int H,
                             uint8_t* __restrict__ out, long long n_items) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_items) return;
    const int KS = H / kTileK;
    const int L = (int)(i & 31), h = (int)((i >> 5) & 1);
    const long long rec = i >> 6;  // record = block * KS + tile
    const int t = (int)(rec % KS);
    const long long blk = rec / KS;
    const long long row = blk * kBlkRows + (L >> 2) + 8 * h;
    uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
    uint32_t s = 0u;
    if (row < V) {
        const uint4* src = reinterpret_cast<const uint4*>(Wq + row * (H / 2) + (size_t)t * 128 + (L & 3) * 32);
        c0 = src[0];
        c1 = src[1];
        s = *reinterpret_cast<const uint32_t*>(sc + row * (H / 16) + (size_t)t * 16 + (L & 3) * 4);
    }
    uint8_t* r = out + rec * kTileBytes;
    uint4* dst = reinterpret_cast<uint4*>(r + h * 1024 + L * 32);
    dst[0] = c0;
    dst[1] = c1;
    *reinterpret_cast<uint32_t*>(r + 2048 + L * 8 + h * 4) = s;
}

// Resident CTAs per SM of a launch shape, cached per (kernel, threads, shared memory, device).
static cudaError_t resident_ctas(const void* kernel, int threads, size_t smem, int& per_sm) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, size_t, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const auto key = std::make_tuple(kernel, threads, smem, dev);
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) {
        per_sm = it->second;
        return cudaSuccess;
    }
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    if (e != cudaSuccess) return e;
    cache[key] = per_sm;
    return cudaSuccess;
}

}  // namespace fp4p

size_t nvfp4_packed_bytes(long long V, int H) {
    if (V < 1 || H < fp4p::kTileK || H % fp4p::kTileK != 0) return 0;
    return (size_t)((V + fp4p::kBlkRows - 1) / fp4p::kBlkRows) * (size_t)(H / fp4p::kTileK) * fp4p::kTileBytes;
}

size_t nvfp4_packed_smem(int nb, int H) { return (size_t)H * 16 * (nb > 8 ? 2 : 1); }

size_t nvfp4_packed_max_smem() { return fp4p::kMaxDynSmem; }

cudaError_t launch_nvfp4_pack(const uint8_t* Wq, const uint8_t* scales, int V, int H, uint8_t* packed, cudaStream_t s) {
    using namespace fp4p;
    const long long n_items = (long long)((V + kBlkRows - 1) / kBlkRows) * (H / kTileK) * 64;
    const long long blocks = (n_items + 255) / 256;
    if (blocks > INT_MAX) return cudaErrorInvalidValue;
    k_nvfp4_pack<<<(unsigned)blocks, 256, 0, s>>>(Wq, scales, V, H, packed, n_items);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_packed(const uint16_t* x, int nb, int H, const uint8_t* packed, float g, const int32_t* cand,
                                int Vc, Workspace ws, int32_t* ids, float* maxlogit, cudaStream_t s,
                                const AcceptTail& tail) {
    using namespace fp4p;
    if (nb < 1 || nb > 16 || H < kTileK || H % kTileK != 0 || Vc < 1 || Vc > INT_MAX - kBlkRows)
        return cudaErrorNotSupported;
    const size_t smem = nvfp4_packed_smem(nb, H);
    if (smem > kMaxDynSmem) return cudaErrorNotSupported;
    Args a{};
    a.x = x;
    a.packed = packed;
    a.cand = cand;
    a.nb = nb;
    a.H = H;
    a.KS = H / kTileK;
    a.Vc = Vc;
    a.n_blk = (Vc + kBlkRows - 1) / kBlkRows;
    a.g = g;
    a.ws = ws;
    a.err = ws.ticket + 1;
    a.ids = ids;
    a.maxlogit = maxlogit;
    a.tail = tail;
    auto kernel = nb <= 8 ? k_nvfp4_packed<1, kWarpsNT1> : k_nvfp4_packed<2, kWarpsNT2>;
    const int threads = 32 * (nb <= 8 ? kWarpsNT1 : kWarpsNT2);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = resident_ctas(reinterpret_cast<const void*>(kernel), threads, smem, per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const int grid = std::max(1, std::min(sm_count() * per_sm, a.n_blk));  // one resident wave
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace vh
