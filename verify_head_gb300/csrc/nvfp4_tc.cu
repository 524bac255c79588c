// Block-scaled 4-bit draft head on the tensor cores: exact f16 dequantisation
// in shared memory feeding tcgen05.mma (kind::f16), fused with the argmax and
// the candidate-id mapping.
//
// Format (NVFP4 weights, "为什么生产推理我默认 vLLM" §3; NVFP4 candidate rows in
// "少读一张大表，草稿路径才真正快起来"): E2M1 codes, element 2i in the low nibble,
// one E4M3 scale per 16 elements along H, one fp32 tensor scale g.
//
// Every E2M1 x E4M3 product has at most 6 significant bits and lies in
// [2^-10, 2688], so it is an f16 value: the dequantised weight is exact.  The
// hidden rows are converted to f16 with a per-row power-of-two prescale 2^k_b
// (largest |x| into [2^14, 2^15)), exact for every element within 2^31 of
// the row's largest.  The MMA accumulates in fp32; the score of hidden row b
// is acc * g * 2^-k_b.
//
// Per CTA (persistent, one per SM, 128-row tiles, K in raw stages of 512):
//   warp 0       TMA producer: codes [128 rows x 256 B], scales [128 x 32 B]
//                and the bf16 hidden slice [16 x 512] of the next stage
//                into a 3-deep raw ring
//   warp 1       TMEM owner and MMA issuer (M = 128, N = 16, K = 16)
//   warps 2..5   epilogue: TMEM -> per-column (hidden row) argmax
//   warps 6..13  dequantisers: raw codes (128-byte swizzled by TMA) -> f16
//                A tile in TMEM (tcgen05.st; the MMA reads A from TMEM) and
//                bf16 hidden slice -> f16 B tile in shared memory, K = 256 per
//                A/B stage (two per raw stage), 3-deep ring
// Scores never leave the SM; per-CTA maxima go out as packed-key atomicMax
// and the last CTA decodes ids.  Waits are bounded (see vh_ptx.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "vh_kernels.h"
#include "vh_ptx.cuh"

namespace vh {
namespace fp4tc {

using namespace ptx;

constexpr int kM = 128;          // weight rows per tile
constexpr int kKs = 512;         // K per raw (TMA) stage: 256 contiguous code bytes per row
constexpr int kKa = 256;         // K per dequantised A/B stage (two per raw stage)
constexpr int kAbPerRaw = kKs / kKa;
constexpr int kN = 16;           // hidden rows per launch (MMA N)
constexpr int kRawStages = 3;
constexpr int kAbStages = 3;
constexpr int kRawCodes = kM * kKs / 2;    // 32 KiB: [128 rows][2 x 128 B], 128-byte swizzled
constexpr int kRawScales = kM * kKs / 16;  // 4 KiB: [128 rows][32 B]
constexpr int kXBox = 256;                 // hidden elements per TMA box (box dims are <= 256)
constexpr int kRawX = kN * kKs * 2;        // 16 KiB: bf16 hidden slice, two [16 rows][256] boxes
constexpr int kRawBytes = kRawCodes + kRawScales + kRawX;
constexpr int kBBytes = kN * kKa * 2;      // 8 KiB: 4 atoms of [16 rows x 128 B]
constexpr int kAtomB = kN * 128;           // 2 KiB
constexpr int kACols = kKa / 2;            // TMEM columns of one A stage (two f16 per column)
constexpr int kDeqWarps = 8;
constexpr int kThreadsFp4 = (2 + 4 + kDeqWarps) * 32;  // 448
constexpr int kKParts = kDeqWarps / 4;  // dequantiser warps per TMEM lane quarter (each a K range)
constexpr int kPartCols = kACols / kKParts;  // TMEM columns of an A stage per warp
static_assert(kDeqWarps == 8 || kDeqWarps == 16, "dequantiser split");
constexpr int kAcc = 4;          // independent accumulators per tile (K-steps rotate over them)
constexpr int kTmemCols = 512;   // A stages at columns 0, 128, 256; accumulators from column 384
constexpr int kDCol = kAbStages * kACols;
constexpr int kDBuf = kAcc * kN; // columns per accumulator buffer (two buffers)

struct alignas(8) Bars {
    unsigned long long raw_full[kRawStages];
    unsigned long long raw_empty[kRawStages];
    unsigned long long ab_full[kAbStages];
    unsigned long long ab_empty[kAbStages];
    unsigned long long tmem_full[2];
    unsigned long long tmem_empty[2];
    unsigned long long mma_done;
    unsigned int tmem_base;
    unsigned int pad;
};

constexpr size_t kSmem = 1024 + (size_t)kAbStages * kBBytes + (size_t)kRawStages * kRawBytes + sizeof(Bars) + 256;

struct Args {
    const uint16_t* x;     // [nb][H] bf16
    const int32_t* cand;   // [Vc] or nullptr
    int nb;
    int H;
    int Vc;
    int n_tiles;
    float g;
    Workspace ws;
    unsigned int* err;
    int32_t* ids;
    float* maxlogit;  // nullable
    AcceptTail tail;  // acceptance scan by the last CTA (draft == nullptr: none)
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, unsigned long long* bar, int x, int y,
                                            unsigned long long policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, unsigned long long* bar, int x, int y,
                                            int z, unsigned long long policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

__device__ __forceinline__ unsigned long long desc_sw128(uint32_t saddr) {
    unsigned long long d = 0;
    d |= (unsigned long long)((saddr >> 4) & 0x3FFFu);
    d |= (unsigned long long)(16u >> 4) << 16;
    d |= (unsigned long long)(1024u >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// kind::f16 instruction descriptor: f16 A and B (format 0), fp32 D, K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d, unsigned long long a, unsigned long long b, uint32_t idesc,
                                        uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Same with A read from tensor memory (lane = row, two f16 of K per column).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d, uint32_t a_tmem, unsigned long long b, uint32_t idesc,
                                               uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// 32 lanes x 32 columns of 32-bit words into TMEM: thread t writes lane base+t.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mma_commit(unsigned long long* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float redux_max_f32(float x) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
    return r;
}

// Four E2M1 pairs (the bytes of `w`, low byte first) -> four f16x2 words,
// the bytes taken through .b8 register views (no shifts or masks).
__device__ __forceinline__ void e2m1x8_h2(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}

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

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__global__ void __launch_bounds__(kThreadsFp4, 1)
    k_nvfp4_tc(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_s,
               const __grid_constant__ CUtensorMap map_x, const Args a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* b_ring = smem;                                             // kAbStages x 4 KiB
    uint8_t* raw_ring = b_ring + (size_t)kAbStages * kBBytes;           // kRawStages x 26 KiB
    Bars* bars = reinterpret_cast<Bars*>(raw_ring + (size_t)kRawStages * kRawBytes);
    unsigned long long* merge = reinterpret_cast<unsigned long long*>(bars + 1);  // [kN]
    __shared__ float s_up[kN], s_down[kN];
    __shared__ unsigned int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, k_stages = H / kKs, ab_stages = H / kKa;

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(&bars->raw_full[s], 1);
            mbar_init(&bars->raw_empty[s], kDeqWarps);
        }
        for (int s = 0; s < kAbStages; ++s) {
            mbar_init(&bars->ab_full[s], kDeqWarps);
            mbar_init(&bars->ab_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tmem_full[b], 1);
            mbar_init(&bars->tmem_empty[b], 4);
        }
        mbar_init(&bars->mma_done, 1);
        fence_barrier_init();
    }
    if (threadIdx.x < kN) merge[threadIdx.x] = 0ull;
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pdl_wait();  // the hidden rows and the workspace may come from the previous kernel
    // per-row power-of-two prescale of the hidden rows (identical in every CTA):
    // warp w takes rows w, w + 14, ..., each lane 16-byte pieces of the row,
    // all loads of a row independent
    for (int b = warp; b < kN; b += kThreadsFp4 / 32) {
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
            s_up[b] = ldexpf(1.f, k);
            s_down[b] = a.g * ldexpf(1.f, -k);
        }
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem_base = bars->tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const unsigned long long pol = policy_evict_first();
            const unsigned long long pol_x = policy_evict_last();
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < a.n_tiles && ok; tile += gridDim.x) {
                for (int ks = 0; ks < k_stages; ++ks, ++it) {
                    const int s = it % kRawStages;
                    if (!mbar_wait(&bars->raw_empty[s], ((it / kRawStages) & 1u) ^ 1u, a.err)) { ok = false; break; }
                    uint8_t* dst = raw_ring + (size_t)s * kRawBytes;
                    mbar_arrive_expect_tx(&bars->raw_full[s], kRawBytes);
                    tma_load_3d(dst, &map_q, &bars->raw_full[s], 0, ks * (kKs / 256), tile * kM, pol);
                    tma_load_2d(dst + kRawCodes, &map_s, &bars->raw_full[s], ks * (kKs / 16), tile * kM, pol);
#pragma unroll
                    for (int xbx = 0; xbx < kKs / kXBox; ++xbx)
                        tma_load_2d(dst + kRawCodes + kRawScales + xbx * (kN * kXBox * 2), &map_x, &bars->raw_full[s],
                                    ks * kKs + xbx * kXBox, 0, pol_x);
                }
            }
            const uint32_t issued = it;
            for (uint32_t j = (issued > (uint32_t)kRawStages ? issued - kRawStages : 0); j < issued; ++j)
                mbar_drain(&bars->raw_full[j % kRawStages], (j / kRawStages) & 1u);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(kM, kN);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < a.n_tiles && ok; tile += gridDim.x, ++local) {
                const uint32_t buf = local & 1u;
                if (!mbar_wait(&bars->tmem_empty[buf], ((local >> 1) & 1u) ^ 1u, a.err)) break;
                tc_after();
                const uint32_t d = tmem_base + kDCol + buf * kDBuf;
                for (int ka = 0; ka < ab_stages; ++ka, ++it) {
                    const int s = it % kAbStages;
                    if (!mbar_wait(&bars->ab_full[s], (it / kAbStages) & 1u, a.err)) { ok = false; break; }
                    tc_after();
                    const uint32_t ta = tmem_base + (uint32_t)(s * kACols);
                    const uint32_t sb = smem_u32(b_ring + (size_t)s * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kKa / 16; ++kk) {
                        const uint32_t atom = kk >> 2, off = (kk & 3) * 32;
                        // consecutive K-steps go to different accumulators so that no MMA waits
                        // on the one before it
                        mma_f16_tmem_a(d + (uint32_t)((kk % kAcc) * kN), ta + kk * 8u,
                                       desc_sw128(sb + atom * kAtomB + off), idesc, (ka > 0 || kk >= kAcc) ? 1u : 0u);
                    }
                    mma_commit(&bars->ab_empty[s]);
                }
                if (ok) mma_commit(&bars->tmem_full[buf]);
            }
            mma_commit(&bars->mma_done);
            mbar_drain(&bars->mma_done, 0u);
        }
    } else if (warp < 6) {
        // ---------------- epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;
        float best_v = -__int_as_float(0x7f800000);
        uint32_t best_g = 0xFFFFFFFFu;  // this lane owns hidden row `lane` (lanes < kN)
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++local) {
            const uint32_t buf = local & 1u;
            if (!mbar_wait(&bars->tmem_full[buf], (local >> 1) & 1u, a.err)) break;
            tc_after();
            float v[16];
            {
                const uint32_t base = tmem_base + ((uint32_t)(quarter * 32) << 16) + kDCol + buf * kDBuf;
                tmem_ld16(base, v);
#pragma unroll
                for (int i = 1; i < kAcc; ++i) {
                    float u[16];
                    tmem_ld16(base + (uint32_t)(i * kN), u);
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] += u[j];
                }
            }
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tmem_empty[buf]);
            const int row0 = tile * kM + quarter * 32;
            const bool valid = row0 + lane < a.Vc;
            float m[16];
            uint32_t bal[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float xv = valid ? v[j] * s_down[j] : -__int_as_float(0x7f800000);
                m[j] = redux_max_f32(xv);
                bal[j] = __ballot_sync(0xFFFFFFFFu, valid && xv == m[j]);
            }
#pragma unroll
            for (int s = 8; s >= 1; s >>= 1) {
                const bool hi = (lane & s) != 0;
#pragma unroll
                for (int i = 0; i < s; ++i) {
                    m[i] = hi ? m[i + s] : m[i];
                    bal[i] = hi ? bal[i + s] : bal[i];
                }
            }
            if (lane < kN && bal[0] != 0u && (best_g == 0xFFFFFFFFu || m[0] > best_v)) {
                best_v = m[0];
                best_g = (uint32_t)(row0 + __ffs(bal[0]) - 1);
            }
        }
        if (lane < a.nb && best_g != 0xFFFFFFFFu && vh_guard(best_g < (uint32_t)a.Vc, a.err)) {
            const uint32_t gid = a.cand ? (uint32_t)__ldg(a.cand + best_g) : best_g;
            atomicMax(&merge[lane], make_key(best_v, gid));
        }
    } else {
        // ---------------- dequantisers (warps 6..13) ----------------
        // Each raw stage (K = 512: sixteen 16-byte code chunks of 32 weights
        // per row) becomes two A/B stages (K = 256).  The A stage lives in
        // TMEM (lane = weight row, two f16 of K per column), written straight
        // from registers with tcgen05.st; a warp may only reach its TMEM lane
        // quarter (warp % 4), so warps 6..9 write columns 0..63 of the stage
        // (K 0..127) for their quarter and warps 10..13 columns 64..127.  The
        // raw codes were stored 128-byte swizzled by the TMA, so the 16-byte
        // loads of 32 consecutive rows are bank-conflict free.
        const int t = threadIdx.x - 6 * 32;  // 0 .. 32 kDeqWarps - 1
        const int quarter = warp & 3, kpart = (warp - 6) >> 2;
        const int row = quarter * 32 + lane;
        constexpr int kXPer = kN * kKa / (kDeqWarps * 32);  // hidden-slice elements per thread and stage
        const int xb = t / (kDeqWarps * 2), xp = t % (kDeqWarps * 2);  // B row / kXPer-element part
        const float up = s_up[xb];
        const uint32_t tmem_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(kpart * kPartCols);
        uint32_t rit = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < a.n_tiles && ok; tile += gridDim.x) {
            for (int ks = 0; ks < k_stages && ok; ++ks, ++rit) {
                const int rs = rit % kRawStages;
                if (!mbar_wait(&bars->raw_full[rs], (rit / kRawStages) & 1u, a.err)) { ok = false; break; }
                const uint32_t raw = smem_u32(raw_ring + (size_t)rs * kRawBytes);
                for (int h = 0; h < kAbPerRaw; ++h) {
                    const uint32_t abit = kAbPerRaw * rit + h;
                    const int as = abit % kAbStages;
                    if (!mbar_wait(&bars->ab_empty[as], ((abit / kAbStages) & 1u) ^ 1u, a.err)) { ok = false; break; }
                    tc_after();
                    constexpr int kChunks = kPartCols / 16;     // 16-byte code chunks (32 weights) per warp
                    const int c0 = h * 8 + kpart * kChunks;   // first chunk (of 16 in the raw row)
                    uint32_t sc8[kChunks / 2];                // scales of blocks 2*c0 .. 2*c0 + 2*kChunks - 1
                    if constexpr (kChunks == 4) {
                        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];"
                                     : "=r"(sc8[0]), "=r"(sc8[kChunks / 2 - 1])
                                     : "r"(raw + (uint32_t)(kRawCodes + row * (kKs / 16) + 2 * c0)));
                    } else {
                        asm volatile("ld.shared.u32 %0, [%1];"
                                     : "=r"(sc8[0])
                                     : "r"(raw + (uint32_t)(kRawCodes + row * (kKs / 16) + 2 * c0)));
                    }
#pragma unroll
                    for (int half = 0; half < kChunks / 2; ++half) {  // 64 weights -> 32 TMEM columns each
                        const uint32_t sc4 = sc8[half];
                        const uint32_t s01 = e4m3x2_h2(sc4 & 0xFFFFu), s23 = e4m3x2_h2(sc4 >> 16);
                        uint32_t out[32];
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int c = c0 + 2 * half + cc;
                            const int seg = row * 2 + (c >> 3);  // 128-byte segment of the swizzled raw tile
                            uint32_t q[4];
                            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                         : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3])
                                         : "r"(raw + (uint32_t)(seg * 128 + (((c & 7) ^ (seg & 7)) * 16))));
                            const uint32_t sp = cc ? s23 : s01;
                            const uint32_t slo = __byte_perm(sp, 0, 0x1010), shi = __byte_perm(sp, 0, 0x3232);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {  // word j = elements 8j .. 8j+7 of the chunk
                                const uint32_t ss = j < 2 ? slo : shi;
                                uint32_t hh[4];
                                e2m1x8_h2(q[j], hh);
                                out[cc * 16 + j * 4 + 0] = hmul2(hh[0], ss);
                                out[cc * 16 + j * 4 + 1] = hmul2(hh[1], ss);
                                out[cc * 16 + j * 4 + 2] = hmul2(hh[2], ss);
                                out[cc * 16 + j * 4 + 3] = hmul2(hh[3], ss);
                            }
                        }
                        tmem_st32(tmem_row + (uint32_t)(as * kACols + half * 32), out);
                    }
#pragma unroll
                    for (int e = 0; e < kXPer / 8; ++e) {  // hidden slice [16][256] bf16 -> f16 B tile (rows >= nb: zeros)
                        const int kx = h * kKa + xp * kXPer + e * 8;  // element within the raw stage
                        const uint32_t src = raw + (uint32_t)(kRawCodes + kRawScales + (kx / kXBox) * (kN * kXBox * 2) +
                                                              xb * (kXBox * 2) + (kx % kXBox) * 2);
                        uint32_t pr[4];
                        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(pr[0]), "=r"(pr[1]), "=r"(pr[2]), "=r"(pr[3]) : "r"(src));
                        const int piece = xp * (kXPer / 8) + e;  // 8-element piece of the stage (4 atoms of 8)
                        const uint32_t b_addr = smem_u32(b_ring + (size_t)as * kBBytes) + (uint32_t)(piece >> 3) * kAtomB +
                                                (uint32_t)xb * 128u + (uint32_t)(((piece & 7) ^ (xb & 7)) * 16);
                        sts128(b_addr, f32x2_h2(bf_lo(pr[0]) * up, bf_hi(pr[0]) * up),
                               f32x2_h2(bf_lo(pr[1]) * up, bf_hi(pr[1]) * up),
                               f32x2_h2(bf_lo(pr[2]) * up, bf_hi(pr[2]) * up),
                               f32x2_h2(bf_lo(pr[3]) * up, bf_hi(pr[3]) * up));
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    tc_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->ab_full[as]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->raw_empty[rs]);
            }
        }
    }

    // ---------------- CTA merge, publish, last-CTA decode ----------------
    tc_before();
    __syncthreads();
    if (warp == 1) {
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
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

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// bf16 hidden rows [nb][H] as a 2-D map with a [16 rows][256] box, no swizzle
// (rows past nb read as zeros).
static bool make_map_x(CUtensorMap* m, const void* base, int nb, int H) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)nb};
    cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {(cuuint32_t)kXBox, (cuuint32_t)kN};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Codes [Vc][H/2] bytes viewed as [Vc][H/256][128]: a box of [128 rows][2][128 B]
// reads 256 contiguous bytes of every row (DRAM streams long row segments
// far better than 128-byte pieces), stored 128-byte swizzled.
static bool make_map_codes(CUtensorMap* m, const void* base, int rows, int H) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)(H / 256), (cuuint64_t)rows};
    cuuint64_t strides[2] = {128, (cuuint64_t)(H / 2)};
    cuuint32_t box[3] = {128, (cuuint32_t)(kKs / 256), (cuuint32_t)kM};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint8 row-major [rows][cols] map, [128 rows][box_cols] box.
static bool make_map_u8(CUtensorMap* m, const void* base, int rows, int cols, int box_cols, CUtensorMapSwizzle sw) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)kM};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fp4tc

cudaError_t launch_nvfp4_tc(const uint16_t* x, int nb, int H, const uint8_t* Wq, const uint8_t* scales, float g,
                            const int32_t* cand, int Vc, Workspace ws, int32_t* ids, float* maxlogit, cudaStream_t s,
                            const AcceptTail& tail) {
    using namespace fp4tc;
    if (nb < 1 || nb > kN || H < kKs || H % kKs != 0 || Vc < 1) return cudaErrorNotSupported;  // H % 512 == 0
    alignas(64) CUtensorMap map_q, map_s, map_x;
    if (!make_map_codes(&map_q, Wq, Vc, H) ||
        !make_map_u8(&map_s, scales, Vc, H / 16, kKs / 16, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map_x(&map_x, x, nb, H))
        return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(k_nvfp4_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    Args a{};
    a.x = x;
    a.cand = cand;
    a.nb = nb;
    a.H = H;
    a.Vc = Vc;
    a.n_tiles = (Vc + kM - 1) / kM;
    a.g = g;
    a.ws = ws;
    a.err = ws.ticket + 1;
    a.ids = ids;
    a.maxlogit = maxlogit;
    a.tail = tail;
    const int grid = std::max(1, std::min(sm_count(), a.n_tiles));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreadsFp4);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_nvfp4_tc, map_q, map_s, map_x, a);
}

}  // namespace vh
