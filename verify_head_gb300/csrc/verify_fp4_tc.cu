// Greedy verification over a block-scaled 4-bit full head on a CTA pair
// (tcgen05 cta_group::2): exact f16 dequantisation in shared memory feeding
// one M = 256 x N = 256 MMA stream, fused with the per-hidden-row argmax and
// the accepted-prefix scan.
//
// Method: the target verifies the draft over the full output head
// ("少读一张大表，草稿路径才真正快起来"; "长上下文推理优化" §5: proposal ->
// target verification -> accept several tokens), here with the head in the
// NVFP4 format of "为什么生产推理我默认 vLLM" §3: E2M1 codes (element 2i in the
// low nibble), one E4M3 scale per 16 elements along H, one fp32 tensor scale g.
//
// Exactness.  Every E2M1 x E4M3 product has at most 6 significant bits and
// lies in [2^-10, 2688], so it is an f16 value: the dequantised weight
// w / g = e2m1 * e4m3 is exact in f16 (one cvt.rn.f16x2.e2m1x2 and one f16x2
// multiply per two weights).  The hidden rows are converted once per call to
// f16 with a per-row power-of-two prescale 2^k_r (largest |x| into
// [2^14, 2^15)), exact for every element within 2^31 of the row's largest;
// the MMA accumulates in fp32 and the score of hidden row r is
// acc * g * 2^-k_r, applied to each column's winning value (a positive
// per-column factor does not move the argmax over W rows).
//
// Mapping.  A cluster of two CTAs walks 256-row tiles of the head (128 rows
// per CTA, tile pt, pt + pairs, ...).  Each CTA holds half of the hidden
// rows (N / 2 of them) in every K-stage; the leader issues
// tcgen05.mma.cta_group::2 (A = the pair's 256 dequantised W rows, B = all N
// hidden rows, K = 16), and each CTA's TMEM receives the accumulator rows of
// its own 128 W rows.
//
// Before the pair kernel, k_hidden_f16 (one CTA per hidden row) writes the
// prescaled f16 rows and the per-row factors g * 2^-k_r into the caller's
// workspace; the pair kernel is a programmatic dependent launch, so its
// prologue and its first code loads overlap the conversion.
//
// Warp roles (480 threads per CTA):
//   warp 0       hidden-row producer: TMA of this CTA's half of the f16 hidden
//                rows, K = 64 per stage, completing on the leader's barrier
//   warp 1       TMEM owner; in the leader, the MMA issuer
//   warps 2..5   epilogue: TMEM -> per-column (hidden row) argmax
//   warp 6       code producer: TMA of the codes (128 contiguous bytes per
//                row, 128-byte swizzled) and the scales, K = 256 per raw stage
//   warps 7..14  dequantisers: raw codes -> f16 A tile (two 128-byte
//                swizzled K-major atoms of K = 64), K = 128 per A stage: each
//                hand-off to the MMA carries 8 MMAs of work
// Every wait is bounded (vh_ptx.cuh); on expiry the waiting thread raises the
// workspace error word and the CTA drains its copies, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "vh_kernels.h"
#include "vh_ptx.cuh"

namespace vh {
namespace fp4v {

using namespace ptx;

constexpr int kM = 128;                    // W rows per CTA per tile
constexpr int kPairM = 2 * kM;             // W rows per pair tile (MMA M)
constexpr int kKx = 64;                    // K per hidden-row stage (one 128-byte f16 swizzle atom)
constexpr int kKa = 128;                   // K per A stage (two swizzle atoms of 16 KiB)
constexpr int kKs = 256;                   // K per raw stage (128 code bytes per row)
constexpr int kAPerRaw = kKs / kKa;        // 2
constexpr int kAStages = 3;
constexpr int kXStages = 4;
constexpr int kRawStages = 3;
constexpr int kAAtom = kM * 128;           // 16 KiB: 128 rows x 64 K
constexpr int kABytes = kAAtom * (kKa / 64);  // 32 KiB
constexpr int kRawCodes = kM * kKs / 2;    // 16 KiB: [128 rows][128 B], 128-byte swizzled
constexpr int kRawScales = kM * kKs / 16;  // 2 KiB: [128 rows][16 B]
constexpr int kRawBytes = kRawCodes + kRawScales;
constexpr int kDeqWarps = 8;
constexpr int kDeqWarp0 = 7;
constexpr int kThreads = (kDeqWarp0 + kDeqWarps) * 32;  // 480
constexpr int kTmemCols = 512;             // two accumulators of up to 256 columns
static_assert(kRawBytes % 1024 == 0 && kABytes % 1024 == 0, "stage alignment");

template <int N>
struct Cfg {
    static constexpr int kXRows = N / 2;                // hidden rows per CTA
    static constexpr int kXBytes = kXRows * kKx * 2;    // per hidden stage
    static constexpr size_t kSmem = 1024 + (size_t)kAStages * kABytes + (size_t)kXStages * kXBytes +
                                    (size_t)kRawStages * kRawBytes + 256 /*barriers*/ + 256 * 8 /*merge*/ + 64;
};

struct alignas(8) Bars {
    unsigned long long raw_full[kRawStages];   // local: code TMA
    unsigned long long raw_empty[kRawStages];  // local: dequantiser warps
    unsigned long long x_full[kXStages];       // leader: both CTAs' hidden-row TMA
    unsigned long long x_empty[kXStages];      // both: MMA completion (multicast)
    unsigned long long a_full[kAStages];       // leader: dequantiser warps of both CTAs
    unsigned long long a_empty[kAStages];      // both: MMA completion (multicast)
    unsigned long long tmem_full[2];           // both
    unsigned long long tmem_empty[2];          // leader: 4 epilogue warps x 2 CTAs
    unsigned long long mma_done;
    unsigned int tmem_base;
    unsigned int pad;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Args {
    int R;        // hidden rows in this launch (1 .. N)
    int H;
    int V;
    int n_ptiles; // ceil(V / 256)
    const float* colscale;  // [R]: g * 2^-k_r of hidden row r
    Workspace ws;
    unsigned int* err;
    int32_t* next_ids;
    float* maxlogit;  // nullable
    AcceptTail tail;
};

// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrive on the leader's A-stage barrier with the default (CTA-scope release)
// semantics.  The dequantised rows a CTA writes are read only by its own SM's
// tensor core (each CTA of the pair supplies its 128 rows of A); the writer's
// fence.proxy.async orders them for that reader.  A cluster-scope release
// here costs a cluster-wide fence per stage and halves the kernel's speed.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// try_wait with cluster-scope acquire: the phase may have been completed by
// the peer CTA's threads, whose shared-memory writes the MMA then reads.
__device__ __forceinline__ bool mbar_try_wait_cluster(unsigned long long* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(unsigned long long* bar, uint32_t parity, unsigned int* err) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        const unsigned long long dt = globaltimer() - t0;
        if (dt > kErrPollNs && *reinterpret_cast<volatile unsigned int*>(err) != 0u) return false;
        if (dt > kTimeoutNs) {
            atomicOr(err, 1u);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, unsigned long long* bar, int x, int y,
                                            unsigned long long policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// TMA into this CTA's shared memory, completing on a barrier of the leader CTA.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int x, int y,
                                                 unsigned long long policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// K-major operand, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ unsigned long long desc_sw128(uint32_t saddr) {
    unsigned long long d = 0;
    d |= (unsigned long long)((saddr >> 4) & 0x3FFFu);
    d |= (unsigned long long)(16u >> 4) << 16;
    d |= (unsigned long long)(1024u >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// kind::f16 instruction descriptor: f16 A and B (format 0), fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void mma_pair(uint32_t tmem_d, unsigned long long adesc, unsigned long long bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void commit_pair(unsigned long long* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((unsigned short)3)
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

// Column argmax over a warp's 32 W rows for 16 hidden columns: v[j] is this
// lane's (W row's) score for column j.  Per column one redux gives the warp
// maximum and one ballot the lanes reaching it; a 4-level select tree hands
// column (lane % 16) to this lane: returns its maximum and ballot.
__device__ __forceinline__ void column_argmax16(const float (&v)[16], bool valid, float& m_out, uint32_t& b_out) {
    const int lane = threadIdx.x & 31;
    float m[16];
    uint32_t b[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float x = valid ? v[j] : -__int_as_float(0x7f800000);
        m[j] = redux_max_f32(x);
        b[j] = __ballot_sync(0xFFFFFFFFu, valid && x == m[j]);
    }
#pragma unroll
    for (int s = 8; s >= 1; s >>= 1) {
        const bool hi = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            m[i] = hi ? m[i + s] : m[i];
            b[i] = hi ? b[i + s] : b[i];
        }
    }
    m_out = m[0];
    b_out = b[0];
}

// ---------------------------------------------------------------------------
// Dequantisation helpers.

// Byte J of `word` (two E2M1 codes) -> f16x2, element 2i in the low half.
template <int J>
__device__ __forceinline__ uint32_t e2m1_h2(uint32_t word) {
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

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two E4M3 scales (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_h2(uint32_t two) {
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(two));
    return h2;
}

// One code word (8 E2M1 weights of one 16-element block) times its f16 scale
// pair (the block scale in both halves) -> 4 f16x2 words, in element order.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t sc, uint32_t (&o)[4]) {
    o[0] = hmul2(e2m1_h2<0>(w), sc);
    o[1] = hmul2(e2m1_h2<1>(w), sc);
    o[2] = hmul2(e2m1_h2<2>(w), sc);
    o[3] = hmul2(e2m1_h2<3>(w), sc);
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint32_t (&v)[4]) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t (&v)[4]) {
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(addr));
}


// ---------------------------------------------------------------------------

template <int N>
__global__ void __launch_bounds__(kThreads, 1)
    k_verify_fp4_pair(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_s,
                      const __grid_constant__ CUtensorMap map_x, const Args a) {
    using C = Cfg<N>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* raw_ring = smem;                                          // kRawStages x 18 KiB (1024-aligned)
    uint8_t* a_ring = raw_ring + (size_t)kRawStages * kRawBytes;       // kAStages x 32 KiB
    uint8_t* x_ring = a_ring + (size_t)kAStages * kABytes;             // kXStages x N/2 x 128 B
    Bars* bars = reinterpret_cast<Bars*>(x_ring + (size_t)kXStages * C::kXBytes);
    unsigned long long* merge = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(bars) + 256);
    __shared__ unsigned int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    const int x_steps = a.H / kKx, a_steps = a.H / kKa, raw_steps = a.H / kKs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(&bars->raw_full[s], 1);
            mbar_init(&bars->raw_empty[s], kDeqWarps);
        }
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(&bars->x_full[s], 1);
            mbar_init(&bars->x_empty[s], 1);
        }
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(&bars->a_full[s], 2 * kDeqWarps);
            mbar_init(&bars->a_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tmem_full[b], 1);
            mbar_init(&bars->tmem_empty[b], 8);
        }
        mbar_init(&bars->mma_done, 1);
        fence_barrier_init();
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x) merge[i] = 0ull;
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_before();
    cluster_sync();
    tc_after();
    const uint32_t tmem_base = bars->tmem_base;

    if (warp == 0) {
        // ---------------- hidden-row producer (both CTAs) ----------------
        if (lane == 0) {
            pdl_wait();  // the f16 hidden rows come from the conversion kernel
            const unsigned long long pol_x = policy_evict_last();
            uint32_t it = 0;
            bool ok = true;
            for (int pt = pair; pt < a.n_ptiles && ok; pt += n_pairs) {
                for (int ks = 0; ks < x_steps; ++ks, ++it) {
                    const int s = it % kXStages;
                    if (!mbar_wait(&bars->x_empty[s], ((it / kXStages) & 1u) ^ 1u, a.err)) { ok = false; break; }
                    if (leader) mbar_arrive_expect_tx(&bars->x_full[s], 2u * (uint32_t)C::kXBytes);
                    tma_load_2d_pair(x_ring + (size_t)s * C::kXBytes, &map_x, map_to_rank(smem_u32(&bars->x_full[s]), 0),
                                     ks * kKx, (int)rank * C::kXRows, pol_x);
                }
            }
            if (leader) {
                const uint32_t issued = it;
                for (uint32_t j = (issued > (uint32_t)kXStages ? issued - kXStages : 0); j < issued; ++j)
                    mbar_drain(&bars->x_full[j % kXStages], (j / kXStages) & 1u);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader only) ----------------
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_f16(kPairM, N);
            uint32_t ita = 0, itx = 0, local = 0;
            bool ok = true;
            for (int pt = pair; pt < a.n_ptiles && ok; pt += n_pairs, ++local) {
                const uint32_t buf = local & 1u;
                if (!mbar_wait(&bars->tmem_empty[buf], ((local >> 1) & 1u) ^ 1u, a.err)) break;
                tc_after();
                const uint32_t d_tmem = tmem_base + buf * 256u;
                for (int ka = 0; ka < a_steps && ok; ++ka, ++ita) {
                    const int as = ita % kAStages;
                    if (!mbar_wait_cluster(&bars->a_full[as], (ita / kAStages) & 1u, a.err)) { ok = false; break; }
                    const uint32_t sa = smem_u32(a_ring + (size_t)as * kABytes);
#pragma unroll
                    for (int xh = 0; xh < kKa / kKx; ++xh, ++itx) {  // one hidden-row stage per A atom
                        const int xs = itx % kXStages;
                        if (!mbar_wait(&bars->x_full[xs], (itx / kXStages) & 1u, a.err)) { ok = false; break; }
                        tc_after();
                        const uint32_t sb = smem_u32(x_ring + (size_t)xs * C::kXBytes);
#pragma unroll
                        for (int kk = 0; kk < kKx / 16; ++kk)
                            mma_pair(d_tmem, desc_sw128(sa + xh * kAAtom + kk * 32), desc_sw128(sb + kk * 32), idesc,
                                     (ka > 0 || xh > 0 || kk > 0) ? 1u : 0u);
                        commit_pair(&bars->x_empty[xs]);
                    }
                    if (!ok) break;
                    commit_pair(&bars->a_empty[as]);
                }
                if (ok) commit_pair(&bars->tmem_full[buf]);
            }
            commit_pair(&bars->mma_done);
            mbar_drain(&bars->mma_done, 0u);
        }
    } else if (warp < 6) {
        // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
        const int quarter = warp & 3;
        constexpr int kG = N / 32;
        float best_v[kG];
        uint32_t best_g[kG];
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            best_v[g] = -__int_as_float(0x7f800000);
            best_g[g] = 0xFFFFFFFFu;
        }
        const uint32_t empty_leader0 = map_to_rank(smem_u32(&bars->tmem_empty[0]), 0);
        const uint32_t empty_leader1 = map_to_rank(smem_u32(&bars->tmem_empty[1]), 0);
        uint32_t local = 0;
        for (int pt = pair; pt < a.n_ptiles; pt += n_pairs, ++local) {
            const uint32_t buf = local & 1u;
            if (!mbar_wait(&bars->tmem_full[buf], (local >> 1) & 1u, a.err)) break;
            tc_after();
            const uint32_t row0 = (uint32_t)(pt * kPairM + (int)rank * kM + quarter * 32);
            const bool valid = (int)(row0 + lane) < a.V;
#pragma unroll
            for (int g = 0; g < kG; ++g) {  // columns 32 g .. 32 g + 31, in two halves; lane l keeps column 32 g + l
                float m = 0.f;
                uint32_t bal = 0u;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float v[16];
                    tmem_ld16(tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * 256u + g * 32u + hf * 16u, v);
                    if (g + 1 == kG && hf == 1) {
                        tc_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(buf ? empty_leader1 : empty_leader0);
                    }
                    float mh;
                    uint32_t bh;
                    column_argmax16(v, valid, mh, bh);
                    if ((lane >> 4) == hf) {
                        m = mh;
                        bal = bh;
                    }
                }
                if (bal != 0u && (best_g[g] == 0xFFFFFFFFu || m > best_v[g])) {
                    best_v[g] = m;
                    best_g[g] = row0 + (uint32_t)(__ffs(bal) - 1);
                }
            }
        }
        pdl_wait();  // the per-row factors come from the conversion kernel
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            const int col = g * 32 + lane;
            if (best_g[g] != 0xFFFFFFFFu && col < a.R && vh_guard(best_g[g] < (uint32_t)a.V, a.err))
                atomicMax(&merge[col], make_key(best_v[g] * __ldg(a.colscale + col), best_g[g]));
        }
    } else if (warp == 6) {
        // ---------------- code producer (each CTA, local barriers) ----------------
        if (lane == 0) {
            const unsigned long long pol = policy_evict_first();
            uint32_t it = 0;
            bool ok = true;
            for (int pt = pair; pt < a.n_ptiles && ok; pt += n_pairs) {
                const int row = pt * kPairM + (int)rank * kM;
                for (int r = 0; r < raw_steps; ++r, ++it) {
                    const int s = it % kRawStages;
                    if (!mbar_wait(&bars->raw_empty[s], ((it / kRawStages) & 1u) ^ 1u, a.err)) { ok = false; break; }
                    uint8_t* dst = raw_ring + (size_t)s * kRawBytes;
                    mbar_arrive_expect_tx(&bars->raw_full[s], kRawBytes);
                    tma_load_2d(dst, &map_q, &bars->raw_full[s], r * (kKs / 2), row, pol);
                    tma_load_2d(dst + kRawCodes, &map_s, &bars->raw_full[s], r * (kKs / 16), row, pol);
                }
            }
            const uint32_t issued = it;
            for (uint32_t j = (issued > (uint32_t)kRawStages ? issued - kRawStages : 0); j < issued; ++j)
                mbar_drain(&bars->raw_full[j % kRawStages], (j / kRawStages) & 1u);
        }
    } else {
        // ---------------- dequantisers (warps 7..14) ----------------
        // Warp w covers W rows 16 w .. 16 w + 15: lane l takes row
        // 16 w + (l % 8) + 8 (l / 16) and half h = (l / 8) % 2 of each K = 128
        // A stage, i.e. 64 weights = 32 code bytes (two 16-byte units of the
        // row's 128-byte raw piece) and four block scales, written as eight
        // 16-byte chunks into swizzle atom h of the A stage.  The 8 lanes of a
        // quarter-warp hold 8 consecutive rows with one h, so both the
        // swizzled code loads and the swizzled A stores hit 8 distinct bank
        // groups.  Row r of an atom sits at (r / 8) * 1024 + (r % 8) * 128,
        // its chunk c at 16 * (c ^ (r % 8)).
        const int t = threadIdx.x - kDeqWarp0 * 32;  // 0..255
        const int wl = t & 31;
        const int row = 16 * (t >> 5) + (wl & 7) + 8 * (wl >> 4), half = (wl >> 3) & 1;
        const uint32_t sw7 = (uint32_t)(row & 7);
        const uint32_t a_row_off = (uint32_t)(half * kAAtom + (row >> 3) * 1024 + (row & 7) * 128);
        const uint32_t a_full_addr0 = leader ? 0u : map_to_rank(smem_u32(&bars->a_full[0]), 0);
        uint32_t rit = 0, ait = 0;
        bool ok = true;
        for (int pt = pair; pt < a.n_ptiles && ok; pt += n_pairs) {
            for (int r = 0; r < raw_steps && ok; ++r, ++rit) {
                const int rs = rit % kRawStages;
                if (!mbar_wait(&bars->raw_full[rs], (rit / kRawStages) & 1u, a.err)) { ok = false; break; }
                const uint32_t raw = smem_u32(raw_ring + (size_t)rs * kRawBytes);
                uint32_t sc[4];  // this row's 16 scale bytes of the raw stage (blocks 0..15)
                lds128(raw + (uint32_t)(kRawCodes + row * 16), sc);
#pragma unroll
                for (int j = 0; j < kAPerRaw; ++j, ++ait) {
                    const int as = ait % kAStages;
                    if (!mbar_wait(&bars->a_empty[as], ((ait / kAStages) & 1u) ^ 1u, a.err)) { ok = false; break; }
                    // code units 4 j + 2 h and 4 j + 2 h + 1 of the row (weights 128 j + 64 h .. + 63)
                    const uint32_t u0 = (uint32_t)(4 * j + 2 * half);
                    uint32_t q[8];
                    {
                        uint32_t q0[4], q1[4];
                        lds128(raw + (uint32_t)(row * 128) + (((u0) ^ sw7) << 4), q0);
                        lds128(raw + (uint32_t)(row * 128) + (((u0 + 1) ^ sw7) << 4), q1);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            q[i] = q0[i];
                            q[4 + i] = q1[i];
                        }
                    }
                    // blocks 8 j + 4 h .. + 3: scale word 2 j + h
                    const uint32_t sw = half ? sc[2 * j + 1] : sc[2 * j];
                    const uint32_t s01 = e4m3x2_h2(sw & 0xFFFFu), s23 = e4m3x2_h2(sw >> 16);
                    const uint32_t sb[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232),
                                            __byte_perm(s23, 0, 0x1010), __byte_perm(s23, 0, 0x3232)};
                    const uint32_t a_base = smem_u32(a_ring + (size_t)as * kABytes) + a_row_off;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {  // word i = weights 8 i .. 8 i + 7 of the 64 = chunk i of the atom row
                        uint32_t o[4];
                        dequant_word(q[i], sb[i >> 1], o);
                        sts128(a_base + (((uint32_t)i ^ sw7) << 4), o);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        if (leader)
                            mbar_arrive(&bars->a_full[as]);
                        else
                            mbar_arrive_remote(a_full_addr0 + (uint32_t)(as * 8));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->raw_empty[rs]);
            }
        }
    }

    // ---------------- pair teardown, publish, last-CTA decode ----------------
    pdl_wait();  // the workspace keys may still be read by an earlier launch
    tc_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
    for (int r = threadIdx.x; r < a.R; r += blockDim.x)
        if (merge[r] != 0ull) atomicMax(a.ws.keys + r, merge[r]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(a.ws.ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int r = threadIdx.x; r < a.R; r += blockDim.x) {
        const unsigned long long k = atomicExch(a.ws.keys + r, 0ull);
        vh_guard(k != 0ull, a.err);  // every hidden row has a winner
        a.next_ids[r] = (int32_t)key_gid(k);
        if (a.maxlogit != nullptr) a.maxlogit[r] = key_score(k);
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
// Host side.

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

// Codes [V][H/2] bytes, [128 rows][128 B] box (K = 256), 128-byte swizzle.
static bool make_map_codes(CUtensorMap* m, const void* base, int rows, int H) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(H / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(H / 2)};
    cuuint32_t box[2] = {(cuuint32_t)(kKs / 2), (cuuint32_t)kM};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scales [V][H/16] bytes, [128 rows][16 B] box, no swizzle.
static bool make_map_scales(CUtensorMap* m, const void* base, int rows, int H) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(H / 16), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(H / 16)};
    cuuint32_t box[2] = {(cuuint32_t)(kKs / 16), (cuuint32_t)kM};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// f16 hidden rows [R][H], [box_rows][64] box, 128-byte swizzle (rows past R
// read as zeros).
static bool make_map_x(CUtensorMap* m, const void* base, int R, int H, int box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)R};
    cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {(cuuint32_t)kKx, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
static cudaError_t launch_pair(const CUtensorMap& map_q, const CUtensorMap& map_s, const CUtensorMap& map_x,
                               const Args& a, cudaStream_t s) {
    const size_t smem = Cfg<N>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(k_verify_fp4_pair<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2u * (unsigned)std::max(1, std::min(sm_count() / 2, a.n_ptiles)));
    static std::atomic<int> clusters_cache[64] = {};  // per device (one per instantiation of this template)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    int clusters = clusters_cache[dev & 63].load(std::memory_order_relaxed);
    if (clusters < 1) {
        if (cudaOccupancyMaxActiveClusters(&clusters, k_verify_fp4_pair<N>, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            return cudaErrorNotSupported;
        }
        clusters_cache[dev & 63].store(clusters, std::memory_order_relaxed);
    }
    cfg.gridDim = dim3(2u * (unsigned)std::max(1, std::min(clusters, a.n_ptiles)));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_verify_fp4_pair<N>, map_q, map_s, map_x, a);
}

// Hidden rows bf16 [R][H] -> f16 [R][H] times 2^k_r (largest |x| of row r
// into [2^14, 2^15); k_r = 0 for an all-zero row), and colscale[r] =
// g * 2^-k_r.  One CTA per row.
__global__ void __launch_bounds__(256) k_hidden_f16(const uint16_t* __restrict__ X, int H, float g,
                                                    uint16_t* __restrict__ Xh, float* __restrict__ colscale) {
    __shared__ float s_max[8];
    pdl_launch_dependents();
    pdl_wait();  // X may come from the previous kernel; Xh may still be read by an earlier launch
    const int r = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t* xr = reinterpret_cast<const uint32_t*>(X + (size_t)r * H);
    float m = 0.f;
    for (int i = threadIdx.x; i < H / 2; i += blockDim.x) {
        const uint32_t pr = xr[i];
        m = fmaxf(m, fmaxf(fabsf(bf_lo(pr)), fabsf(bf_hi(pr))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) s_max[warp] = m;
    __syncthreads();
    m = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) m = fmaxf(m, s_max[w]);
    const int k = m > 0.f ? min(127, 141 - (int)((__float_as_uint(m) >> 23) & 0xFF)) : 0;
    const float up = ldexpf(1.f, k);
    uint32_t* out = reinterpret_cast<uint32_t*>(Xh + (size_t)r * H);
    for (int i = threadIdx.x; i < H / 2; i += blockDim.x) {
        const uint32_t pr = xr[i];
        uint32_t h2;
        asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(h2) : "f"(bf_lo(pr) * up), "f"(bf_hi(pr) * up));
        out[i] = h2;
    }
    if (threadIdx.x == 0) colscale[r] = g * ldexpf(1.f, -k);
}

}  // namespace fp4v

cudaError_t launch_hidden_f16(const uint16_t* X, int R, int H, float g, uint16_t* Xh, float* colscale, cudaStream_t s) {
    using namespace fp4v;
    if (R < 1 || H < 2 || H % 2 != 0) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)R);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_hidden_f16, X, H, g, Xh, colscale);
}

cudaError_t launch_verify_fp4_pair(const uint16_t* Xh, const float* colscale, int R, int H, const uint8_t* Wq,
                                   const uint8_t* scales, int V, Workspace ws, int32_t* next_ids, float* maxlogit,
                                   const AcceptTail& tail, cudaStream_t s) {
    using namespace fp4v;
    if (R < 1 || R > 256 || H < kKs || H % kKs != 0 || V < 1) return cudaErrorNotSupported;  // H % 256 == 0
    const int N = R <= 128 ? 128 : 256;
    alignas(64) CUtensorMap map_q, map_s, map_x;
    if (!make_map_codes(&map_q, Wq, V, H) || !make_map_scales(&map_s, scales, V, H) ||
        !make_map_x(&map_x, Xh, R, H, N / 2))
        return cudaErrorNotSupported;
    Args a{};
    a.R = R;
    a.H = H;
    a.V = V;
    a.n_ptiles = (V + kPairM - 1) / kPairM;
    a.colscale = colscale;
    a.ws = ws;
    a.err = ws.ticket + 1;
    a.next_ids = next_ids;
    a.maxlogit = maxlogit;
    a.tail = tail;
    return N == 128 ? launch_pair<128>(map_q, map_s, map_x, a, s) : launch_pair<256>(map_q, map_s, map_x, a, s);
}

}  // namespace vh
