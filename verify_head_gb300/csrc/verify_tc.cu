// Greedy verification on the 5th-generation tensor cores (tcgen05 + TMEM +
// TMA): skinny GEMM S = W_full · Xᵀ fused with the per-hidden-row argmax
// and the accepted-prefix scan.
//
// Method: the target keeps the full 248,320-row output head and verifies the
// draft ("少读一张大表，草稿路径才真正快起来"); greedy verification accepts the
// leading draft tokens that equal the target's own choice ("长上下文推理优化"
// §5: MTP proposal -> target verification -> accept several tokens).
//
// Mapping.  One persistent CTA per SM walks 128-row tiles of W (tile t,
// t + grid, ...).  For each tile the MMA computes D[128 W rows][N] with
// A = W tile (M = 128, K-major) and B = all R <= 256 hidden rows (N = R
// rounded up to 16, K-major), K = H in stages of 64 (one 128-byte swizzle
// atom).  D lives in TMEM; two accumulator buffers of 256 columns let the
// epilogue of tile i overlap the MMAs of tile i+1.  Scores never leave the
// SM: the epilogue reads 32 columns at a time (thread = W row, register =
// hidden row); per column one redux.sync.max.f32 gives the warp maximum and
// one ballot the lowest W row reaching it, and a select tree hands column j
// to lane j.  Running maxima stay in registers across tiles; at the end the
// four epilogue warps merge in shared memory and publish one atomicMax per
// hidden row; the last CTA (ticket) decodes ids, runs the acceptance scan
// and re-zeroes the workspace.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner and
// MMA issuer, warps 2..5 = epilogue (TMEM lane quarter = warp % 4).
//
// Every wait is bounded (about 2 s of %globaltimer); on expiry the waiting
// thread sets the workspace error word, skips the rest of its work, and the
// CTA still drains its copies, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "vh_kernels.h"
#include "vh_verify.h"
#include "vh_ptx.cuh"

namespace vh {
namespace tc {

constexpr int kBlockM = 128;      // W rows per tile (MMA M)
constexpr int kBlockK = 64;       // K per stage (one 128 B swizzle atom of bf16)
constexpr int kMaxN = 256;        // hidden rows per launch (MMA N <= 256)
constexpr int kMaxStagesTc = 8;    // deepest ring of any instance
constexpr int kThreadsTc = 192;
constexpr int kEpiWarp0 = 2;
constexpr int kStageA = kBlockM * kBlockK * 2;  // 16 KiB
constexpr int kTmemCols = 512;                  // two 256-column accumulators

struct alignas(8) Barriers {
    unsigned long long full[kMaxStagesTc];
    unsigned long long empty[kMaxStagesTc];
    unsigned long long tmem_full[2];
    unsigned long long tmem_empty[2];
    unsigned long long mma_done;
    unsigned int tmem_base;
    unsigned int pad;
};

// Shared memory of k_verify_tc<STAGES, NMAX>: a ring of STAGES x (16 KiB of W +
// NMAX x 128 B of hidden rows).
__host__ __device__ constexpr size_t smem_bytes_tc(int stages, int nmax) {
    return 1024 /*alignment slack*/ + (size_t)stages * (kStageA + (size_t)nmax * kBlockK * 2) + sizeof(Barriers) +
           kMaxN * 8 /*merge*/ + 64;
}

struct TcArgs {
    int R;        // hidden rows in this launch (1..256)
    int N;        // MMA N = R rounded up to 16
    int H;
    int V;
    int n_tiles;  // ceil(V / 128)
    Workspace ws;
    unsigned int* err;
    int32_t* next_ids;
    float* maxlogit;
    AcceptTail tail;
    const int32_t* cand;  // draft head: next_ids[r] = cand[winning row]; nullptr for verify
};

// ---------------------------------------------------------------------------
// tcgen05 / TMA wrappers (barriers and bulk copies: vh_ptx.cuh).

using ptx::globaltimer;
using ptx::mbar_arrive;
using ptx::mbar_arrive_expect_tx;
using ptx::mbar_drain;
using ptx::mbar_init;
using ptx::mbar_try_wait;
using ptx::mbar_wait;
using ptx::policy_evict_first;
using ptx::policy_evict_last;
using ptx::smem_u32;

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, unsigned long long* bar, int x, int y,
                                            unsigned long long policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), tile base 1024-byte aligned.
__device__ __forceinline__ unsigned long long smem_desc_sw128(uint32_t saddr) {
    unsigned long long d = 0;
    d |= (unsigned long long)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (unsigned long long)(16u >> 4) << 16;                   // leading byte offset (unused here)
    d |= (unsigned long long)(1024u >> 4) << 32;                 // stride byte offset
    d |= 1ull << 46;                                             // descriptor version (tcgen05)
    d |= 2ull << 61;                                             // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4)                     // D format: f32
           | (1u << 7)                   // A format: bf16
           | (1u << 10)                  // B format: bf16
           | ((uint32_t)(N >> 3) << 17)  // N / 8
           | ((uint32_t)(M >> 4) << 24); // M / 16
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, unsigned long long adesc, unsigned long long bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(unsigned long long* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 columns of fp32 from TMEM: thread t gets lane (base + t),
// columns col .. col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float redux_max_f32(float x) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
    return r;
}

// Column argmax over the warp's 32 W rows for 32 hidden columns at once.
// v[j] is this lane's (W row's) score for column j.  For every column the
// warp maximum comes from one redux and the lowest winning lane from one
// ballot; a 5-level select tree then hands column `lane` to this lane:
// returns its maximum and the ballot of lanes reaching it (0 = none valid).
__device__ __forceinline__ void column_argmax32(const float (&v)[32], bool valid, float& m_out, uint32_t& b_out) {
    const int lane = threadIdx.x & 31;
    float m[32];
    uint32_t b[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float x = valid ? v[j] : -__int_as_float(0x7f800000);
        m[j] = redux_max_f32(x);
        b[j] = __ballot_sync(0xFFFFFFFFu, valid && x == m[j]);
    }
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
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

template <int kStages, int NMAX>
__global__ void __launch_bounds__(kThreadsTc, 1)
    k_verify_tc(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x, const TcArgs a) {
    static_assert(kStages <= kMaxStagesTc && NMAX % 8 == 0 && NMAX <= kMaxN, "ring shape");
    constexpr int kStageB = NMAX * kBlockK * 2;  // hidden rows of one stage (1024-byte multiple)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stage_a = smem;                                  // kStages x 16 KiB (W tiles)
    uint8_t* stage_b = smem + (size_t)kStages * kStageA;      // kStages x NMAX x 128 B (hidden rows)
    Barriers* bars = reinterpret_cast<Barriers*>(stage_b + (size_t)kStages * kStageB);
    unsigned long long* merge = reinterpret_cast<unsigned long long*>(bars + 1);  // [kMaxN]
    __shared__ unsigned int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k_stages = a.H / kBlockK;
    const uint32_t b_bytes = (uint32_t)a.N * kBlockK * 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tmem_full[b], 1);
            mbar_init(&bars->tmem_empty[b], 4);  // one arrival per epilogue warp
        }
        mbar_init(&bars->mma_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    for (int i = threadIdx.x; i < kMaxN; i += blockDim.x) merge[i] = 0ull;
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    // Programmatic dependent launch: the next kernel may start its own prologue now.  The head is
    // read-only, so the first ring of W stages is requested before this kernel waits for the previous
    // one; the hidden rows, the draft ids and the workspace are touched only after the wait.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const unsigned long long pol_w = policy_evict_first();
            const unsigned long long pol_x = policy_evict_last();
            uint32_t it = 0;  // global k-stage counter
            bool ok = true, waited = false;
            // hidden-row loads of the first ring (stage j = it = j, K stage j % k_stages), once the
            // previous kernel is done
            auto release_first_ring = [&](uint32_t n) {
                asm volatile("griddepcontrol.wait;" ::: "memory");
                for (uint32_t j = 0; j < n; ++j)
                    tma_load_2d(stage_b + (size_t)j * kStageB, &map_x, &bars->full[j], (int)(j % k_stages) * kBlockK,
                                0, pol_x);
                waited = true;
            };
            for (int tile = blockIdx.x; tile < a.n_tiles && ok; tile += gridDim.x) {
                for (int ks = 0; ks < k_stages; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(&bars->empty[s], ph ^ 1u, a.err)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bars->full[s], (uint32_t)kStageA + b_bytes);
                    tma_load_2d(stage_a + (size_t)s * kStageA, &map_w, &bars->full[s], ks * kBlockK,
                                tile * kBlockM, pol_w);
                    if (waited)
                        tma_load_2d(stage_b + (size_t)s * kStageB, &map_x, &bars->full[s], ks * kBlockK, 0, pol_x);
                    else if (it + 1 == (uint32_t)kStages)
                        release_first_ring(it + 1);
                }
            }
            if (!waited) release_first_ring(it);  // fewer K stages in all than the ring holds, or a failed wait
            // drain: every issued load must land before the CTA may exit
            const uint32_t issued = it;
            for (uint32_t j = (issued > (uint32_t)kStages ? issued - kStages : 0); j < issued; ++j)
                mbar_drain(&bars->full[j % kStages], (j / kStages) & 1u);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kBlockM, a.N);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < a.n_tiles && ok; tile += gridDim.x, ++local) {
                const uint32_t buf = local & 1u;
                if (!mbar_wait(&bars->tmem_empty[buf], ((local >> 1) & 1u) ^ 1u, a.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * 256u;
                for (int ks = 0; ks < k_stages; ++ks, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait(&bars->full[s], (it / kStages) & 1u, a.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(stage_a + (size_t)s * kStageA);
                    const uint32_t sb = smem_u32(stage_b + (size_t)s * kStageB);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        mma_bf16(d_tmem, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32), idesc,
                                 (ks > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&bars->empty[s]);
                }
                if (ok) mma_commit(&bars->tmem_full[buf]);
            }
            // all MMAs issued by this thread have completed once this arrives
            mma_commit(&bars->mma_done);
            mbar_drain(&bars->mma_done, 0u);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;  // TMEM lanes quarter*32 .. +31
        const int ngroups = (a.N + 31) / 32;
        float best_v[kMaxN / 32];
        uint32_t best_g[kMaxN / 32];
#pragma unroll
        for (int g = 0; g < kMaxN / 32; ++g) {
            best_v[g] = -__int_as_float(0x7f800000);
            best_g[g] = 0xFFFFFFFFu;  // none yet
        }
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++local) {
            const uint32_t buf = local & 1u;
            if (!mbar_wait(&bars->tmem_full[buf], (local >> 1) & 1u, a.err)) break;
            tc_fence_after();
            const uint32_t row0 = (uint32_t)(tile * kBlockM + quarter * 32);  // id of lane 0's W row
            const bool valid = (int)(row0 + lane) < a.V;
#pragma unroll
            for (int g = 0; g < kMaxN / 32; ++g) {
                if (g < ngroups) {
                    float v[32];
                    tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * 256u + g * 32u, v);
                    if (g + 1 == ngroups) {  // accumulator fully read: hand it back to the MMA warp
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->tmem_empty[buf]);
                    }
                    float m;
                    uint32_t bal;
                    column_argmax32(v, valid, m, bal);
                    // tiles arrive in increasing row order: strict '>' keeps the lower id on ties
                    if (bal != 0u && (best_g[g] == 0xFFFFFFFFu || m > best_v[g])) {
                        best_v[g] = m;
                        best_g[g] = row0 + (uint32_t)(__ffs(bal) - 1);
                    }
                }
            }
        }
#pragma unroll
        for (int g = 0; g < kMaxN / 32; ++g)
            if (g < ngroups && best_g[g] != 0xFFFFFFFFu)
                atomicMax(&merge[g * 32 + lane], make_key(best_v[g], best_g[g]));
    }

    // ---------------- CTA merge, publish, last-CTA decode ----------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the workspace may come from the previous kernel
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
        const uint32_t gid = key_gid(k);
        a.next_ids[r] = (int32_t)((a.cand != nullptr && gid < (uint32_t)a.V) ? (uint32_t)__ldg(a.cand + gid) : gid);
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
// CTA-pair variant for 129..256 hidden rows (tcgen05 cta_group::2).
//
// Two CTAs of a cluster share each MMA: M = 256 W rows (128 from each CTA's
// shared memory), N = 256 hidden rows (128 from each CTA), K = 16.  Each CTA
// therefore stages only half of the hidden tile (16 KiB per K-stage instead
// of 32), which halves the shared-memory traffic per SM and lets the ring
// hold 6 stages of 32 KiB.  The leader CTA (rank 0) issues the MMAs; both
// CTAs' TMA loads complete on the leader's barrier, and the MMA completion
// is multicast to both CTAs' barriers.  Each CTA's TMEM receives the
// accumulator rows of its own 128 W rows, so the epilogue is unchanged.

constexpr int kStages2 = 6;
constexpr int kStageA2 = kBlockM * kBlockK * 2;  // 16 KiB: this CTA's 128 W rows
constexpr int kStageB2 = 128 * kBlockK * 2;      // 16 KiB: this CTA's 128 hidden rows
constexpr int kPairM = 2 * kBlockM;              // W rows per pair tile

struct alignas(8) Barriers2 {
    unsigned long long full[kStages2];   // leader only: both CTAs' loads land here
    unsigned long long empty[kStages2];  // both CTAs: the MMA multicasts its completion
    unsigned long long tmem_full[2];     // both CTAs
    unsigned long long tmem_empty[2];    // leader only: 4 epilogue warps x 2 CTAs
    unsigned long long mma_done;
    unsigned int tmem_base;
    unsigned int pad;
};

constexpr size_t kSmem2 = 1024 + (size_t)kStages2 * (kStageA2 + kStageB2) + sizeof(Barriers2) + kMaxN * 8 + 64;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared-memory address of the same object in CTA `rank` of the cluster.
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

// TMA load into this CTA's shared memory, completing on a barrier that may
// live in the peer CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int x, int y,
                                                 unsigned long long policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, unsigned long long adesc, unsigned long long bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at this offset in both CTAs once all prior MMAs are done.
__device__ __forceinline__ void mma_commit_pair(unsigned long long* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((unsigned short)3)
        : "memory");
}

__global__ void __launch_bounds__(kThreadsTc, 1)
    k_verify_tc2(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x, const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stage_a = smem;                                   // kStages2 x 16 KiB (this CTA's W rows)
    uint8_t* stage_b = smem + (size_t)kStages2 * kStageA2;     // kStages2 x 16 KiB (this CTA's hidden rows)
    Barriers2* bars = reinterpret_cast<Barriers2*>(stage_b + (size_t)kStages2 * kStageB2);
    unsigned long long* merge = reinterpret_cast<unsigned long long*>(bars + 1);  // [kMaxN]
    __shared__ unsigned int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    const int n_ptiles = (a.V + kPairM - 1) / kPairM;
    const int k_stages = a.H / kBlockK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tmem_full[b], 1);
            mbar_init(&bars->tmem_empty[b], 8);  // 4 epilogue warps in each CTA
        }
        mbar_init(&bars->mma_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    for (int i = threadIdx.x; i < kMaxN; i += blockDim.x) merge[i] = 0ull;
    if (warp == 1) {  // one warp in each CTA of the pair allocates the paired TMEM
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        if (lane == 0) {
            const unsigned long long pol_w = policy_evict_first();
            const unsigned long long pol_x = policy_evict_last();
            uint32_t it = 0;
            bool ok = true;
            for (int pt = pair; pt < n_ptiles && ok; pt += n_pairs) {
                for (int ks = 0; ks < k_stages; ++ks, ++it) {
                    const int s = it % kStages2;
                    if (!mbar_wait(&bars->empty[s], ((it / kStages2) & 1u) ^ 1u, a.err)) { ok = false; break; }
                    const uint32_t full_leader = map_to_rank(smem_u32(&bars->full[s]), 0);
                    if (leader) mbar_arrive_expect_tx(&bars->full[s], 2u * (uint32_t)(kStageA2 + kStageB2));
                    tma_load_2d_pair(stage_a + (size_t)s * kStageA2, &map_w, full_leader, ks * kBlockK,
                                     pt * kPairM + (int)rank * kBlockM, pol_w);
                    tma_load_2d_pair(stage_b + (size_t)s * kStageB2, &map_x, full_leader, ks * kBlockK,
                                     (int)rank * 128, pol_x);
                }
            }
            if (leader) {  // drain: the leader's barriers see both CTAs' loads
                const uint32_t issued = it;
                for (uint32_t j = (issued > (uint32_t)kStages2 ? issued - kStages2 : 0); j < issued; ++j)
                    mbar_drain(&bars->full[j % kStages2], (j / kStages2) & 1u);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader CTA only) ----------------
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_bf16(kPairM, 256);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int pt = pair; pt < n_ptiles && ok; pt += n_pairs, ++local) {
                const uint32_t buf = local & 1u;
                if (!mbar_wait(&bars->tmem_empty[buf], ((local >> 1) & 1u) ^ 1u, a.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * 256u;
                for (int ks = 0; ks < k_stages; ++ks, ++it) {
                    const int s = it % kStages2;
                    if (!mbar_wait(&bars->full[s], (it / kStages2) & 1u, a.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(stage_a + (size_t)s * kStageA2);
                    const uint32_t sb = smem_u32(stage_b + (size_t)s * kStageB2);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk)
                        mma_bf16_pair(d_tmem, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32), idesc,
                                      (ks > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_pair(&bars->empty[s]);
                }
                if (ok) mma_commit_pair(&bars->tmem_full[buf]);
            }
            mma_commit_pair(&bars->mma_done);
            mbar_drain(&bars->mma_done, 0u);
        }
    } else {
        // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
        const int quarter = warp & 3;
        float best_v[kMaxN / 32];
        uint32_t best_g[kMaxN / 32];
#pragma unroll
        for (int g = 0; g < kMaxN / 32; ++g) {
            best_v[g] = -__int_as_float(0x7f800000);
            best_g[g] = 0xFFFFFFFFu;
        }
        const uint32_t empty_leader0 = map_to_rank(smem_u32(&bars->tmem_empty[0]), 0);
        const uint32_t empty_leader1 = map_to_rank(smem_u32(&bars->tmem_empty[1]), 0);
        uint32_t local = 0;
        for (int pt = pair; pt < n_ptiles; pt += n_pairs, ++local) {
            const uint32_t buf = local & 1u;
            if (!mbar_wait(&bars->tmem_full[buf], (local >> 1) & 1u, a.err)) break;
            tc_fence_after();
            const uint32_t row0 = (uint32_t)(pt * kPairM + (int)rank * kBlockM + quarter * 32);
            const bool valid = (int)(row0 + lane) < a.V;
#pragma unroll
            for (int g = 0; g < kMaxN / 32; ++g) {
                float v[32];
                tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * 256u + g * 32u, v);
                if (g + 1 == kMaxN / 32) {  // accumulator fully read: release it to the leader's MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(buf ? empty_leader1 : empty_leader0);
                }
                float m;
                uint32_t bal;
                column_argmax32(v, valid, m, bal);
                if (bal != 0u && (best_g[g] == 0xFFFFFFFFu || m > best_v[g])) {
                    best_v[g] = m;
                    best_g[g] = row0 + (uint32_t)(__ffs(bal) - 1);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < kMaxN / 32; ++g)
            if (best_g[g] != 0xFFFFFFFFu && vh_guard(best_g[g] < (uint32_t)a.V, a.err))
                atomicMax(&merge[g * 32 + lane], make_key(best_v[g], best_g[g]));
    }

    // ---------------- pair teardown, publish, last-CTA decode ----------------
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still signal or read it
    if (warp == 1) {
        tc_fence_after();
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
        const uint32_t gid = key_gid(k);
        a.next_ids[r] = (int32_t)((a.cand != nullptr && gid < (uint32_t)a.V) ? (uint32_t)__ldg(a.cand + gid) : gid);
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
// Host side: tensor maps through the driver entry point (no libcuda link).

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

// 2-D bf16 row-major [rows][H] map with a [box_rows][64] box, 128 B swizzle.
static bool make_map(CUtensorMap* m, const void* base, int rows, int H, int box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBlockK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


// CTA-pair launch (R in 129..256): clusters of 2, grid = 2 x the resident clusters.
static cudaError_t launch_verify_tc2(const uint16_t* X, int R, int H, const uint16_t* W, int V, Workspace ws,
                                     int32_t* next_ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s,
                                     const int32_t* cand) {
    alignas(64) CUtensorMap map_w, map_x;
    if (!make_map(&map_w, W, V, H, kBlockM) || !make_map(&map_x, X, R, H, 128)) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(k_verify_tc2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem2);
    if (e != cudaSuccess) return e;
    TcArgs a{};
    a.R = R;
    a.N = 256;
    a.H = H;
    a.V = V;
    a.n_tiles = (V + kPairM - 1) / kPairM;
    a.ws = ws;
    a.err = ws.ticket + 1;
    a.next_ids = next_ids;
    a.maxlogit = maxlogit;
    a.tail = tail;
    a.cand = cand;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreadsTc);
    cfg.dynamicSmemBytes = kSmem2;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2u * (unsigned)std::max(1, std::min(sm_count() / 2, a.n_tiles)));
    static std::atomic<int> clusters_cache[64] = {};  // resident pairs, per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    int clusters = clusters_cache[dev & 63].load(std::memory_order_relaxed);
    if (clusters < 1) {
        if (cudaOccupancyMaxActiveClusters(&clusters, k_verify_tc2, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            return cudaErrorNotSupported;
        }
        clusters_cache[dev & 63].store(clusters, std::memory_order_relaxed);
    }
    cfg.gridDim = dim3(2u * (unsigned)std::max(1, std::min(clusters, a.n_tiles)));
    return cudaLaunchKernelEx(&cfg, k_verify_tc2, map_w, map_x, a);
}
}  // namespace tc

static cudaError_t launch_tc(const uint16_t* X, int R, int H, const uint16_t* W, int V, Workspace ws,
                             int32_t* next_ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s,
                             const int32_t* cand) {
    using namespace tc;
    if (R < 1 || R > kMaxN || H < kBlockK || H % kBlockK != 0 || V < 1) return cudaErrorNotSupported;
    if (R > 128) {
        cudaError_t e = launch_verify_tc2(X, R, H, W, V, ws, next_ids, maxlogit, tail, s, cand);
        if (e != cudaErrorNotSupported) return e;  // otherwise fall through to the single-CTA kernel
    }
    const int N = (R + 15) / 16 * 16;
    alignas(64) CUtensorMap map_w, map_x;
    if (!make_map(&map_w, W, V, H, kBlockM) || !make_map(&map_x, X, R, H, N)) return cudaErrorNotSupported;
    TcArgs a{};
    a.R = R;
    a.N = N;
    a.H = H;
    a.V = V;
    a.n_tiles = (V + kBlockM - 1) / kBlockM;
    a.ws = ws;
    a.err = ws.ticket + 1;
    a.next_ids = next_ids;
    a.maxlogit = maxlogit;
    a.tail = tail;
    a.cand = cand;
    const int grid = std::max(1, std::min(sm_count(), a.n_tiles));
    // ring depth by width: up to 64 hidden rows take eight stages (20 / 32 / 64 rows on the
    // 248,320 x 2048 head: 157.7-158.1 us against 158.1-160.1 with six and 165.9-167.9 with
    // four), 65-128 rows fit six (128 rows: 166.9 against 172-174 us with four)
    auto go = [&](auto kernel, size_t smem) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kThreadsTc);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, map_w, map_x, a);
    };
    if (N <= 64) return go(k_verify_tc<8, 64>, smem_bytes_tc(8, 64));
    if (N <= 128) return go(k_verify_tc<6, 128>, smem_bytes_tc(6, 128));
    return go(k_verify_tc<4, 256>, smem_bytes_tc(4, 256));
}

cudaError_t launch_verify_tc(const uint16_t* X, int R, int H, const uint16_t* W, int V, Workspace ws,
                             int32_t* next_ids, float* maxlogit, const AcceptTail& tail, cudaStream_t s) {
    return launch_tc(X, R, H, W, V, ws, next_ids, maxlogit, tail, s, nullptr);
}

cudaError_t launch_draft_tc(const uint16_t* x, int nb, int H, const uint16_t* W, const int32_t* cand, int n_rows,
                            Workspace ws, int32_t* ids, float* maxlogit, cudaStream_t s) {
    if (cand == nullptr) return cudaErrorNotSupported;
    return launch_tc(x, nb, H, W, n_rows, ws, ids, maxlogit, AcceptTail{}, s, cand);
}

}  // namespace vh
