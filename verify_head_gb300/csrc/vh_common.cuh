// Device helpers shared by the head kernels: argmax keys, bf16 unpacking,
// streaming loads.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace vh {

constexpr int kThreads = 256;  // threads per CTA of the CUDA-core kernels
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------------------
// Argmax keys.  A (score, global id) pair is packed into one 64-bit word so
// that unsigned comparison orders first by score and then by LOWER id:
//   key = ord(score) << 32 | (0xFFFFFFFF - gid)
// ord() maps fp32 to a monotone uint32 (NaN -> -inf, -0 -> +0 first), so a
// 64-bit atomicMax merges partial argmaxes in any order with the same result.
// Key 0 never encodes a real pair and marks an empty slot.

__device__ __forceinline__ uint32_t ord_f32(float f) {
    if (f != f) f = -__int_as_float(0x7f800000);  // NaN -> -inf
    f = f + 0.0f;                                  // -0 -> +0
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float unord_f32(uint32_t o) {
    uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}

__device__ __forceinline__ unsigned long long make_key(float score, uint32_t gid) {
    return ((unsigned long long)ord_f32(score) << 32) | (unsigned long long)(0xFFFFFFFFu - gid);
}

__device__ __forceinline__ uint32_t key_gid(unsigned long long k) { return 0xFFFFFFFFu - (uint32_t)k; }
__device__ __forceinline__ float key_score(unsigned long long k) { return unord_f32((uint32_t)(k >> 32)); }

// ---------------------------------------------------------------------------
// 32-byte streaming load (one 256-bit access per lane): read-only path, no L1
// allocation, L2 evict-first.  Weights are read exactly once per call.

struct __align__(32) U32x8 {
    uint32_t v[8];
};

__device__ __forceinline__ U32x8 ld_stream32(const void* p) {
    U32x8 r;
    asm volatile(
        "ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]), "=r"(r.v[5]), "=r"(r.v[6]),
          "=r"(r.v[7])
        : "l"(p));
    return r;
}

// Low / high bf16 of a packed pair, widened exactly to fp32.
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// Workspace layout: a 16-byte header (uint32 ticket counter at byte 0, uint32
// error word at byte 4, 8 bytes unused) followed by keys[rows] (uint64).  The
// caller zeroes it once; every kernel leaves ticket and keys zeroed again.
// The error word is only ever set (bits below), never cleared by a kernel.

struct Workspace {
    unsigned long long* keys;
    unsigned int* ticket;  // ticket[1] is the error word
};

constexpr size_t kWsHeaderBytes = 16;
constexpr size_t kWsErrorOffset = 4;
__host__ __device__ constexpr size_t ws_keys_bytes(int rows) { return ((size_t)rows * 8 + 15) / 16 * 16; }
__host__ __device__ constexpr size_t ws_total_bytes(int rows) { return kWsHeaderBytes + ws_keys_bytes(rows); }
__host__ __device__ constexpr size_t round16(size_t n) { return (n + 15) / 16 * 16; }

// Error-word bits.  kErrTimeout: a bounded wait gave up.  kErrIndex: a
// device-side index guard of the VH_DEBUG build failed (the access was
// skipped).  In the normal build every guard is the constant `true`.
constexpr unsigned int kErrTimeout = 1u;
constexpr unsigned int kErrIndex = 2u;

#ifdef VH_DEBUG
__device__ __forceinline__ bool vh_guard(bool ok, unsigned int* err) {
    if (!ok) atomicOr(err, kErrIndex);
    return ok;
}
#else
__device__ __forceinline__ bool vh_guard(bool, unsigned int*) { return true; }
#endif

// Views of a workspace base pointer (the row count does not move anything).
__host__ __device__ inline Workspace ws_view(void* base) {
    Workspace w;
    w.ticket = static_cast<unsigned int*>(base);
    w.keys = reinterpret_cast<unsigned long long*>(static_cast<char*>(base) + kWsHeaderBytes);
    return w;
}

}  // namespace vh
