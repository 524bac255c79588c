"""Seeded synthetic inputs for the draft head and the verify head.

This module generates inputs only: normal bf16 tensors, sorted candidate id
sets, the block-scaled 4-bit encoding of a normal fp32 head, and corrupted
draft ids.  It performs none of the head arithmetic (no scores, no argmax, no
acceptance scan) and is shared, unchanged, by the oracle tests, the CUDA
parity tests and the benchmark.

The workload recipes follow the head shapes of "少读一张大表，草稿路径才真正快起来"
(cnblogs, Qwen3.8 Flash dual-Spark tuning log): a 248,320-row full output head,
a 65,536-row candidate table and MTP3 (three draft tokens per round).  Those
pages built their candidate sets from a local corpus that is not available;
seeded uniformly random sorted subsets stand in for it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libvhsynth.so")

V_FULL = 248_320  # rows of the full output head (the pages' vocabulary)

# Stream ids: each kind of input draws from its own counter stream.
STREAM_W = 1
STREAM_CAND = 2
STREAM_HIDDEN = 3
STREAM_VHIDDEN = 4
STREAM_CORRUPT = 5
STREAM_W4 = 6
STREAM_DYN = 7

_lib = None


def build(force: bool = False) -> str:
    """Compile libvhsynth.so with gcc (portable C, no arch flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
             "-D_POSIX_C_SOURCE=200809L", _SRC, "-o", tmp, "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _nthreads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, i64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.vh_synth_normal_bf16.argtypes = [u64, u64, u64, i64, dbl, vp, i32]
        L.vh_synth_normal_f32.argtypes = [u64, u64, u64, i64, dbl, vp, i32]
        L.vh_synth_normal_bf16_rows.argtypes = [u64, u64, vp, i64, i64, dbl, vp, i32]
        L.vh_synth_sorted_subset.argtypes = [u64, u64, i64, i64, vp]
        L.vh_synth_sorted_subset.restype = i32
        L.vh_synth_corrupt_ids.argtypes = [u64, u64, vp, i64, ctypes.c_int32, dbl, vp]
        L.vh_synth_nvfp4_quantize.argtypes = [vp, i64, i64, vp, vp, ctypes.POINTER(ctypes.c_float), i32]
        L.vh_synth_nvfp4_quantize.restype = i32
        L.vh_synth_nvfp4_quantize_with_g.argtypes = [vp, i64, i64, ctypes.c_float, vp, vp, i32]
        L.vh_synth_nvfp4_quantize_with_g.restype = i32
        L.vh_synth_fingerprint.argtypes = [vp, i64]
        L.vh_synth_fingerprint.restype = u64
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------------------
# Primitive generators.

def normal_bf16(seed: int, stream: int, shape, sigma: float, offset: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of sigma * N(0, 1), element i = counter offset+i."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    lib().vh_synth_normal_bf16(seed, stream, offset, n, sigma, _ptr(out), _nthreads())
    return out.reshape(shape)


def normal_f32(seed: int, stream: int, shape, sigma: float, offset: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    lib().vh_synth_normal_f32(seed, stream, offset, n, sigma, _ptr(out), _nthreads())
    return out.reshape(shape)


def normal_bf16_rows(seed: int, stream: int, rows: np.ndarray, H: int, sigma: float) -> np.ndarray:
    """Rows `rows` of the [*, H] tensor normal_bf16(seed, stream, [*, H], sigma)."""
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    out = np.empty((rows.size, H), dtype=np.uint16)
    lib().vh_synth_normal_bf16_rows(seed, stream, _ptr(rows), rows.size, H, sigma, _ptr(out), _nthreads())
    return out


def sorted_subset(seed: int, stream: int, n_total: int, k: int) -> np.ndarray:
    """k distinct ids from [0, n_total), ascending (Floyd's sampling)."""
    out = np.empty(k, dtype=np.int32)
    rc = lib().vh_synth_sorted_subset(seed, stream, n_total, k, _ptr(out))
    if rc != 0:
        raise ValueError(f"sorted_subset failed ({rc})")
    return out


def corrupt_ids(seed: int, stream: int, truth: np.ndarray, V: int, p: float) -> np.ndarray:
    """Replace each id independently w.p. p by a uniform id from [0, V) minus the true id."""
    truth = np.ascontiguousarray(truth, dtype=np.int32)
    out = np.empty_like(truth)
    lib().vh_synth_corrupt_ids(seed, stream, _ptr(truth), truth.size, V, p, _ptr(out))
    return out


def nvfp4_quantize(w: np.ndarray, g: float | None = None):
    """Encode fp32 [rows, H] into (codes u8[rows, H/2], scales u8[rows, H/16], g)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, H = w.shape
    q = np.empty((rows, H // 2), dtype=np.uint8)
    s = np.empty((rows, H // 16), dtype=np.uint8)
    if g is None:
        gg = ctypes.c_float(0.0)
        rc = lib().vh_synth_nvfp4_quantize(_ptr(w), rows, H, _ptr(q), _ptr(s), ctypes.byref(gg), _nthreads())
        g = gg.value
    else:
        rc = lib().vh_synth_nvfp4_quantize_with_g(_ptr(w), rows, H, g, _ptr(q), _ptr(s), _nthreads())
    if rc != 0:
        raise ValueError("nvfp4_quantize: H must be a positive multiple of 16")
    return q, s, float(g)


def fingerprint(a: np.ndarray) -> int:
    a = np.ascontiguousarray(a)
    return int(lib().vh_synth_fingerprint(_ptr(a), a.nbytes))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# Workload recipes.  Each returns numpy arrays only.

@dataclass
class DraftCase:
    """Inputs of one draft-head workload: `steps` hidden batches of [B, H]."""
    name: str
    hidden: list            # list of uint16 [B, H] arrays (bf16 bits), one per draft step
    W: np.ndarray           # uint16 [Vc, H] candidate head (bf16 bits)
    cand_ids: np.ndarray    # int32 [Vc], ascending, distinct
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.hidden[0].shape[0]

    @property
    def H(self):
        return self.W.shape[1]

    @property
    def Vc(self):
        return self.W.shape[0]


@dataclass
class Nvfp4Case:
    name: str
    hidden: list            # list of uint16 [B, H]
    q: np.ndarray           # uint8 [Vc, H/2]
    s: np.ndarray           # uint8 [Vc, H/16]
    g: float
    cand_ids: np.ndarray    # int32 [Vc]
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.hidden[0].shape[0]

    @property
    def H(self):
        return self.q.shape[1] * 2

    @property
    def Vc(self):
        return self.q.shape[0]


@dataclass
class VerifyCase:
    """Verify inputs; draft_ids is None until the caller supplies the target's greedy ids."""
    name: str
    X: np.ndarray           # uint16 [B*(k+1), H]
    W: np.ndarray | None    # uint16 [V, H] (None when only a sample of rows is generated)
    B: int
    k: int
    V: int
    seed_w: int
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def H(self):
        return self.X.shape[1]

    def draft_ids_from(self, greedy_next_ids: np.ndarray, p: float = 0.45) -> np.ndarray:
        """Draft ids [B, k]: the greedy id of rows (b, j<k) corrupted w.p. p."""
        nid = np.asarray(greedy_next_ids, dtype=np.int32).reshape(self.B, self.k + 1)
        truth = np.ascontiguousarray(nid[:, : self.k])
        return corrupt_ids(self.seed, STREAM_CORRUPT, truth, self.V, p).reshape(self.B, self.k)


def draft_hidden(seed: int, steps: int, B: int, H: int) -> list:
    return [normal_bf16(seed, STREAM_HIDDEN, (B, H), 1.0, offset=s * B * H) for s in range(steps)]


def full_head(seed: int, V: int, H: int, sigma: float = 0.02) -> np.ndarray:
    return normal_bf16(seed, STREAM_W, (V, H), sigma)


def head_rows(seed: int, rows: np.ndarray, H: int, sigma: float = 0.02) -> np.ndarray:
    """Rows of full_head(seed, *, H) without generating the rest."""
    return normal_bf16_rows(seed, STREAM_W, rows, H, sigma)


def tiny_case():
    """Tiny check: V=4096 x H=256 head ~N(0, 0.02), 1,024 sorted candidates,
    B=1 x 3 draft steps, verify on B=1, k=3 (4 positions).  Seed 1."""
    seed, V, H, Vc = 1, 4096, 256, 1024
    W_full = full_head(seed, V, H)
    cand = sorted_subset(seed, STREAM_CAND, V, Vc)
    draft = DraftCase("tiny", draft_hidden(seed, 3, 1, H), np.ascontiguousarray(W_full[cand]), cand,
                      {"V": V, "seed": seed})
    X = normal_bf16(seed, STREAM_VHIDDEN, (4, H), 1.0)
    verify = VerifyCase("tiny-verify", X, W_full, 1, 3, V, seed, seed)
    return draft, verify, W_full


def draft_case(Vc: int = 65_536, H: int = 2048, B: int = 1, steps: int = 3, seed: int = 2,
               cand_seed: int | None = None, V: int = V_FULL) -> DraftCase:
    """Candidate draft head: Vc sorted distinct rows of the seeded V x H head
    (W_cand = W_full[cand_ids], a separate copy), `steps` fresh hidden batches."""
    cs = seed if cand_seed is None else cand_seed
    cand = sorted_subset(cs, STREAM_CAND, V, Vc) if Vc < V else np.arange(V, dtype=np.int32)
    W = head_rows(seed, cand, H)
    return DraftCase(f"draft-{Vc}x{H}-B{B}", draft_hidden(seed, steps, B, H), W, cand,
                     {"V": V, "seed": seed, "cand_seed": cs})


def verify_case(B: int = 64, k: int = 3, H: int = 2048, V: int = V_FULL, seed_w: int = 2, seed: int = 4,
                with_head: bool = True) -> VerifyCase:
    """Batched greedy verify: B sequences x (k+1) positions of hidden ~N(0,1)
    (seed `seed`) against the seeded V x H head (seed `seed_w`)."""
    X = normal_bf16(seed, STREAM_VHIDDEN, (B * (k + 1), H), 1.0)
    W = full_head(seed_w, V, H) if with_head else None
    return VerifyCase(f"verify-B{B}-k{k}-{V}x{H}", X, W, B, k, V, seed_w, seed)


def nvfp4_case(Vc: int = 65_536, H: int = 4096, B: int = 1, steps: int = 3, seed: int = 5,
               V: int = V_FULL) -> Nvfp4Case:
    """Block-scaled 4-bit draft head: fp32 N(0, 0.02) rows encoded as E2M1 codes,
    one E4M3 scale per 16 elements along H and one fp32 tensor scale."""
    cand = sorted_subset(seed, STREAM_CAND, V, Vc)
    w = normal_f32(seed, STREAM_W4, (Vc, H), 0.02)
    q, s, g = nvfp4_quantize(w)
    return Nvfp4Case(f"nvfp4-{Vc}x{H}-B{B}", draft_hidden(seed, steps, B, H), q, s, g, cand,
                     {"V": V, "seed": seed})


def nvfp4_head(seed: int = 2, V: int = V_FULL, H: int = 2048):
    """Block-scaled 4-bit full head: the fp32 N(0, 0.02) rows of stream W4
    (seed `seed`) encoded as in nvfp4_case -> (codes, scales, g)."""
    return nvfp4_quantize(normal_f32(seed, STREAM_W4, (V, H), 0.02))


def gather_row_ids(seed: int = 6, V: int = V_FULL, n_fixed: int = 32_768, n_dynamic: int = 16_384,
                   step: int = 0) -> np.ndarray:
    """Candidate rows read in place from the full head: a fixed sorted set of
    n_fixed ids followed by a per-step sorted set of n_dynamic ids (the two
    may overlap), as int32 [n_fixed + n_dynamic]."""
    fixed = sorted_subset(seed, STREAM_CAND, V, n_fixed)
    dyn = sorted_subset(seed * 1000 + step, STREAM_DYN, V, n_dynamic)
    return np.concatenate([fixed, dyn]).astype(np.int32)
