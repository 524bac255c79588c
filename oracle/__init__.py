"""CPU oracle for the draft head and the greedy verify head.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it to check and to time against; the CUDA
library never imports, links or calls it, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp32 sequential sums of the
bf16 / 4-bit-decoded values, first maximum wins).  This file only compiles it
and marshals numpy arrays.

Parity status per function (what pins it; see tests/test_oracle_pins.py):
  draft_argmax        exact-integer brute force, fp64 brute force, numpy fp64
                      matmul on the tiny workload, restricted-vs-full
                      invariant, closed-form special cases
  draft_argmax_nvfp4  exhaustive E2M1/E4M3 tables (closed form and torch's
                      float8_e4m3fn), fp64 brute force with exact rational
                      decoding, nibble/scale-order fixtures, equality with
                      draft_argmax on an exactly representable head
  draft_argmax_gather exact-integer brute force with unsorted and repeated
                      ids, equality with draft_argmax on the sorted set
  verify_greedy_nvfp4 equality with verify_greedy on an exactly representable
                      head (g = 1), hand-built acceptance fixtures
  verify_greedy       exact-integer brute force, hand-built acceptance
                      fixtures (tests/golden/accept_cases.txt), equality with
                      draft_argmax over the identity candidate set
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so (portable C; fp contraction off for cross-arch equality)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
             _SRC, "-o", tmp, "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


def threads() -> int:
    """Host cores available to this process (the oracle's thread count)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, i32, vp, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
        L.vh_oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.vh_oracle_bf16_to_f32.restype = f32
        L.vh_oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        L.vh_oracle_e2m1_value.restype = f32
        L.vh_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.vh_oracle_e4m3_value.restype = f32
        L.vh_oracle_dot_bf16.argtypes = [vp, vp, i64]
        L.vh_oracle_dot_bf16.restype = f32
        L.vh_oracle_dot_nvfp4.argtypes = [vp, vp, vp, f32, i64]
        L.vh_oracle_dot_nvfp4.restype = f32
        L.vh_oracle_draft_argmax.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp, i32]
        L.vh_oracle_draft_argmax.restype = i32
        L.vh_oracle_draft_argmax_nvfp4.argtypes = [vp, vp, vp, f32, vp, i64, i64, i64, vp, vp, vp, i32]
        L.vh_oracle_draft_argmax_nvfp4.restype = i32
        L.vh_oracle_draft_argmax_gather.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp, vp, i32]
        L.vh_oracle_draft_argmax_gather.restype = i32
        L.vh_oracle_accept_len.argtypes = [vp, vp, i64]
        L.vh_oracle_accept_len.restype = ctypes.c_int32
        L.vh_oracle_verify_greedy.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, i64, vp, vp, vp, vp, i32]
        L.vh_oracle_verify_greedy.restype = i32
        L.vh_oracle_verify_greedy_nvfp4.argtypes = [vp, vp, vp, f32, vp, i64, i64, i64, i64, vp, i64, vp, vp, vp,
                                                    vp, i32]
        L.vh_oracle_verify_greedy_nvfp4.restype = i32
        L.vh_oracle_scores_bf16.argtypes = [vp, vp, i64, i64, vp, i32]
        L.vh_oracle_scores_nvfp4.argtypes = [vp, vp, vp, f32, i64, i64, vp, i32]
        L.vh_oracle_decode_nvfp4.argtypes = [vp, vp, f32, i64, i64, vp]
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def bf16_to_f32(bits: int) -> float:
    return float(lib().vh_oracle_bf16_to_f32(int(bits)))


def e2m1_value(code: int) -> float:
    return float(lib().vh_oracle_e2m1_value(int(code)))


def e4m3_value(code: int) -> float:
    return float(lib().vh_oracle_e4m3_value(int(code)))


def dot_bf16(x, w) -> float:
    x, px = _c(x, np.uint16)
    w, pw = _c(w, np.uint16)
    assert x.size == w.size
    return float(lib().vh_oracle_dot_bf16(px, pw, x.size))


def draft_argmax(x, W, cand_ids, nthreads: int | None = None):
    """x uint16 [B,H], W uint16 [Vc,H], cand_ids int32 [Vc] -> (ids, maxlogit, second)."""
    x, px = _c(x, np.uint16)
    W, pW = _c(W, np.uint16)
    cand, pc = _c(cand_ids, np.int32)
    B, H = x.shape
    Vc = W.shape[0]
    assert W.shape[1] == H and cand.size == Vc
    ids = np.empty(B, np.int32)
    ml = np.empty(B, np.float32)
    sec = np.empty(B, np.float32)
    rc = lib().vh_oracle_draft_argmax(px, pW, pc, B, H, Vc, ids.ctypes.data, ml.ctypes.data, sec.ctypes.data,
                                      nthreads or threads())
    if rc != 0:
        raise ValueError(f"oracle draft_argmax failed ({rc})")
    return ids, ml, sec


def draft_argmax_nvfp4(x, q, s, g, cand_ids, nthreads: int | None = None):
    x, px = _c(x, np.uint16)
    q, pq = _c(q, np.uint8)
    s, ps = _c(s, np.uint8)
    cand, pc = _c(cand_ids, np.int32)
    B, H = x.shape
    Vc = q.shape[0]
    assert q.shape[1] * 2 == H and s.shape == (Vc, H // 16) and cand.size == Vc
    ids = np.empty(B, np.int32)
    ml = np.empty(B, np.float32)
    sec = np.empty(B, np.float32)
    rc = lib().vh_oracle_draft_argmax_nvfp4(px, pq, ps, float(g), pc, B, H, Vc, ids.ctypes.data, ml.ctypes.data,
                                            sec.ctypes.data, nthreads or threads())
    if rc != 0:
        raise ValueError(f"oracle draft_argmax_nvfp4 failed ({rc})")
    return ids, ml, sec


def draft_argmax_gather(x, W_full, row_ids, nthreads: int | None = None):
    """x uint16 [B,H], W_full uint16 [V,H], row_ids int32 [n] -> (ids, maxlogit, second)."""
    x, px = _c(x, np.uint16)
    W, pW = _c(W_full, np.uint16)
    r, pr = _c(row_ids, np.int32)
    B, H = x.shape
    V = W.shape[0]
    assert W.shape[1] == H
    ids = np.empty(B, np.int32)
    ml = np.empty(B, np.float32)
    sec = np.empty(B, np.float32)
    rc = lib().vh_oracle_draft_argmax_gather(px, pW, pr, B, H, r.size, V, ids.ctypes.data, ml.ctypes.data,
                                             sec.ctypes.data, nthreads or threads())
    if rc != 0:
        raise ValueError(f"oracle draft_argmax_gather failed ({rc})")
    return ids, ml, sec


def accept_len(next_ids_b, draft_b) -> int:
    n, pn = _c(next_ids_b, np.int32)
    d, pd = _c(draft_b, np.int32)
    return int(lib().vh_oracle_accept_len(pn, pd, d.size))


def verify_greedy(X, W, draft_ids, B: int, k: int, rows=None, nthreads: int | None = None):
    """X uint16 [B*(k+1),H], W uint16 [V,H], draft_ids int32 [B,k] (may be None)
    -> (accept_len [B] or None, next_ids [R], maxlogit [R], second [R]).

    With `rows`, only those rows are scored (entries for other rows are -1 /
    NaN) and accept_len is None."""
    X, pX = _c(X, np.uint16)
    W, pW = _c(W, np.uint16)
    R, H = X.shape
    V = W.shape[0]
    assert R == B * (k + 1) and W.shape[1] == H
    if draft_ids is not None:
        d, pd = _c(draft_ids, np.int32)
        assert d.size == B * k
    else:
        d, pd = None, None
    nid = np.full(R, -1, np.int32)
    ml = np.full(R, np.nan, np.float32)
    sec = np.full(R, np.nan, np.float32)
    acc = np.empty(B, np.int32)
    if rows is not None:
        rr, pr = _c(rows, np.int32)
        nr = rr.size
    else:
        rr, pr, nr = None, None, 0
    rc = lib().vh_oracle_verify_greedy(pX, pW, pd, B, k, H, V, pr, nr, nid.ctypes.data, acc.ctypes.data,
                                       ml.ctypes.data, sec.ctypes.data, nthreads or threads())
    if rc != 0:
        raise ValueError(f"oracle verify_greedy failed ({rc})")
    return (acc if (rows is None and d is not None) else None), nid, ml, sec


def verify_greedy_nvfp4(X, q, s, g, draft_ids, B: int, k: int, rows=None, nthreads: int | None = None):
    """As verify_greedy with the 4-bit head (q [V,H/2], s [V,H/16], g)."""
    X, pX = _c(X, np.uint16)
    q, pq = _c(q, np.uint8)
    s, ps = _c(s, np.uint8)
    R, H = X.shape
    V = q.shape[0]
    assert R == B * (k + 1) and q.shape[1] * 2 == H and s.shape == (V, H // 16)
    if draft_ids is not None:
        d, pd = _c(draft_ids, np.int32)
    else:
        d, pd = None, None
    nid = np.full(R, -1, np.int32)
    ml = np.full(R, np.nan, np.float32)
    sec = np.full(R, np.nan, np.float32)
    acc = np.empty(B, np.int32)
    if rows is not None:
        rr, pr = _c(rows, np.int32)
        nr = rr.size
    else:
        rr, pr, nr = None, None, 0
    rc = lib().vh_oracle_verify_greedy_nvfp4(pX, pq, ps, float(g), pd, B, k, H, V, pr, nr, nid.ctypes.data,
                                             acc.ctypes.data, ml.ctypes.data, sec.ctypes.data, nthreads or threads())
    if rc != 0:
        raise ValueError(f"oracle verify_greedy_nvfp4 failed ({rc})")
    return (acc if (rows is None and d is not None) else None), nid, ml, sec


def scores_bf16(x_row, W, nthreads: int | None = None):
    x, px = _c(x_row, np.uint16)
    W, pW = _c(W, np.uint16)
    out = np.empty(W.shape[0], np.float32)
    lib().vh_oracle_scores_bf16(px, pW, W.shape[0], W.shape[1], out.ctypes.data, nthreads or threads())
    return out


def scores_nvfp4(x_row, q, s, g, nthreads: int | None = None):
    x, px = _c(x_row, np.uint16)
    q, pq = _c(q, np.uint8)
    s, ps = _c(s, np.uint8)
    out = np.empty(q.shape[0], np.float32)
    lib().vh_oracle_scores_nvfp4(px, pq, ps, float(g), q.shape[0], q.shape[1] * 2, out.ctypes.data,
                                 nthreads or threads())
    return out


def decode_nvfp4(q, s, g):
    q, pq = _c(q, np.uint8)
    s, ps = _c(s, np.uint8)
    n, H = q.shape[0], q.shape[1] * 2
    out = np.empty((n, H), np.float32)
    lib().vh_oracle_decode_nvfp4(pq, ps, float(g), n, H, out.ctypes.data)
    return out
