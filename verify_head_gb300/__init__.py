"""Python binding of libverifyhead.so (restricted-vocabulary MTP draft head and
greedy speculative verification, GB300 / sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  If the compiled
library is missing, every call raises: there is no fallback.

Entry points mirror the C ABI in include/verifyhead.h:
    mtp_draft_head_argmax, mtp_draft_head_argmax_nvfp4,
    spec_verify_greedy (spec_verify_greedy_path), vh_workspace_bytes.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libverifyhead.so")

VH_OK = 0
VH_ERR_NULL = -1
VH_ERR_SHAPE = -2
VH_ERR_ALIGN = -3
VH_ERR_WORKSPACE = -4
VH_ERR_LAUNCH = -5
VH_ERR_DEVICE = -6

VH_PATH_AUTO = 0
VH_PATH_CUDA_CORE = 1
VH_PATH_TENSOR = 2
VH_PATH_WARP_MMA = 3

# Every symbol the header declares (checked by the ABI tests).
EXPORTS = (
    "vh_version", "vh_status_string", "vh_workspace_bytes", "mtp_draft_head_argmax",
    "mtp_draft_head_argmax_nvfp4", "spec_verify_greedy", "spec_verify_greedy_path",
    "mtp_draft_head_argmax_static_ws", "mtp_draft_head_argmax_gather", "vh_workspace_error_offset",
    "vh_selftest_bounded_wait", "spec_verify_greedy_nvfp4", "vh_verify_nvfp4_workspace_bytes",
    "mtp_draft_head_argmax_nvfp4_path", "vh_nvfp4_packed_bytes", "vh_nvfp4_pack",
    "mtp_draft_head_argmax_nvfp4_packed", "spec_verify_greedy_nvfp4_packed",
)


class VHError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None
_debug_lib = None
_use_debug = False


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    from . import buildlib as _b
    return _b.build(force=force, verbose=verbose, debug=debug)


def _load(path: str):
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run verify_head_gb300.build() (nvcc, sm_103a)")
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def lib():
    """The loaded library (raises if it has not been built).  Inside
    `debug_library()` this is the VH_DEBUG build."""
    global _lib
    if _use_debug:
        return _debug_lib
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


@contextlib.contextmanager
def debug_library():
    """Route every call in the block through libverifyhead_debug.so (built on
    first use): the same kernels with device-side index guards that set bit 2
    of the workspace error word instead of touching memory out of range."""
    global _debug_lib, _use_debug
    if _debug_lib is None:
        from . import buildlib as _b
        _debug_lib = _load(_b.build(debug=True))
    prev, _use_debug = _use_debug, True
    try:
        yield _debug_lib
    finally:
        _use_debug = prev


def _declare(L):
    """ctypes signatures of every exported entry point."""
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.vh_version.restype = i32
    L.vh_version.argtypes = []
    L.vh_status_string.restype = ctypes.c_char_p
    L.vh_status_string.argtypes = [i32]
    L.vh_workspace_bytes.restype = sz
    L.vh_workspace_bytes.argtypes = [i32]
    L.mtp_draft_head_argmax.restype = i32
    L.mtp_draft_head_argmax.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp, sz, vp]
    L.mtp_draft_head_argmax_nvfp4.restype = i32
    L.mtp_draft_head_argmax_nvfp4.argtypes = [vp, vp, vp, ctypes.c_float, vp, i32, i32, i32, vp, vp, vp, sz, vp]
    L.spec_verify_greedy.restype = i32
    L.spec_verify_greedy.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    L.spec_verify_greedy_nvfp4.restype = i32
    L.spec_verify_greedy_nvfp4.argtypes = [vp, vp, vp, ctypes.c_float, vp, i32, i32, i32, i32, vp, vp, vp, vp, sz,
                                           vp]
    L.vh_workspace_error_offset.restype = sz
    L.vh_workspace_error_offset.argtypes = []
    L.vh_selftest_bounded_wait.restype = i32
    L.vh_selftest_bounded_wait.argtypes = [vp, ctypes.c_uint, vp]
    L.mtp_draft_head_argmax_gather.restype = i32
    L.mtp_draft_head_argmax_gather.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    L.mtp_draft_head_argmax_static_ws.restype = i32
    L.mtp_draft_head_argmax_static_ws.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp]
    L.vh_verify_nvfp4_workspace_bytes.restype = sz
    L.vh_verify_nvfp4_workspace_bytes.argtypes = [i32, i32]
    L.mtp_draft_head_argmax_nvfp4_path.restype = i32
    L.mtp_draft_head_argmax_nvfp4_path.argtypes = [vp, vp, vp, ctypes.c_float, vp, i32, i32, i32, vp, vp, vp, sz, vp,
                                                   i32]
    L.vh_nvfp4_packed_bytes.restype = sz
    L.vh_nvfp4_packed_bytes.argtypes = [i32, i32]
    L.vh_nvfp4_pack.restype = i32
    L.vh_nvfp4_pack.argtypes = [vp, vp, i32, i32, vp, sz, vp]
    L.mtp_draft_head_argmax_nvfp4_packed.restype = i32
    L.mtp_draft_head_argmax_nvfp4_packed.argtypes = [vp, vp, ctypes.c_float, vp, i32, i32, i32, vp, vp, vp, sz, vp]
    L.spec_verify_greedy_nvfp4_packed.restype = i32
    L.spec_verify_greedy_nvfp4_packed.argtypes = [vp, vp, ctypes.c_float, vp, i32, i32, i32, i32, vp, vp, vp, vp, sz,
                                                  vp]
    L.spec_verify_greedy_path.restype = i32
    L.spec_verify_greedy_path.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp, i32]


def status_string(status: int) -> str:
    return lib().vh_status_string(int(status)).decode()


def vh_workspace_bytes(rows: int) -> int:
    return int(lib().vh_workspace_bytes(int(rows)))


def vh_verify_nvfp4_workspace_bytes(rows: int, H: int) -> int:
    return int(lib().vh_verify_nvfp4_workspace_bytes(int(rows), int(H)))


def workspace_error(ws) -> int:
    """The error word of a workspace tensor: 0, or bit 1 (a bounded wait
    expired) and / or bit 2 (an index guard of the debug build fired) set by
    some call that used it.  Copies 4 bytes to the host (synchronising)."""
    off = int(lib().vh_workspace_error_offset())
    return int(ws[off:off + 4].cpu().view(__import__("torch").int32).item())


def _check(status: int, where: str):
    if status != VH_OK:
        raise VHError(status, where)


# ----------------------------------------------------------------------------
# torch-facing helpers (device memory and streams only).

def _torch():
    import torch
    return torch


def _ptr(t):
    # a plain int: the declared c_void_p argument types convert it
    return None if t is None else t.data_ptr()


_raw_stream = None  # torch's raw current-stream query, when this torch build has one


def _stream_ptr(stream):
    """cudaStream_t of `stream`, or of torch's current stream on the current device."""
    global _raw_stream
    torch = _torch()
    if stream is None:
        if _raw_stream is None:
            _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", False)
        if _raw_stream:
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("verify_head_gb300 takes CUDA tensors only")
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous (row-major)")


def workspace(rows: int, device=None):
    """A zeroed workspace for calls producing up to `rows` argmax rows."""
    torch = _torch()
    return torch.zeros(vh_workspace_bytes(rows), dtype=torch.uint8, device=device or "cuda")


def verify_nvfp4_workspace(rows: int, H: int, device=None):
    """A zeroed workspace for spec_verify_greedy_nvfp4 with `rows` hidden rows of width H."""
    torch = _torch()
    return torch.zeros(vh_verify_nvfp4_workspace_bytes(rows, H), dtype=torch.uint8, device=device or "cuda")


def mtp_draft_head_argmax(hidden, W_cand, cand_ids, ids=None, maxlogit=None, ws=None, stream=None):
    """hidden [B,H] bf16, W_cand [Vc,H] bf16, cand_ids [Vc] int32 -> (ids [B] int32, maxlogit [B] fp32)."""
    torch = _torch()
    _require_cuda(hidden, W_cand, cand_ids)
    B, H = hidden.shape
    Vc = W_cand.shape[0]
    if W_cand.shape[1] != H or cand_ids.numel() != Vc or hidden.element_size() != 2 or W_cand.element_size() != 2:
        raise ValueError("shape/dtype mismatch")
    if ids is None:
        ids = torch.empty(B, dtype=torch.int32, device=hidden.device)
    if maxlogit is None:
        maxlogit = torch.empty(B, dtype=torch.float32, device=hidden.device)
    if ws is None:
        ws = workspace(B, hidden.device)
    st = lib().mtp_draft_head_argmax(_ptr(hidden), _ptr(W_cand), _ptr(cand_ids), B, H, Vc, _ptr(ids), _ptr(maxlogit),
                                     _ptr(ws), ws.numel(), _stream_ptr(stream))
    _check(st, "mtp_draft_head_argmax")
    return ids, maxlogit


def mtp_draft_head_argmax_gather(hidden, W_full, row_ids, ids=None, maxlogit=None, ws=None, stream=None):
    """hidden [B,H] bf16, W_full [V,H] bf16, row_ids [n] int32 (rows of W_full to score, any order)
    -> (ids [B] int32 = winning row ids, maxlogit [B] fp32)."""
    torch = _torch()
    _require_cuda(hidden, W_full, row_ids)
    B, H = hidden.shape
    V = W_full.shape[0]
    if W_full.shape[1] != H or hidden.element_size() != 2 or W_full.element_size() != 2:
        raise ValueError("shape/dtype mismatch")
    if ids is None:
        ids = torch.empty(B, dtype=torch.int32, device=hidden.device)
    if maxlogit is None:
        maxlogit = torch.empty(B, dtype=torch.float32, device=hidden.device)
    if ws is None:
        ws = workspace(B, hidden.device)
    st = lib().mtp_draft_head_argmax_gather(_ptr(hidden), _ptr(W_full), _ptr(row_ids), B, H, row_ids.numel(), V,
                                            _ptr(ids), _ptr(maxlogit), _ptr(ws), ws.numel(), _stream_ptr(stream))
    _check(st, "mtp_draft_head_argmax_gather")
    return ids, maxlogit


def mtp_draft_head_argmax_nvfp4(hidden, Wq, scales, tensor_scale, cand_ids, ids=None, maxlogit=None, ws=None,
                                stream=None, path: int = VH_PATH_AUTO):
    """hidden [B,H] bf16, Wq [Vc,H/2] uint8, scales [Vc,H/16] uint8 (E4M3), tensor_scale float.
    `path` picks the kernel family (VH_PATH_AUTO / VH_PATH_CUDA_CORE / VH_PATH_TENSOR)."""
    torch = _torch()
    _require_cuda(hidden, Wq, scales, cand_ids)
    B, H = hidden.shape
    Vc = Wq.shape[0]
    if Wq.shape[1] * 2 != H or tuple(scales.shape) != (Vc, H // 16) or cand_ids.numel() != Vc:
        raise ValueError("shape mismatch")
    if ids is None:
        ids = torch.empty(B, dtype=torch.int32, device=hidden.device)
    if maxlogit is None:
        maxlogit = torch.empty(B, dtype=torch.float32, device=hidden.device)
    if ws is None:
        ws = workspace(B, hidden.device)
    st = lib().mtp_draft_head_argmax_nvfp4_path(_ptr(hidden), _ptr(Wq), _ptr(scales), float(tensor_scale),
                                                _ptr(cand_ids), B, H, Vc, _ptr(ids), _ptr(maxlogit), _ptr(ws),
                                                ws.numel(), _stream_ptr(stream), int(path))
    _check(st, "mtp_draft_head_argmax_nvfp4")
    return ids, maxlogit


def spec_verify_greedy(hidden, W_full, draft_ids, B: int, k: int, accept_len=None, next_ids=None, row_maxlogit=None,
                       ws=None, stream=None, path: int = VH_PATH_AUTO, want_maxlogit: bool = True):
    """hidden [B*(k+1),H] bf16, W_full [V,H] bf16, draft_ids [B,k] int32
    -> (accept_len [B], next_ids [B*(k+1)], row_maxlogit [B*(k+1)] or None).
    `path`: VH_PATH_AUTO / VH_PATH_CUDA_CORE / VH_PATH_TENSOR / VH_PATH_WARP_MMA."""
    torch = _torch()
    _require_cuda(hidden, W_full, draft_ids)
    R, H = hidden.shape
    V = W_full.shape[0]
    if R != B * (k + 1) or W_full.shape[1] != H or draft_ids.numel() != B * k:
        raise ValueError("shape mismatch")
    dev = hidden.device
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if next_ids is None:
        next_ids = torch.empty(R, dtype=torch.int32, device=dev)
    if row_maxlogit is None and want_maxlogit:
        row_maxlogit = torch.empty(R, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(R, dev)
    st = lib().spec_verify_greedy_path(_ptr(hidden), _ptr(W_full), _ptr(draft_ids), B, k, H, V, _ptr(accept_len),
                                       _ptr(next_ids), _ptr(row_maxlogit), _ptr(ws), ws.numel(), _stream_ptr(stream),
                                       int(path))
    _check(st, "spec_verify_greedy")
    return accept_len, next_ids, row_maxlogit


def spec_verify_greedy_nvfp4(hidden, Wq, scales, tensor_scale, draft_ids, B: int, k: int, accept_len=None,
                             next_ids=None, row_maxlogit=None, ws=None, stream=None, want_maxlogit: bool = True):
    """hidden [B*(k+1),H] bf16, Wq [V,H/2] uint8, scales [V,H/16] uint8, draft_ids [B,k] int32
    -> (accept_len [B], next_ids [B*(k+1)], row_maxlogit or None)."""
    torch = _torch()
    _require_cuda(hidden, Wq, scales, draft_ids)
    R, H = hidden.shape
    V = Wq.shape[0]
    if R != B * (k + 1) or Wq.shape[1] * 2 != H or tuple(scales.shape) != (V, H // 16) or draft_ids.numel() != B * k:
        raise ValueError("shape mismatch")
    dev = hidden.device
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if next_ids is None:
        next_ids = torch.empty(R, dtype=torch.int32, device=dev)
    if row_maxlogit is None and want_maxlogit:
        row_maxlogit = torch.empty(R, dtype=torch.float32, device=dev)
    if ws is None:
        ws = verify_nvfp4_workspace(R, H, dev)
    st = lib().spec_verify_greedy_nvfp4(_ptr(hidden), _ptr(Wq), _ptr(scales), float(tensor_scale), _ptr(draft_ids), B,
                                        k, H, V, _ptr(accept_len), _ptr(next_ids), _ptr(row_maxlogit), _ptr(ws),
                                        ws.numel(), _stream_ptr(stream))
    _check(st, "spec_verify_greedy_nvfp4")
    return accept_len, next_ids, row_maxlogit


def vh_nvfp4_packed_bytes(V: int, H: int) -> int:
    return int(lib().vh_nvfp4_packed_bytes(V, H))


def nvfp4_pack(Wq, scales, packed=None, stream=None):
    """Wq [V,H/2] uint8, scales [V,H/16] uint8 (row-major, CUDA) -> the tiled
    copy (uint8 CUDA tensor of vh_nvfp4_packed_bytes(V, H) bytes) that the
    *_nvfp4_packed calls read.  Done once per head (the weights are static)."""
    torch = _torch()
    _require_cuda(Wq, scales)
    V, H = Wq.shape[0], Wq.shape[1] * 2
    if tuple(scales.shape) != (V, H // 16):
        raise ValueError("shape mismatch")
    n = vh_nvfp4_packed_bytes(V, H)
    if n == 0:
        raise VHError(VH_ERR_SHAPE, "nvfp4_pack")
    if packed is None:
        packed = torch.empty(n, dtype=torch.uint8, device=Wq.device)
    st = lib().vh_nvfp4_pack(_ptr(Wq), _ptr(scales), V, H, _ptr(packed), packed.numel(), _stream_ptr(stream))
    _check(st, "vh_nvfp4_pack")
    return packed


def mtp_draft_head_argmax_nvfp4_packed(hidden, packed, tensor_scale, cand_ids, ids=None, maxlogit=None, ws=None,
                                       stream=None):
    """hidden [B,H] bf16, packed = nvfp4_pack(...) of the candidate table (Vc = cand_ids.numel() rows)."""
    torch = _torch()
    _require_cuda(hidden, packed, cand_ids)
    B, H = hidden.shape
    Vc = cand_ids.numel()
    if packed.numel() < vh_nvfp4_packed_bytes(Vc, H) or hidden.element_size() != 2:
        raise ValueError("shape mismatch")
    if ids is None:
        ids = torch.empty(B, dtype=torch.int32, device=hidden.device)
    if maxlogit is None:
        maxlogit = torch.empty(B, dtype=torch.float32, device=hidden.device)
    if ws is None:
        ws = workspace(B, hidden.device)
    st = lib().mtp_draft_head_argmax_nvfp4_packed(_ptr(hidden), _ptr(packed), float(tensor_scale), _ptr(cand_ids), B,
                                                  H, Vc, _ptr(ids), _ptr(maxlogit), _ptr(ws), ws.numel(),
                                                  _stream_ptr(stream))
    _check(st, "mtp_draft_head_argmax_nvfp4_packed")
    return ids, maxlogit


def spec_verify_greedy_nvfp4_packed(hidden, packed, tensor_scale, draft_ids, B: int, k: int, V: int, accept_len=None,
                                    next_ids=None, row_maxlogit=None, ws=None, stream=None,
                                    want_maxlogit: bool = True):
    """hidden [B*(k+1),H] bf16, packed = nvfp4_pack(...) of the full V-row head, draft_ids [B,k] int32
    -> (accept_len [B], next_ids [B*(k+1)], row_maxlogit or None)."""
    torch = _torch()
    _require_cuda(hidden, packed, draft_ids)
    R, H = hidden.shape
    if R != B * (k + 1) or draft_ids.numel() != B * k or packed.numel() < vh_nvfp4_packed_bytes(V, H):
        raise ValueError("shape mismatch")
    dev = hidden.device
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if next_ids is None:
        next_ids = torch.empty(R, dtype=torch.int32, device=dev)
    if row_maxlogit is None and want_maxlogit:
        row_maxlogit = torch.empty(R, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(R, dev)
    st = lib().spec_verify_greedy_nvfp4_packed(_ptr(hidden), _ptr(packed), float(tensor_scale), _ptr(draft_ids), B, k,
                                               H, V, _ptr(accept_len), _ptr(next_ids), _ptr(row_maxlogit), _ptr(ws),
                                               ws.numel(), _stream_ptr(stream))
    _check(st, "spec_verify_greedy_nvfp4_packed")
    return accept_len, next_ids, row_maxlogit
