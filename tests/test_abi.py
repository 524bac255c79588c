"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks return the documented status without launching (CPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "verifyhead.h")


@pytest.fixture(scope="module")
def vh():
    import verify_head_gb300 as vh
    vh.build()
    return vh


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^VH_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("mtp_draft_head_argmax", "mtp_draft_head_argmax_nvfp4", "spec_verify_greedy", "vh_workspace_bytes",
              "vh_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(vh):
    lib = ctypes.CDLL(vh.LIB_PATH)
    names = declared_symbols()
    assert names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(vh.EXPORTS) == names


def test_status_strings_and_workspace(vh):
    assert vh.lib().vh_version() >= 10000
    for st in range(-6, 1):
        assert vh.status_string(st)
    assert vh.status_string(-99) == "unknown status"
    assert vh.vh_workspace_bytes(0) == 0
    assert vh.vh_workspace_bytes(1) == 32
    assert vh.vh_workspace_bytes(256) == 256 * 8 + 16
    assert vh.vh_workspace_bytes(3) % 16 == 0
    assert vh.lib().vh_workspace_error_offset() == 4


# Fake, aligned, never-dereferenced addresses: argument checks run before any
# device access, so these calls return without touching memory.
P = 0x10000


def draft(vh, **kw):
    a = dict(hidden=P, W=P, cand=P, B=1, H=256, Vc=1024, ids=P, ml=P, ws=P, wsb=64, stream=None)
    a.update(kw)
    return vh.lib().mtp_draft_head_argmax(a["hidden"], a["W"], a["cand"], a["B"], a["H"], a["Vc"], a["ids"], a["ml"],
                                          a["ws"], a["wsb"], a["stream"])


def nvfp4(vh, **kw):
    a = dict(hidden=P, q=P, s=P, g=1.0, cand=P, B=1, H=256, Vc=1024, ids=P, ml=P, ws=P, wsb=64, stream=None)
    a.update(kw)
    return vh.lib().mtp_draft_head_argmax_nvfp4(a["hidden"], a["q"], a["s"], a["g"], a["cand"], a["B"], a["H"],
                                                a["Vc"], a["ids"], a["ml"], a["ws"], a["wsb"], a["stream"])


def verify(vh, **kw):
    a = dict(hidden=P, W=P, d=P, B=2, k=3, H=256, V=4096, acc=P, nid=P, ml=P, ws=P, wsb=1024, stream=None, path=0)
    a.update(kw)
    return vh.lib().spec_verify_greedy_path(a["hidden"], a["W"], a["d"], a["B"], a["k"], a["H"], a["V"], a["acc"],
                                            a["nid"], a["ml"], a["ws"], a["wsb"], a["stream"], a["path"])


def test_draft_argument_checks(vh):
    assert draft(vh, hidden=None) == vh.VH_ERR_NULL
    assert draft(vh, W=None) == vh.VH_ERR_NULL
    assert draft(vh, cand=None) == vh.VH_ERR_NULL
    assert draft(vh, ids=None) == vh.VH_ERR_NULL
    assert draft(vh, ml=None) == vh.VH_ERR_NULL
    assert draft(vh, ws=None) == vh.VH_ERR_NULL
    assert draft(vh, B=0) == vh.VH_ERR_SHAPE
    assert draft(vh, B=257) == vh.VH_ERR_SHAPE
    assert draft(vh, H=264) == vh.VH_ERR_SHAPE  # H % 16 != 0
    assert draft(vh, H=0) == vh.VH_ERR_SHAPE
    assert draft(vh, Vc=0) == vh.VH_ERR_SHAPE
    assert draft(vh, W=P + 16) == vh.VH_ERR_ALIGN  # W needs 32-byte alignment
    assert draft(vh, hidden=P + 8) == vh.VH_ERR_ALIGN
    assert draft(vh, wsb=16) == vh.VH_ERR_WORKSPACE


def test_nvfp4_argument_checks(vh):
    assert nvfp4(vh, q=None) == vh.VH_ERR_NULL
    assert nvfp4(vh, s=None) == vh.VH_ERR_NULL
    assert nvfp4(vh, H=272) == vh.VH_ERR_SHAPE  # H % 64 != 0
    assert nvfp4(vh, g=0.0) == vh.VH_ERR_SHAPE
    assert nvfp4(vh, g=float("nan")) == vh.VH_ERR_SHAPE
    assert nvfp4(vh, g=float("inf")) == vh.VH_ERR_SHAPE
    assert nvfp4(vh, q=P + 16) == vh.VH_ERR_ALIGN
    assert nvfp4(vh, wsb=8) == vh.VH_ERR_WORKSPACE


def test_verify_argument_checks(vh):
    assert verify(vh, d=None) == vh.VH_ERR_NULL
    assert verify(vh, acc=None) == vh.VH_ERR_NULL
    assert verify(vh, nid=None) == vh.VH_ERR_NULL
    assert verify(vh, k=0) == vh.VH_ERR_SHAPE
    assert verify(vh, k=16) == vh.VH_ERR_SHAPE
    assert verify(vh, B=0) == vh.VH_ERR_SHAPE
    assert verify(vh, B=20000, k=3) == vh.VH_ERR_SHAPE  # more than 65536 rows
    assert verify(vh, V=0) == vh.VH_ERR_SHAPE
    assert verify(vh, H=272, path=vh.VH_PATH_TENSOR) == vh.VH_ERR_SHAPE
    assert verify(vh, path=7) == vh.VH_ERR_SHAPE
    assert verify(vh, W=P + 16) == vh.VH_ERR_ALIGN
    assert verify(vh, ml=P + 2) == vh.VH_ERR_ALIGN
    assert verify(vh, wsb=vh.vh_workspace_bytes(8) - 1) == vh.VH_ERR_WORKSPACE


def verify4(vh, **kw):
    a = dict(hidden=P, q=P, s=P, g=1.0, d=P, B=8, k=3, H=512, V=4096, acc=P, nid=P, ml=P, ws=P, wsb=None, stream=None)
    a.update(kw)
    if a["wsb"] is None:
        a["wsb"] = vh.vh_verify_nvfp4_workspace_bytes(a["B"] * (a["k"] + 1), a["H"])
    return vh.lib().spec_verify_greedy_nvfp4(a["hidden"], a["q"], a["s"], a["g"], a["d"], a["B"], a["k"], a["H"],
                                             a["V"], a["acc"], a["nid"], a["ml"], a["ws"], a["wsb"], a["stream"])


def test_verify_nvfp4_workspace_size(vh):
    # argmax part, then rows*H*2 bytes of f16 rows and 4 bytes per row, each rounded up to 16
    assert vh.vh_verify_nvfp4_workspace_bytes(0, 512) == 0
    assert vh.vh_verify_nvfp4_workspace_bytes(4, 0) == 0
    assert vh.vh_verify_nvfp4_workspace_bytes(256, 2048) == vh.vh_workspace_bytes(256) + 256 * 2048 * 2 + 1024
    assert vh.vh_verify_nvfp4_workspace_bytes(3, 64) == vh.vh_workspace_bytes(3) + 384 + 16
    assert vh.vh_verify_nvfp4_workspace_bytes(5, 512) % 16 == 0


def test_verify_nvfp4_argument_checks(vh):
    assert verify4(vh, q=None) == vh.VH_ERR_NULL
    assert verify4(vh, ws=None) == vh.VH_ERR_NULL
    assert verify4(vh, H=520) == vh.VH_ERR_SHAPE  # H % 64 != 0
    assert verify4(vh, k=16) == vh.VH_ERR_SHAPE
    assert verify4(vh, g=-1.0) == vh.VH_ERR_SHAPE
    assert verify4(vh, q=P + 16) == vh.VH_ERR_ALIGN
    # the argmax-only workspace is too small: the f16 scratch is missing
    assert verify4(vh, wsb=vh.vh_workspace_bytes(32)) == vh.VH_ERR_WORKSPACE
    assert verify4(vh, wsb=vh.vh_verify_nvfp4_workspace_bytes(32, 512) - 1) == vh.VH_ERR_WORKSPACE


def test_valid_call_without_gpu_reports_device(vh):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the device check passes")
    assert draft(vh) == vh.VH_ERR_DEVICE
    assert verify(vh, ml=None) == vh.VH_ERR_DEVICE


def test_binding_refuses_cpu_tensors(vh):
    import torch
    x = torch.zeros(1, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        vh.mtp_draft_head_argmax(x, torch.zeros(4, 16, dtype=torch.bfloat16), torch.arange(4, dtype=torch.int32))


def test_debug_build_exports_the_same_symbols(vh):
    """The VH_DEBUG build (index guards) compiles and exports the same ABI."""
    from verify_head_gb300 import buildlib
    path = buildlib.build(debug=True)
    lib = ctypes.CDLL(path)
    for n in declared_symbols():
        assert hasattr(lib, n), n
