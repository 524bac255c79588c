"""The draft-head entry point that allocates nothing.

mtp_draft_head_argmax_static_ws is for callers that cannot allocate device
memory or hand over a workspace (an engine's per-step hook or plugin API
with no allocator, a decode loop with a fixed memory plan).  It keeps its
scratch in a fixed array inside the library; this test checks, through the
C ABI, that two calls in a row return what the workspace-taking entry point
returns for the same inputs, and that a batch larger than the array's limit
is refused.  Collected last on purpose (file name), so that a failure here
comes after every other test has run.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import synth
    import verify_head_gb300 as vh
    vh.build()
    synth.build()
    return torch, vh, synth


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_static_scratch_matches_workspace_entry_point(env):
    torch, vh, synth = env
    L = vh.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    case = synth.draft_case(Vc=20_000, H=512, B=3, steps=2, seed=17)
    W = _dev(torch, case.W.view(np.int16))
    cand = _dev(torch, case.cand_ids)
    ws = torch.zeros(vh.vh_workspace_bytes(case.B), dtype=torch.uint8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    # two calls in a row with different hidden vectors (and a smaller batch on
    # the second), each checked against the workspace entry point
    for step, B in ((0, 3), (1, 1)):
        x = _dev(torch, case.hidden[step][:B].view(np.int16))
        ids_a = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        ml_a = torch.full((B,), float("nan"), dtype=torch.float32, device="cuda")
        ids_b = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        ml_b = torch.full((B,), float("nan"), dtype=torch.float32, device="cuda")
        st = L.mtp_draft_head_argmax_static_ws(p(x), p(W), p(cand), B, case.H, case.Vc, p(ids_a), p(ml_a), stream)
        assert st == vh.VH_OK, vh.status_string(st)
        st = L.mtp_draft_head_argmax(p(x), p(W), p(cand), B, case.H, case.Vc, p(ids_b), p(ml_b), p(ws), ws.numel(),
                                     stream)
        assert st == vh.VH_OK, vh.status_string(st)
        torch.cuda.synchronize()
        a_ids, b_ids = ids_a.cpu().numpy(), ids_b.cpu().numpy()
        a_ml, b_ml = ml_a.cpu().numpy(), ml_b.cpu().numpy()
        np.testing.assert_array_equal(a_ids, b_ids)
        assert np.all(np.abs(a_ml - b_ml) <= 2e-2)
        assert np.all(np.isin(a_ids, case.cand_ids))


def test_static_scratch_several_launch_groups_against_the_oracle(env):
    """20 hidden rows run as three launch groups (8 + 8 + 4) that share the
    array within one call, then 1 row: ids exact against the oracle where its
    top-1 / top-2 gap exceeds 1e-2 (inside that band an id scoring within 1e-2
    of the maximum), max logits within 2e-2, and equal to the workspace entry
    point."""
    import oracle
    from parity_util import TOL_BF16, check_ids
    torch, vh, synth = env
    oracle.build()
    L = vh.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    case = synth.draft_case(Vc=30_000, H=512, B=20, steps=2, seed=23)
    W = _dev(torch, case.W.view(np.int16))
    cand = _dev(torch, case.cand_ids)
    ws = torch.zeros(vh.vh_workspace_bytes(20), dtype=torch.uint8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    for step, B in ((0, 20), (1, 1)):
        xh = np.ascontiguousarray(case.hidden[step][:B])
        x = _dev(torch, xh.view(np.int16))
        ids_a = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        ml_a = torch.full((B,), float("nan"), dtype=torch.float32, device="cuda")
        ids_b = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        ml_b = torch.full((B,), float("nan"), dtype=torch.float32, device="cuda")
        st = L.mtp_draft_head_argmax_static_ws(p(x), p(W), p(cand), B, case.H, case.Vc, p(ids_a), p(ml_a), stream)
        assert st == vh.VH_OK, vh.status_string(st)
        st = L.mtp_draft_head_argmax(p(x), p(W), p(cand), B, case.H, case.Vc, p(ids_b), p(ml_b), p(ws), ws.numel(),
                                     stream)
        assert st == vh.VH_OK, vh.status_string(st)
        torch.cuda.synchronize()
        a_ids, a_ml = ids_a.cpu().numpy(), ml_a.cpu().numpy()
        np.testing.assert_array_equal(a_ids, ids_b.cpu().numpy())
        np.testing.assert_array_equal(a_ml, ml_b.cpu().numpy())
        o_ids, o_ml, o_sec = oracle.draft_argmax(xh, case.W, case.cand_ids)

        def score_of(r, gid):
            c = int(np.searchsorted(case.cand_ids, gid))
            assert case.cand_ids[c] == gid
            return oracle.dot_bf16(xh[r], case.W[c])

        check_ids(a_ids, a_ml, o_ids, o_ml, o_sec, score_of, TOL_BF16)


def test_static_scratch_rejects_batches_over_the_limit(env):
    torch, vh, _ = env
    L = vh.lib()
    x = torch.zeros(257, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    cand = torch.arange(8, dtype=torch.int32, device="cuda")
    ids = torch.zeros(257, dtype=torch.int32, device="cuda")
    ml = torch.zeros(257, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = L.mtp_draft_head_argmax_static_ws(p(x), p(W), p(cand), 257, 64, 8, p(ids), p(ml), None)
    assert st == vh.VH_ERR_WORKSPACE
