"""Failure detection without a GPU fault: a bounded wait that nothing
completes gives up, raises the flag, and the context stays usable."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vh():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import verify_head_gb300 as vh
    vh.build()
    return vh


def test_bounded_wait_times_out_and_context_survives(vh):
    import torch
    import synth
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = vh.lib().vh_selftest_bounded_wait(ctypes.c_void_p(flag.data_ptr()), 5000,
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == vh.VH_OK
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    # the context is still healthy: a normal call works and leaves no error
    case = synth.draft_case(Vc=4096, H=256, B=1, steps=1, seed=3)
    ws = vh.workspace(1)
    W = torch.from_numpy(case.W.view(np.int16)).cuda().view(torch.bfloat16)
    x = torch.from_numpy(case.hidden[0].view(np.int16)).cuda().view(torch.bfloat16)
    ids, _ = vh.mtp_draft_head_argmax(x, W, torch.from_numpy(case.cand_ids).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert int(ids.item()) in set(case.cand_ids.tolist())
    assert vh.workspace_error(ws) == 0


def test_selftest_argument_checks(vh):
    assert vh.lib().vh_selftest_bounded_wait(None, 10, None) == vh.VH_ERR_NULL
    assert vh.lib().vh_selftest_bounded_wait(ctypes.c_void_p(0x10002), 10, None) == vh.VH_ERR_ALIGN
    assert vh.lib().vh_selftest_bounded_wait(ctypes.c_void_p(0x10000), 0, None) == vh.VH_ERR_SHAPE
    assert vh.lib().vh_selftest_bounded_wait(ctypes.c_void_p(0x10000), 2_000_000, None) == vh.VH_ERR_SHAPE


def test_tensor_core_kernels_leave_error_word_clear(vh):
    import torch
    import synth
    V, H, B, k = 3000, 256, 64, 3
    W = torch.from_numpy(synth.normal_bf16(1, 1, (V, H), 0.02).view(np.int16)).cuda().view(torch.bfloat16)
    X = torch.from_numpy(synth.normal_bf16(2, 4, (B * (k + 1), H), 1.0).view(np.int16)).cuda().view(torch.bfloat16)
    d = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    ws = vh.workspace(B * (k + 1))
    vh.spec_verify_greedy(X, W, d, B, k, ws=ws, path=vh.VH_PATH_TENSOR)
    torch.cuda.synchronize()
    assert vh.workspace_error(ws) == 0
    assert int(ws.count_nonzero()) == 0
