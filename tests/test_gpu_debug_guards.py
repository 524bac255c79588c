"""The VH_DEBUG build (device-side index guards in place of a sanitizer): on
tiny, ragged and edge shapes every kernel family returns the oracle's answer
and leaves the workspace error word clear, i.e. no guard fired."""
import numpy as np
import pytest

from parity_util import TOL_4BIT, TOL_BF16, check_ids, to_torch, to_torch_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vh():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import verify_head_gb300 as vh
    vh.build()
    return vh


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="module")
def syn():
    import synth
    synth.build()
    return synth


def _err(vh, ws):
    return vh.workspace_error(ws)


@pytest.mark.parametrize("Vc,H,B", [(1, 16, 1), (7, 64, 2), (1025, 272, 3), (4099, 2048, 1)])
def test_debug_draft(vh, orc, syn, Vc, H, B):
    import torch
    W = syn.normal_bf16(Vc, 1, (Vc, H), 0.02)
    cand = syn.sorted_subset(Vc, 2, 248_320, Vc)
    x = syn.normal_bf16(B, 3, (B, H), 1.0)
    with vh.debug_library():
        ws = vh.workspace(B)
        ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(x), to_torch_bf16(W), to_torch(cand), ws=ws)
        torch.cuda.synchronize()
        assert _err(vh, ws) == 0
    o_ids, o_ml, o_sec = orc.draft_argmax(x, W, cand)

    def score_of(r, gid):
        return orc.dot_bf16(x[r], W[int(np.searchsorted(cand, gid))])

    check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec, score_of, TOL_BF16)


def test_debug_gather_with_skipped_ids(vh, orc, syn):
    """Out-of-range row ids are skipped by design: no guard may fire for them."""
    import torch
    V, H = 3000, 256
    W = syn.normal_bf16(V, 1, (V, H), 0.02)
    rows = np.concatenate([syn.sorted_subset(7, 2, V, 500), np.array([-5, V, V + 100], np.int32)]).astype(np.int32)
    x = syn.normal_bf16(8, 3, (1, H), 1.0)
    with vh.debug_library():
        ws = vh.workspace(1)
        ids, _ = vh.mtp_draft_head_argmax_gather(to_torch_bf16(x), to_torch_bf16(W), to_torch(rows), ws=ws)
        torch.cuda.synchronize()
        assert _err(vh, ws) == 0
    o_ids, _, _ = orc.draft_argmax_gather(x, W, rows)
    assert int(ids[0]) == int(o_ids[0])


@pytest.mark.parametrize("Vc,H,B", [(777, 128, 1), (3001, 1024, 1), (1500, 1024, 3), (1000, 512, 17)])
def test_debug_nvfp4_draft(vh, orc, syn, Vc, H, B):
    import torch
    cand = syn.sorted_subset(Vc, 2, 248_320, Vc)
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(Vc, 6, (Vc, H), 0.02))
    x = syn.normal_bf16(B, 3, (B, H), 1.0)
    with vh.debug_library():
        ws = vh.workspace(B)
        ids, ml = vh.mtp_draft_head_argmax_nvfp4(to_torch_bf16(x), to_torch(q), to_torch(s), g, to_torch(cand), ws=ws)
        torch.cuda.synchronize()
        assert _err(vh, ws) == 0
    o_ids, o_ml, o_sec = orc.draft_argmax_nvfp4(x, q, s, g, cand)

    def score_of(r, gid):
        c = int(np.searchsorted(cand, gid))
        return float(orc.scores_nvfp4(x[r], q[c:c + 1], s[c:c + 1], g, nthreads=1)[0])

    check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec, score_of, TOL_4BIT)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("B,k,V,H", [(3, 2, 129, 192), (43, 2, 900, 128), (64, 3, 1100, 256)])
def test_debug_verify(vh, orc, syn, path, B, k, V, H):
    import torch
    W = syn.normal_bf16(V + H, 1, (V, H), 0.02)
    X = syn.normal_bf16(B + k, 4, (B * (k + 1), H), 1.0)
    draft = np.zeros((B, k), np.int32)
    with vh.debug_library():
        ws = vh.workspace(B * (k + 1))
        _, nid, ml = vh.spec_verify_greedy(to_torch_bf16(X), to_torch_bf16(W), to_torch(draft), B, k, ws=ws,
                                           path=path)
        torch.cuda.synchronize()
        assert _err(vh, ws) == 0
    _, o_nid, o_ml, o_sec = orc.verify_greedy(X, W, None, B, k)
    check_ids(nid.cpu().numpy(), ml.cpu().numpy(), o_nid, o_ml, o_sec, lambda r, v: orc.dot_bf16(X[r], W[v]),
              TOL_BF16)


@pytest.mark.parametrize("B,k,V,H", [(4, 3, 1000, 512), (5, 3, 2000, 512), (33, 3, 2500, 512), (75, 3, 900, 512)])
def test_debug_verify_nvfp4(vh, orc, syn, B, k, V, H):
    import torch
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(V + H, 6, (V, H), 0.02))
    X = syn.normal_bf16(B + k, 4, (B * (k + 1), H), 1.0)
    draft = np.zeros((B, k), np.int32)
    with vh.debug_library():
        ws = vh.verify_nvfp4_workspace(B * (k + 1), H)
        _, nid, ml = vh.spec_verify_greedy_nvfp4(to_torch_bf16(X), to_torch(q), to_torch(s), g, to_torch(draft), B, k,
                                                 ws=ws)
        torch.cuda.synchronize()
        assert _err(vh, ws) == 0
    _, o_nid, o_ml, o_sec = orc.verify_greedy_nvfp4(X, q, s, g, None, B, k)

    def score_of(r, v):
        return float(orc.scores_nvfp4(X[r], q[v:v + 1], s[v:v + 1], g, nthreads=1)[0])

    check_ids(nid.cpu().numpy(), ml.cpu().numpy(), o_nid, o_ml, o_sec, score_of, TOL_4BIT)
