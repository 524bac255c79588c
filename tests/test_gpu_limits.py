"""Largest shapes the C ABI accepts (H = 65,536, B = 256 draft rows, k = 15),
each kernel family against the oracle, and the first shapes past the limits
refused on the host."""
import numpy as np
import pytest

from parity_util import TOL_4BIT, TOL_BF16, accept_scan, check_ids, to_torch, to_torch_bf16

pytestmark = pytest.mark.gpu

H_MAX = 65_536


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


@pytest.mark.parametrize("Vc,H,B", [(300, H_MAX, 1), (257, H_MAX, 3), (700, 256, 256)])
def test_draft_at_limits(vh, orc, syn, Vc, H, B):
    import torch
    W = syn.normal_bf16(Vc + 3, 1, (Vc, H), 0.02)
    cand = syn.sorted_subset(Vc, 2, 248_320, Vc)
    x = syn.normal_bf16(B + 5, 3, (B, H), 1.0)
    ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(x), to_torch_bf16(W), to_torch(cand))
    torch.cuda.synchronize()
    o_ids, o_ml, o_sec = orc.draft_argmax(x, W, cand)

    def score_of(r, gid):
        return orc.dot_bf16(x[r], W[int(np.searchsorted(cand, gid))])

    check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec, score_of, TOL_BF16)


@pytest.mark.parametrize("Vc,B", [(200, 1), (300, 2)])
def test_nvfp4_draft_at_max_width(vh, orc, syn, Vc, B):
    import torch
    cand = syn.sorted_subset(Vc, 2, 248_320, Vc)
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(Vc + 7, 6, (Vc, H_MAX), 0.02))
    x = syn.normal_bf16(B + 9, 3, (B, H_MAX), 1.0)
    ids, ml = vh.mtp_draft_head_argmax_nvfp4(to_torch_bf16(x), to_torch(q), to_torch(s), g, to_torch(cand))
    torch.cuda.synchronize()
    o_ids, o_ml, o_sec = orc.draft_argmax_nvfp4(x, q, s, g, cand)

    def score_of(r, gid):
        c = int(np.searchsorted(cand, gid))
        return float(orc.scores_nvfp4(x[r], q[c:c + 1], s[c:c + 1], g, nthreads=1)[0])

    check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec, score_of, TOL_4BIT)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("B,k,V", [(2, 1, 300), (1, 15, 200)])
def test_verify_at_max_width(vh, orc, syn, path, B, k, V):
    import torch
    W = syn.normal_bf16(V + 11, 1, (V, H_MAX), 0.02)
    X = syn.normal_bf16(B + 13, 4, (B * (k + 1), H_MAX), 1.0)
    draft = np.zeros((B, k), np.int32)
    acc, nid, ml = vh.spec_verify_greedy(to_torch_bf16(X), to_torch_bf16(W), to_torch(draft), B, k, path=path)
    torch.cuda.synchronize()
    _, o_nid, o_ml, o_sec = orc.verify_greedy(X, W, None, B, k)
    check_ids(nid.cpu().numpy(), ml.cpu().numpy(), o_nid, o_ml, o_sec, lambda r, v: orc.dot_bf16(X[r], W[v]),
              TOL_BF16)
    np.testing.assert_array_equal(acc.cpu().numpy(), accept_scan(nid.cpu().numpy(), draft, B, k))


def test_nvfp4_verify_pair_at_max_width(vh, orc, syn):
    """20 rows (the CTA-pair kernel, N = 128) over a 300 x 65,536 4-bit head."""
    import torch
    B, k, V = 5, 3, 300
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(V + 17, 6, (V, H_MAX), 0.02))
    X = syn.normal_bf16(B + 19, 4, (B * (k + 1), H_MAX), 1.0)
    draft = np.zeros((B, k), np.int32)
    acc, nid, ml = vh.spec_verify_greedy_nvfp4(to_torch_bf16(X), to_torch(q), to_torch(s), g, to_torch(draft), B, k)
    torch.cuda.synchronize()
    _, o_nid, o_ml, o_sec = orc.verify_greedy_nvfp4(X, q, s, g, None, B, k)

    def score_of(r, v):
        return float(orc.scores_nvfp4(X[r], q[v:v + 1], s[v:v + 1], g, nthreads=1)[0])

    check_ids(nid.cpu().numpy(), ml.cpu().numpy(), o_nid, o_ml, o_sec, score_of, TOL_4BIT)
    np.testing.assert_array_equal(acc.cpu().numpy(), accept_scan(nid.cpu().numpy(), draft, B, k))


def test_shapes_past_the_limits_are_refused(vh):
    import torch
    x = torch.zeros(1, H_MAX + 16, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(4, H_MAX + 16, dtype=torch.bfloat16, device="cuda")
    c = torch.arange(4, dtype=torch.int32, device="cuda")
    with pytest.raises(vh.VHError) as e:
        vh.mtp_draft_head_argmax(x, W, c)
    assert e.value.status == vh.VH_ERR_SHAPE
    x = torch.zeros(257, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vh.VHError) as e:
        vh.mtp_draft_head_argmax(x, W, c)
    assert e.value.status == vh.VH_ERR_SHAPE
    X = torch.zeros(17, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vh.VHError) as e:
        vh.spec_verify_greedy(X, W, torch.zeros(1, 16, dtype=torch.int32, device="cuda"), 1, 16)
    assert e.value.status == vh.VH_ERR_SHAPE
