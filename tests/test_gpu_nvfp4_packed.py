"""The 4-bit head in the tiled layout (vh_nvfp4_pack + *_nvfp4_packed) against
the oracle, which reads the row-major codes and scales.

The layout is a pure permutation of the row-major bytes, so the pack is
checked byte for byte against a numpy restatement of the documented layout;
scores, ids and accept lengths are checked against the oracle under the
usual rules (ids exact where the top-1 / top-2 gap exceeds 1e-2, max logit
within 5e-2), plus exact ties on integer-valued heads.
"""
import numpy as np
import pytest

from parity_util import TOL_4BIT, accept_scan, check_accept, check_ids, to_torch, to_torch_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vh():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import verify_head_gb300 as vh
    vh.build()
    vh.lib()
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


def pack_numpy(q, s):
    """The tiled layout written out with numpy: records of 16 rows x 256
    elements; [h][lane][32 code bytes] then [lane][h][4 scale bytes]."""
    V, H = q.shape[0], q.shape[1] * 2
    nb, KS = (V + 15) // 16, H // 256
    qp = np.zeros((nb * 16, H // 2), np.uint8)
    sp = np.zeros((nb * 16, H // 16), np.uint8)
    qp[:V], sp[:V] = q, s
    # row 16b + L/4 + 8h, code bytes 128t + 32(L%4) + [0, 32)
    qr = qp.reshape(nb, 2, 8, KS, 4, 32)             # [b][h][r][t][g][byte]
    codes = qr.transpose(0, 3, 1, 2, 4, 5).reshape(nb, KS, 2048)
    sr = sp.reshape(nb, 2, 8, KS, 4, 4)              # [b][h][r][t][g][scale]
    scales = sr.transpose(0, 3, 2, 4, 1, 5).reshape(nb, KS, 256)  # [b][t][lane = r*4+g][h][4]
    return np.concatenate([codes, scales], axis=2).reshape(-1)


def packed_of(vh, q, s):
    return vh.nvfp4_pack(to_torch(q), to_torch(s))


@pytest.mark.parametrize("V,H", [(1, 256), (17, 512), (1000, 1024), (4099, 4096), (33, 6144)])
def test_pack_layout_bytes(vh, syn, V, H):
    import torch
    q, s, _ = syn.nvfp4_quantize(syn.normal_f32(V, 6, (V, H), 0.02))
    p = packed_of(vh, q, s)
    torch.cuda.synchronize()
    assert p.numel() == vh.vh_nvfp4_packed_bytes(V, H) == (V + 15) // 16 * 9 * H
    np.testing.assert_array_equal(p.cpu().numpy(), pack_numpy(q, s))


def run_packed(vh, x, P, g, cand):
    import torch
    ids, ml = vh.mtp_draft_head_argmax_nvfp4_packed(to_torch_bf16(x), P, g, to_torch(cand))
    torch.cuda.synchronize()
    return ids.cpu().numpy(), ml.cpu().numpy()


def check_packed(vh, orc, x, q, s, g, cand, P=None):
    P = packed_of(vh, q, s) if P is None else P
    g_ids, g_ml = run_packed(vh, x, P, g, cand)
    o_ids, o_ml, o_sec = orc.draft_argmax_nvfp4(x, q, s, g, cand)

    def score_of(r, gid):
        c = int(np.searchsorted(cand, gid))
        assert cand[c] == gid
        return float(orc.scores_nvfp4(x[r], q[c:c + 1], s[c:c + 1], g, nthreads=1)[0])

    check_ids(g_ids, g_ml, o_ids, o_ml, o_sec, score_of, TOL_4BIT)
    return g_ids, g_ml


# one partial block; fewer blocks than warps; every KS from 1 to 24; B = 1,
# 8, 9 (two n8 tiles), 16, 17 and 40 (several passes); ragged last blocks
@pytest.mark.parametrize("Vc,H,B", [(1, 256, 1), (5, 4096, 3), (17, 2048, 2), (100, 1024, 8), (2049, 512, 9),
                                    (33, 256, 24), (3001, 768, 16), (70_001, 4096, 1), (4097, 6144, 5),
                                    (1500, 1280, 17), (20_000, 256, 40), (12_345, 4096, 8)])
def test_packed_draft_shapes(vh, orc, syn, Vc, H, B):
    cand = syn.sorted_subset(Vc + 1, 2, 248_320, Vc)
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(Vc + 2, 6, (Vc, H), 0.02))
    x = syn.normal_bf16(B + 3, 3, (B, H), 1.0)
    check_packed(vh, orc, x, q, s, g, cand)


@pytest.mark.parametrize("B", [1, 8, 16])
def test_packed_draft_full_size_65536x4096(vh, orc, syn, B):
    """The 4-bit draft workload (65,536 x 4096), three steps."""
    case = syn.nvfp4_case(Vc=65_536, H=4096, B=B, steps=3, seed=5)
    P = packed_of(vh, case.q, case.s)
    for x in case.hidden:
        check_packed(vh, orc, x, case.q, case.s, case.g, case.cand_ids, P=P)


def test_packed_equals_row_major_kernels(vh, syn):
    """Same table, row-major and tiled: ids agree outside near-ties and max
    logits agree to rounding."""
    import torch
    Vc, H, B = 9000, 2048, 8
    cand = syn.sorted_subset(77, 2, 248_320, Vc)
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(78, 6, (Vc, H), 0.02))
    x = syn.normal_bf16(79, 3, (B, H), 1.0)
    a_ids, a_ml = run_packed(vh, x, packed_of(vh, q, s), g, cand)
    b_ids, b_ml = vh.mtp_draft_head_argmax_nvfp4(to_torch_bf16(x), to_torch(q), to_torch(s), g, to_torch(cand))
    torch.cuda.synchronize()
    assert np.max(np.abs(a_ml - b_ml.cpu().numpy())) < 1e-3
    assert np.mean(a_ids == b_ids.cpu().numpy()) > 0.8


def test_packed_ties_lowest_id(vh, orc, syn):
    """Duplicate top rows in different blocks, warps and CTAs, and inside one
    block: every hidden row gets the lowest candidate id among them."""
    Vc, H, B = 40_000, 1024, 12
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(11, 6, (Vc, H), 0.02))
    top = [30_007, 39, 39_999, 2048, 47, 40, 16 * 17 + 3]
    q[top] = 0x77  # +6 in every element
    s[top] = 0x7E  # scale 448
    cand = syn.sorted_subset(12, 2, 248_320, Vc)
    x = np.full((B, H), 0x3F80, np.uint16)  # +1.0
    ids, ml = run_packed(vh, x, packed_of(vh, q, s), g, cand)
    assert list(ids) == [int(cand[min(top)])] * B
    o_ids, o_ml, _ = orc.draft_argmax_nvfp4(x, q, s, g, cand)
    assert list(o_ids) == list(ids)
    np.testing.assert_allclose(ml, o_ml, rtol=0, atol=TOL_4BIT)


def run_verify_packed(vh, X, P, g, draft, B, k, V):
    import torch
    acc, nid, ml = vh.spec_verify_greedy_nvfp4_packed(to_torch_bf16(X), P, g, to_torch(draft), B, k, V)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nid.cpu().numpy(), ml.cpu().numpy()


# 1 / 4 sequences: one pass (4 / 16 rows); 5 / 20: several passes, the scan in the last
@pytest.mark.parametrize("B,k,V,H", [(1, 3, 3001, 512), (4, 3, 2000, 1024), (5, 3, 1500, 256), (20, 3, 900, 2048),
                                     (2, 15, 700, 512)])
def test_packed_verify_shapes(vh, orc, syn, B, k, V, H):
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(V + H, 6, (V, H), 0.02))
    X = syn.normal_bf16(B + k, 4, (B * (k + 1), H), 1.0)
    _, o_nid, o_ml, o_sec = orc.verify_greedy_nvfp4(X, q, s, g, None, B, k)
    draft = syn.corrupt_ids(V, syn.STREAM_CORRUPT, o_nid.reshape(B, k + 1)[:, :k].copy(), V, 0.45)
    o_acc = np.array([orc.accept_len(o_nid[b * (k + 1): b * (k + 1) + k], draft[b]) for b in range(B)], np.int32)
    g_acc, g_nid, g_ml = run_verify_packed(vh, X, packed_of(vh, q, s), g, draft, B, k, V)
    check_ids(g_nid, g_ml, o_nid, o_ml, o_sec,
              lambda r, v: float(orc.scores_nvfp4(X[r], q[v:v + 1], s[v:v + 1], g, nthreads=1)[0]), TOL_4BIT)
    check_accept(g_acc, g_nid, o_acc, o_ml, o_sec, draft, B, k)
    np.testing.assert_array_equal(g_acc, accept_scan(g_nid, draft, B, k))


def test_packed_verify_65536x4096(vh, orc, syn):
    """4 sequences x 4 positions against the 65,536 x 4096 4-bit head."""
    c = syn.nvfp4_case(Vc=65_536, H=4096, B=1, steps=1, seed=5)
    X = syn.normal_bf16(7, syn.STREAM_VHIDDEN, (16, 4096), 1.0)
    B, k, V = 4, 3, 65_536
    _, o_nid, o_ml, o_sec = orc.verify_greedy_nvfp4(X, c.q, c.s, c.g, None, B, k)
    draft = syn.corrupt_ids(7, syn.STREAM_CORRUPT, o_nid.reshape(B, k + 1)[:, :k].copy(), V, 0.45)
    o_acc = np.array([orc.accept_len(o_nid[b * (k + 1): b * (k + 1) + k], draft[b]) for b in range(B)], np.int32)
    g_acc, g_nid, g_ml = run_verify_packed(vh, X, packed_of(vh, c.q, c.s), c.g, draft, B, k, V)
    check_ids(g_nid, g_ml, o_nid, o_ml, o_sec,
              lambda r, v: float(orc.scores_nvfp4(X[r], c.q[v:v + 1], c.s[v:v + 1], c.g, nthreads=1)[0]), TOL_4BIT)
    check_accept(g_acc, g_nid, o_acc, o_ml, o_sec, draft, B, k)


def test_packed_chain_and_graph_replay(vh, orc, syn):
    """The 4-bit draft chain on the tiled head (three calls back to back, then
    the same chain as a CUDA graph) against the oracle."""
    import torch
    B = 8
    case = syn.nvfp4_case(Vc=65_536, H=4096, B=B, steps=3, seed=5)
    P, cd = packed_of(vh, case.q, case.s), to_torch(case.cand_ids)
    xs = [to_torch_bf16(h) for h in case.hidden]
    ws = vh.workspace(B)
    ids = [torch.empty(B, dtype=torch.int32, device="cuda") for _ in range(3)]
    mls = [torch.empty(B, dtype=torch.float32, device="cuda") for _ in range(3)]

    def calls():
        for i in range(3):
            vh.mtp_draft_head_argmax_nvfp4_packed(xs[i], P, case.g, cd, ids=ids[i], maxlogit=mls[i], ws=ws)

    calls()
    torch.cuda.synchronize()
    runs = [[t.cpu().numpy().copy() for t in ids + mls]]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    torch.cuda.current_stream().wait_stream(s)
    for t in ids + mls:
        t.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    runs.append([t.cpu().numpy().copy() for t in ids + mls])
    for i in range(3):
        x = case.hidden[i]
        o_ids, o_ml, o_sec = orc.draft_argmax_nvfp4(x, case.q, case.s, case.g, case.cand_ids)

        def score_of(r, gid, x=x):
            c = int(np.searchsorted(case.cand_ids, gid))
            return float(orc.scores_nvfp4(x[r], case.q[c:c + 1], case.s[c:c + 1], case.g, nthreads=1)[0])

        for run in runs:
            check_ids(run[i], run[3 + i], o_ids, o_ml, o_sec, score_of, TOL_4BIT)
    assert int(ws.count_nonzero()) == 0


def test_packed_rejects_bad_shapes(vh):
    import torch
    x = torch.zeros(1, 320, dtype=torch.bfloat16, device="cuda")
    P = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    c = torch.arange(10, dtype=torch.int32, device="cuda")
    with pytest.raises(vh.VHError) as e:  # H % 256 != 0
        vh.mtp_draft_head_argmax_nvfp4_packed(x, P, 1.0, c)
    assert e.value.status == vh.VH_ERR_SHAPE
    assert vh.vh_nvfp4_packed_bytes(10, 320) == 0
    x = torch.zeros(1, 8192, dtype=torch.bfloat16, device="cuda")  # 16 f16 rows of 8192 exceed shared memory
    P = torch.zeros(vh.vh_nvfp4_packed_bytes(10, 8192), dtype=torch.uint8, device="cuda")
    with pytest.raises(vh.VHError) as e:
        vh.mtp_draft_head_argmax_nvfp4_packed(x, P, 1.0, c)
    assert e.value.status == vh.VH_ERR_SHAPE
