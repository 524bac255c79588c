"""The bf16 head on warp-level MMAs fed from the weight stream (k_gemv_mma_bf16):
the draft head for 2-16 hidden rows (its default there; 9-16 rows need H <=
5120) and greedy verify (on VH_PATH_WARP_MMA, and under AUTO for up to 16
rows against heads under 384 MiB), against the CPU oracle through the C ABI."""
import os

import numpy as np
import pytest

from parity_util import TOL_BF16, check_accept, check_ids, to_torch, to_torch_bf16

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


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


def run_draft(vh, x, W, cand):
    import torch
    ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(x), to_torch_bf16(W), to_torch(cand))
    torch.cuda.synchronize()
    return ids.cpu().numpy(), ml.cpu().numpy()


def check_draft(vh, orc, x, W, cand):
    g_ids, g_ml = run_draft(vh, x, W, cand)
    o_ids, o_ml, o_sec = orc.draft_argmax(x, W, cand)

    def score_of(r, gid):
        c = int(np.searchsorted(cand, gid))
        assert cand[c] == gid, "GPU returned an id outside the candidate set"
        return orc.dot_bf16(x[r], W[c])

    check_ids(g_ids, g_ml, o_ids, o_ml, o_sec, score_of, TOL_BF16)
    return g_ids, g_ml


# 8-row groups: Vc = 1 / 7 / 8 / 9 cover one partial group, exactly one, one plus one row; the widest H
# the kernel takes is 10,240 for up to 8 hidden rows and 5,120 for 9-16 (the hidden rows fill 160 KiB of
# shared memory); past 5,120 a batch of 9-16 runs as groups of 8 (and past 10,240 on the CUDA-core GEMV)
@pytest.mark.parametrize("Vc,H,B", [(1, 256, 2), (7, 256, 3), (8, 512, 8), (9, 512, 5), (1001, 1024, 8),
                                    (20_011, 2048, 2), (3000, 4096, 8), (700, 8192, 4), (500, 10240, 3),
                                    (300, 10496, 2), (9, 256, 9), (1001, 1024, 12), (20_011, 2048, 16),
                                    (3000, 5120, 16), (600, 5376, 13), (4097, 512, 24)])
def test_draft_shapes(vh, orc, syn, Vc, H, B):
    cand = syn.sorted_subset(Vc + H + 3, 2, 300_000, Vc)
    W = syn.normal_bf16(Vc + 17, 1, (Vc, H), 0.02)
    x = syn.normal_bf16(B + 19, 3, (B, H), 1.0)
    check_draft(vh, orc, x, W, cand)


@pytest.mark.parametrize("B", [2, 8, 16])
def test_draft_full_size_65536x2048(vh, orc, syn, B):
    case = syn.draft_case(Vc=65_536, H=2048, B=B, steps=1, seed=2)
    check_draft(vh, orc, case.hidden[0], case.W, case.cand_ids)


def test_draft_long_steps_on_a_768_mib_table(vh, orc, syn):
    """2-16 rows against a table of 768 MiB or more take the 512-element steps
    (1 KiB of each head row per load step): 4 rows on 201,003 x 2048 (785 MiB,
    a ragged last 8-row group) against the oracle."""
    Vc, H, B = 201_003, 2048, 4
    cand = syn.sorted_subset(61, 2, 2_000_000, Vc)
    W = syn.normal_bf16(62, 1, (Vc, H), 0.02)
    x = syn.normal_bf16(63, 3, (B, H), 1.0)
    assert Vc * H * 2 >= 768 << 20
    check_draft(vh, orc, x, W, cand)


def test_draft_ties_across_group_warp_and_cta_boundaries(vh, syn):
    """One winning row planted at many places (both sides of 8-row group
    boundaries, scattered over the table so that warp ranges and CTA ranges
    cut between copies, and the last row): every hidden row must return the
    lowest candidate id among the copies, with the copies' exact score."""
    Vc, H, B = 65_536, 256, 16
    W = syn.normal_bf16(41, 1, (Vc, H), 0.02)
    # non-negative hidden rows (sign bits cleared) and an all-ones winner: every hidden row scores it
    # sum |x| ~ 200, far above the rest (~1); 16 rows use the upper half of the MMA's A operand as well
    x = syn.normal_bf16(42, 3, (B, H), 1.0) & np.uint16(0x7FFF)
    cand = syn.sorted_subset(43, 2, 248_320, Vc)
    sign = np.full(H, 0x3F80, np.uint16)  # +1
    planted = sorted({7, 8, 15, 16, 255, 256, 431, 432, 1023, 1024, 4095, 4096, 8191, 8192, 12_345, 20_000,
                      32_767, 32_768, 40_960, 50_001, 65_528, 65_535})
    for r in planted:
        W[r] = sign
    g_ids, g_ml = run_draft(vh, x, W, cand)
    assert list(g_ids) == [int(cand[planted[0]])] * B
    # every copy scores bit-identically (H = 256 is one 256-element step, so no group is cut between
    # warps): the max logit equals the planted row's score from a one-row table
    import torch
    _, ml2 = vh.mtp_draft_head_argmax(to_torch_bf16(x), to_torch_bf16(W[planted[-1]:planted[-1] + 1]),
                                      to_torch(cand[planted[-1]:planted[-1] + 1]))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g_ml, ml2.cpu().numpy())


def test_draft_zero_head_ties_to_first_candidate(vh, syn):
    Vc, H, B = 5000, 512, 6
    cand = syn.sorted_subset(51, 2, 248_320, Vc)
    W = np.zeros((Vc, H), np.uint16)
    x = syn.normal_bf16(52, 3, (B, H), 1.0)
    g_ids, g_ml = run_draft(vh, x, W, cand)
    assert list(g_ids) == [int(cand[0])] * B
    assert list(g_ml) == [0.0] * B


def run_verify(vh, X, W, draft, B, k, path):
    import torch
    acc, nid, ml = vh.spec_verify_greedy(to_torch_bf16(X), to_torch_bf16(W), to_torch(draft), B, k, path=path)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nid.cpu().numpy(), ml.cpu().numpy()


def check_verify(vh, orc, syn, X, W, B, k, path, seed):
    _, o_nid, o_ml, o_sec = orc.verify_greedy(X, W, None, B, k)
    draft = syn.corrupt_ids(seed, syn.STREAM_CORRUPT, o_nid.reshape(B, k + 1)[:, :k].copy(), W.shape[0], 0.45)
    o_acc = np.array([orc.accept_len(o_nid[b * (k + 1): b * (k + 1) + k], draft[b]) for b in range(B)], np.int32)
    g_acc, g_nid, g_ml = run_verify(vh, X, W, draft, B, k, path)
    check_ids(g_nid, g_ml, o_nid, o_ml, o_sec, lambda r, v: orc.dot_bf16(X[r], W[v]), TOL_BF16)
    check_accept(g_acc, g_nid, o_acc, o_ml, o_sec, draft, B, k)


# VH_PATH_WARP_MMA: 2-16 rows in one pass (8 per pass past H = 5120), 20 rows in two
@pytest.mark.parametrize("B,k,V,H", [(1, 3, 5000, 256), (2, 3, 3001, 512), (1, 7, 2049, 1024), (1, 1, 777, 2048),
                                     (1, 3, 40_000, 4096), (3, 3, 1500, 256), (1, 3, 9, 512), (4, 3, 20_000, 2048),
                                     (1, 15, 3001, 1024), (3, 2, 1000, 6144), (5, 3, 2500, 512)])
def test_verify_shapes(vh, orc, syn, B, k, V, H):
    path = vh.VH_PATH_WARP_MMA
    W = syn.normal_bf16(V + H + 5, 1, (V, H), 0.02)
    X = syn.normal_bf16(B + k + 7, 4, (B * (k + 1), H), 1.0)
    check_verify(vh, orc, syn, X, W, B, k, path, seed=B * 100 + k + 1)


# AUTO takes the warp MMAs for up to 16 rows against heads under 384 MiB (H % 256 == 0, H <= 5120 above 8 rows)
@pytest.mark.parametrize("B,k,V,H", [(1, 3, 4096, 256), (2, 3, 20_000, 512), (1, 7, 3001, 2048), (4, 3, 9000, 1024),
                                     (3, 3, 5000, 5120)])
def test_verify_auto_small_heads(vh, orc, syn, B, k, V, H):
    W = syn.normal_bf16(V + H + 9, 1, (V, H), 0.02)
    X = syn.normal_bf16(B + k + 13, 4, (B * (k + 1), H), 1.0)
    check_verify(vh, orc, syn, X, W, B, k, vh.VH_PATH_AUTO, seed=B * 100 + k + 7)


def test_warp_mma_path_refuses_other_widths(vh):
    import torch
    X = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(16, 128, dtype=torch.bfloat16, device="cuda")
    d = torch.zeros(1, 3, dtype=torch.int32, device="cuda")
    with pytest.raises(vh.VHError) as e:
        vh.spec_verify_greedy(X, W, d, 1, 3, path=vh.VH_PATH_WARP_MMA)
    assert e.value.status == vh.VH_ERR_SHAPE


def _load_verify_golden():
    rows, seqs, meta = {}, {}, {}
    with open(os.path.join(HERE, "golden", "verify_b64_k3_248320x2048.txt")) as f:
        for line in f:
            p = line.split()
            if not p or p[0].startswith("#"):
                continue
            if p[0] == "row":
                rows[int(p[1])] = (int(p[2]), float.fromhex(p[3]), float.fromhex(p[4]))
            elif p[0] == "seq":
                seqs[int(p[1])] = ([int(v) for v in p[2:5]], int(p[5]))
            else:
                meta[p[0]] = p[1:]
    return rows, seqs, meta


@pytest.mark.parametrize("n_seq", [1, 2, 3, 4])
def test_batch1_verify_full_head_against_stored_oracle(vh, orc, syn, n_seq):
    """The batch-1 to batch-4 MTP3 verify on the warp-MMA path against the
    full 248,320 x 2048 head: the first sequences of the stored full-size
    oracle results (4, 8, 12 or 16 rows)."""
    rows, seqs, meta = _load_verify_golden()
    case = syn.verify_case(B=64, k=3, H=2048, V=syn.V_FULL, seed_w=2, seed=4, with_head=True)
    assert syn.fingerprint(case.X) == int(meta["fingerprint_x"][0])
    R = 4 * n_seq
    X = np.ascontiguousarray(case.X[:R])
    draft = np.array([seqs[b][0] for b in range(n_seq)], np.int32)
    o_nid = np.array([rows[r][0] for r in range(R)], np.int32)
    o_ml = np.array([rows[r][1] for r in range(R)])
    o_sec = np.array([rows[r][2] for r in range(R)])
    o_acc = np.array([seqs[b][1] for b in range(n_seq)], np.int32)
    g_acc, g_nid, g_ml = run_verify(vh, X, case.W, draft, n_seq, 3, vh.VH_PATH_WARP_MMA)
    check_ids(g_nid, g_ml, o_nid, o_ml, o_sec, lambda r, v: orc.dot_bf16(X[r], case.W[v]), TOL_BF16)
    check_accept(g_acc, g_nid, o_acc, o_ml, o_sec, draft, n_seq, 3)
