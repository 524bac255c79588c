"""The one-row bf16 draft head at H = 256 and 512, which runs on the warp
MMAs fed from the weight stream (k_gemv_mma_bf16 with one real hidden row),
against the CPU oracle through the C ABI: both widths, fewer rows than SMs
or than one 8-row group, ties across the 8-row groups and the CTA split,
unsorted candidate ids, and back-to-back calls with the head rewritten in
place between two of them."""
import numpy as np
import pytest

from parity_util import TOL_BF16, check_ids, to_torch, to_torch_bf16

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


def run_draft(vh, x, W, cand):
    import torch
    ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(x), to_torch_bf16(W), to_torch(cand))
    torch.cuda.synchronize()
    return ids.cpu().numpy(), ml.cpu().numpy()


def check_draft(vh, orc, x, W, cand):
    g_ids, g_ml = run_draft(vh, x, W, cand)
    o_ids, o_ml, o_sec = orc.draft_argmax(x, W, cand)
    pos = {int(c): i for i, c in enumerate(cand)}

    def score_of(r, gid):
        assert gid in pos, "GPU returned an id outside the candidate set"
        return orc.dot_bf16(x[r], W[pos[gid]])

    check_ids(g_ids, g_ml, o_ids, o_ml, o_sec, score_of, TOL_BF16)


# 1 row, part of one 8-row group, fewer groups than SMs, one row either side of a group seam, ragged last
# groups, and tables of 100 and 250 MiB
@pytest.mark.parametrize("Vc,H", [(1, 256), (1, 512), (7, 256), (151, 512), (152, 256), (153, 512), (1000, 256),
                                  (4865, 512), (20_011, 256), (200_000, 256), (250_000, 512)])
def test_one_row_shapes(vh, orc, syn, Vc, H):
    cand = syn.sorted_subset(Vc + H, 2, 300_000, Vc)
    W = syn.normal_bf16(Vc + 31, 1, (Vc, H), 0.02)
    x = syn.normal_bf16(H + 7, 3, (1, H), 1.0)
    check_draft(vh, orc, x, W, cand)


def _seams(Vc):
    """Rows either side of 8-row group seams spread over the table (so that
    CTAs and warps cut between copies), and the last row."""
    rows = set()
    for g in (1, 2, 7, 100, 1000, 2500, 4000, Vc // 8 - 1):
        rows |= {8 * g - 1, 8 * g}
    rows |= {12_345, Vc - 1}
    return sorted(x for x in rows if 0 <= x < Vc)


@pytest.mark.parametrize("H", [256, 512])
@pytest.mark.parametrize("shuffled", [False, True])
def test_one_row_ties_at_group_and_cta_seams(vh, syn, H, shuffled):
    """One winning row planted on both sides of group seams across the table:
    the lowest candidate id among the copies wins (with shuffled ids that is
    not the first copy), and every copy scores bit-identically."""
    Vc = 40_000
    W = syn.normal_bf16(71, 1, (Vc, H), 0.02)
    # small-integer hidden values: the planted rows score the integer sum |x| exactly in any summation order
    xi = np.random.default_rng(72 + H).integers(-8, 9, size=(1, H)).astype(np.float32)
    x = (xi.view(np.uint32) >> 16).astype(np.uint16)
    cand = syn.sorted_subset(73, 2, 248_320, Vc)
    if shuffled:
        cand = np.random.default_rng(H).permutation(cand).astype(np.int32)
    sign = np.where(xi[0] < 0, 0xBF80, 0x3F80).astype(np.uint16)  # -1 / +1: every copy scores sum |x|
    planted = _seams(Vc)
    for r in planted:
        W[r] = sign
    g_ids, g_ml = run_draft(vh, x, W, cand)
    assert int(g_ids[0]) == int(min(cand[planted]))
    assert float(g_ml[0]) == float(np.abs(xi).sum())
    # the same row alone in a one-row table scores the same bits
    _, ml1 = run_draft(vh, x, W[planted[-1]:planted[-1] + 1], cand[planted[-1]:planted[-1] + 1])
    assert g_ml[0] == ml1[0]


def test_one_row_zero_head_unsorted_ids(vh, syn):
    Vc, H = 9000, 512
    cand = np.random.default_rng(5).permutation(syn.sorted_subset(81, 2, 248_320, Vc)).astype(np.int32)
    W = np.zeros((Vc, H), np.uint16)
    x = syn.normal_bf16(82, 3, (1, H), 1.0)
    g_ids, g_ml = run_draft(vh, x, W, cand)
    assert int(g_ids[0]) == int(cand.min()) and float(g_ml[0]) == 0.0


def test_one_row_back_to_back_calls_and_rewritten_head(vh, orc, syn):
    """Three calls with no host sync between them (each prefetches its first
    rows before waiting on the previous one), then the head rewritten in place
    by a torch copy right before a fourth call: every result matches the
    oracle on the head it was given."""
    import torch
    Vc, H = 100_000, 512
    cand = syn.sorted_subset(91, 2, 248_320, Vc)
    W1 = syn.normal_bf16(92, 1, (Vc, H), 0.02)
    W2 = syn.normal_bf16(93, 1, (Vc, H), 0.02)
    xs = syn.normal_bf16(94, 3, (4, H), 1.0)
    Wd = to_torch_bf16(W1)
    cd = to_torch(cand)
    outs = []
    for i in range(3):
        outs.append(vh.mtp_draft_head_argmax(to_torch_bf16(xs[i:i + 1]), Wd, cd))
    Wd.copy_(to_torch_bf16(W2))
    outs.append(vh.mtp_draft_head_argmax(to_torch_bf16(xs[3:4]), Wd, cd))
    torch.cuda.synchronize()
    pos = {int(c): i for i, c in enumerate(cand)}
    for i, (ids, ml) in enumerate(outs):
        W = W1 if i < 3 else W2
        o_ids, o_ml, o_sec = orc.draft_argmax(xs[i:i + 1], W, cand)
        check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec,
                  lambda r, gid, W=W, i=i: orc.dot_bf16(xs[i], W[pos[gid]]), TOL_BF16)
