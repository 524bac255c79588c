"""The bf16 draft head for batches of 17-256 hidden rows, which run as one
pass of the tcgen05 contraction over the candidate table when H % 64 == 0
(the CTA pair above 128 rows), against the CPU oracle through the C ABI:
ragged batch sizes and table sizes, the full 65,536 x 2048 table at 64 rows,
ties across 128-row tile seams, an all-zero head, and widths that fall back
to launch groups of 8."""
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

    def score_of(r, gid):
        c = int(np.searchsorted(cand, gid))
        assert cand[c] == gid, "GPU returned an id outside the candidate set"
        return orc.dot_bf16(x[r], W[c])

    check_ids(g_ids, g_ml, o_ids, o_ml, o_sec, score_of, TOL_BF16)


# 17-128 rows: one CTA per SM; 129-256: the CTA pair; H = 704 is a multiple of 64 only; H = 1008 is not
# (groups of 8 on the CUDA-core GEMV)
@pytest.mark.parametrize("Vc,H,B", [(1, 256, 17), (7, 64, 24), (129, 128, 31), (1001, 1024, 33), (20_011, 2048, 64),
                                    (3000, 704, 100), (5000, 512, 129), (2000, 2048, 200), (1500, 4096, 256),
                                    (777, 1008, 20)])
def test_draft_batch_shapes(vh, orc, syn, Vc, H, B):
    cand = syn.sorted_subset(Vc + B, 2, 300_000, Vc)
    W = syn.normal_bf16(Vc + H + 3, 1, (Vc, H), 0.02)
    x = syn.normal_bf16(B + 11, 3, (B, H), 1.0)
    check_draft(vh, orc, x, W, cand)


def test_draft_batch_full_size_65536x2048_64_rows(vh, orc, syn):
    case = syn.draft_case(Vc=65_536, H=2048, B=64, steps=1, seed=2)
    check_draft(vh, orc, case.hidden[0], case.W, case.cand_ids)


def test_draft_batch_ties_across_tile_seams(vh, syn):
    """One winning row planted on both sides of 128-row tile seams (and the
    256-row seams of the CTA pair) and in the last partial tile: every hidden
    row returns the lowest candidate id among the copies, with the copies'
    score for that row bit-identical to a one-row table's."""
    Vc, H = 40_000, 512
    W = syn.normal_bf16(91, 1, (Vc, H), 0.02)
    cand = syn.sorted_subset(93, 2, 248_320, Vc)
    planted = sorted({127, 128, 255, 256, 383, 384, 1023, 1024, 20_095, 20_096, 39_935, 39_936, Vc - 1})
    for r in planted:
        W[r] = np.uint16(0x3F80)  # +1: with non-negative hidden rows every copy scores sum(x), far above the rest
    for B in (40, 160):
        x = syn.normal_bf16(92 + B, 3, (B, H), 1.0) & np.uint16(0x7FFF)
        g_ids, g_ml = run_draft(vh, x, W, cand)
        assert list(g_ids) == [int(cand[planted[0]])] * B
        _, ml1 = run_draft(vh, x, W[planted[-1]:planted[-1] + 1], cand[planted[-1]:planted[-1] + 1])
        np.testing.assert_array_equal(g_ml, ml1)


def test_draft_batch_zero_head_ties_to_first_candidate(vh, syn):
    Vc, H, B = 3000, 256, 50
    cand = syn.sorted_subset(95, 2, 248_320, Vc)
    W = np.zeros((Vc, H), np.uint16)
    x = syn.normal_bf16(96, 3, (B, H), 1.0)
    g_ids, g_ml = run_draft(vh, x, W, cand)
    assert list(g_ids) == [int(cand[0])] * B
    assert list(g_ml) == [0.0] * B
