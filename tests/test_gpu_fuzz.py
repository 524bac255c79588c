"""Seeded random shapes through every entry point against the oracle: batch
sizes, widths (every allowed multiple), table sizes, k and gathered id lists
drawn at random, so that kernel selection boundaries, ragged tails and group
splits are hit in combinations no hand-picked list covers (62 cases by
default; VH_FUZZ_SCALE multiplies every family)."""
import os

import numpy as np
import pytest

from parity_util import TOL_4BIT, TOL_BF16, accept_scan, check_ids, to_torch, to_torch_bf16

pytestmark = pytest.mark.gpu

MAC_BUDGET = 120_000_000  # oracle multiply-adds per case
SCALE = int(os.environ.get("VH_FUZZ_SCALE", "1"))  # more cases per family for a longer run


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


def _rows_for(rng, budget, per_row, lo=1, hi=40_000):
    return int(max(lo, min(hi, rng.integers(lo, hi + 1), budget // max(per_row, 1))))


@pytest.mark.parametrize("case", range(10 * SCALE))
def test_fuzz_draft_bf16(vh, orc, syn, case):
    import torch
    rng = np.random.default_rng(900 + case)
    B = int(rng.choice([1, 1, 1, 2, 3, 5, 8, 9, 17]))
    H = 16 * int(rng.integers(1, 257))  # 16 .. 4096
    Vc = _rows_for(rng, MAC_BUDGET, B * H)
    W = syn.normal_bf16(1000 + case, 1, (Vc, H), 0.02)
    cand = syn.sorted_subset(1000 + case, 2, 248_320, Vc)
    x = syn.normal_bf16(2000 + case, 3, (B, H), 1.0)
    ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(x), to_torch_bf16(W), to_torch(cand))
    torch.cuda.synchronize()
    o_ids, o_ml, o_sec = orc.draft_argmax(x, W, cand)
    check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec,
              lambda r, g: orc.dot_bf16(x[r], W[int(np.searchsorted(cand, g))]), TOL_BF16)


@pytest.mark.parametrize("case", range(6 * SCALE))
def test_fuzz_gather(vh, orc, syn, case):
    import torch
    rng = np.random.default_rng(950 + case)
    B = int(rng.choice([1, 1, 2, 4]))
    H = 16 * int(rng.integers(1, 129))
    V = int(rng.integers(1, 30_000))
    n = _rows_for(rng, MAC_BUDGET, B * H, hi=20_000)
    rows = rng.integers(-50, V + 50, size=n).astype(np.int32)  # unsorted, repeats, out-of-range ids
    rows[int(rng.integers(0, n))] = int(rng.integers(0, V))     # at least one valid id
    W = syn.normal_bf16(3000 + case, 1, (V, H), 0.02)
    x = syn.normal_bf16(4000 + case, 3, (B, H), 1.0)
    ids, ml = vh.mtp_draft_head_argmax_gather(to_torch_bf16(x), to_torch_bf16(W), to_torch(rows))
    torch.cuda.synchronize()
    o_ids, o_ml, o_sec = orc.draft_argmax_gather(x, W, rows)
    check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec, lambda r, v: orc.dot_bf16(x[r], W[v]),
              TOL_BF16)


@pytest.mark.parametrize("case", range(8 * SCALE))
def test_fuzz_draft_nvfp4(vh, orc, syn, case):
    import torch
    rng = np.random.default_rng(1100 + case)
    B = int(rng.choice([1, 1, 2, 3, 8, 16, 17]))
    H = int(rng.choice([64 * int(rng.integers(1, 65)), 512 * int(rng.integers(1, 9))]))
    Vc = _rows_for(rng, MAC_BUDGET // 2, B * H, hi=20_000)
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(5000 + case, 6, (Vc, H), 0.02))
    cand = syn.sorted_subset(5000 + case, 2, 248_320, Vc)
    x = syn.normal_bf16(6000 + case, 3, (B, H), 1.0)
    ids, ml = vh.mtp_draft_head_argmax_nvfp4(to_torch_bf16(x), to_torch(q), to_torch(s), g, to_torch(cand))
    torch.cuda.synchronize()
    o_ids, o_ml, o_sec = orc.draft_argmax_nvfp4(x, q, s, g, cand)

    def score_of(r, gid):
        c = int(np.searchsorted(cand, gid))
        return float(orc.scores_nvfp4(x[r], q[c:c + 1], s[c:c + 1], g, nthreads=1)[0])

    check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec, score_of, TOL_4BIT)


@pytest.mark.parametrize("case", range(10 * SCALE))
def test_fuzz_verify_bf16(vh, orc, syn, case):
    import torch
    rng = np.random.default_rng(1200 + case)
    k = int(rng.integers(1, 16))
    B = int(rng.integers(1, max(2, 300 // (k + 1))))
    R = B * (k + 1)
    H = 64 * int(rng.integers(1, 33))
    V = _rows_for(rng, MAC_BUDGET, R * H, hi=30_000)
    path = int(rng.choice([0, 1, 2]))
    W = syn.normal_bf16(7000 + case, 1, (V, H), 0.02)
    X = syn.normal_bf16(8000 + case, 4, (R, H), 1.0)
    draft = rng.integers(0, V, size=(B, k)).astype(np.int32)
    acc, nid, ml = vh.spec_verify_greedy(to_torch_bf16(X), to_torch_bf16(W), to_torch(draft), B, k, path=path)
    torch.cuda.synchronize()
    _, o_nid, o_ml, o_sec = orc.verify_greedy(X, W, None, B, k)
    nid = nid.cpu().numpy()
    check_ids(nid, ml.cpu().numpy(), o_nid, o_ml, o_sec, lambda r, v: orc.dot_bf16(X[r], W[v]), TOL_BF16)
    np.testing.assert_array_equal(acc.cpu().numpy(), accept_scan(nid, draft, B, k))


@pytest.mark.parametrize("case", range(8 * SCALE))
def test_fuzz_warp_mma_bf16(vh, orc, syn, case):
    """The bf16 head on warp-level MMAs: the draft at 2-16 rows (its default
    for widths that are multiples of 256; 9-16 rows in one pass up to H =
    5,120, in 8-row passes above) and the verify on VH_PATH_WARP_MMA (one or
    several passes of up to 16 rows), at every width it takes up to 10,240."""
    import torch
    rng = np.random.default_rng(1400 + case)
    H = 256 * int(rng.integers(1, 41))  # 256 .. 10,240
    if case % 2 == 0:
        B = int(rng.integers(2, 17))
        Vc = _rows_for(rng, MAC_BUDGET, B * H)
        W = syn.normal_bf16(10_000 + case, 1, (Vc, H), 0.02)
        cand = syn.sorted_subset(10_000 + case, 2, 248_320, Vc)
        x = syn.normal_bf16(11_000 + case, 3, (B, H), 1.0)
        ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(x), to_torch_bf16(W), to_torch(cand))
        torch.cuda.synchronize()
        o_ids, o_ml, o_sec = orc.draft_argmax(x, W, cand)
        check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec,
                  lambda r, g: orc.dot_bf16(x[r], W[int(np.searchsorted(cand, g))]), TOL_BF16)
    else:
        k = int(rng.integers(1, 8))
        B = int(rng.integers(1, max(2, 24 // (k + 1))))
        R = B * (k + 1)
        V = _rows_for(rng, MAC_BUDGET, R * H, hi=30_000)
        W = syn.normal_bf16(12_000 + case, 1, (V, H), 0.02)
        X = syn.normal_bf16(13_000 + case, 4, (R, H), 1.0)
        draft = rng.integers(0, V, size=(B, k)).astype(np.int32)
        acc, nid, ml = vh.spec_verify_greedy(to_torch_bf16(X), to_torch_bf16(W), to_torch(draft), B, k,
                                             path=vh.VH_PATH_WARP_MMA)
        torch.cuda.synchronize()
        _, o_nid, o_ml, o_sec = orc.verify_greedy(X, W, None, B, k)
        nid = nid.cpu().numpy()
        check_ids(nid, ml.cpu().numpy(), o_nid, o_ml, o_sec, lambda r, v: orc.dot_bf16(X[r], W[v]), TOL_BF16)
        np.testing.assert_array_equal(acc.cpu().numpy(), accept_scan(nid, draft, B, k))


@pytest.mark.parametrize("case", range(6 * SCALE))
def test_fuzz_verify_nvfp4(vh, orc, syn, case):
    import torch
    rng = np.random.default_rng(1300 + case)
    k = int(rng.integers(1, 8))
    B = int(rng.integers(1, max(2, 300 // (k + 1))))
    R = B * (k + 1)
    H = int(rng.choice([64 * int(rng.integers(1, 17)), 512 * int(rng.integers(1, 5))]))
    V = _rows_for(rng, MAC_BUDGET // 2, R * H, hi=20_000)
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(9000 + case, 6, (V, H), 0.02))
    X = syn.normal_bf16(9500 + case, 4, (R, H), 1.0)
    draft = rng.integers(0, V, size=(B, k)).astype(np.int32)
    acc, nid, ml = vh.spec_verify_greedy_nvfp4(to_torch_bf16(X), to_torch(q), to_torch(s), g, to_torch(draft), B, k)
    torch.cuda.synchronize()
    _, o_nid, o_ml, o_sec = orc.verify_greedy_nvfp4(X, q, s, g, None, B, k)
    nid = nid.cpu().numpy()

    def score_of(r, v):
        return float(orc.scores_nvfp4(X[r], q[v:v + 1], s[v:v + 1], g, nthreads=1)[0])

    check_ids(nid, ml.cpu().numpy(), o_nid, o_ml, o_sec, score_of, TOL_4BIT)
    np.testing.assert_array_equal(acc.cpu().numpy(), accept_scan(nid, draft, B, k))


@pytest.mark.parametrize("case", range(6 * SCALE))
def test_fuzz_nvfp4_mma(vh, orc, syn, case):
    """2..8 rows at every width of the warp-level-MMA kernel (H = 256 * 2^i <=
    4096), ragged heads: the draft entry point, and verify with at most 8 rows."""
    import torch
    rng = np.random.default_rng(1400 + case)
    H = 256 << int(rng.integers(0, 5))
    B = int(rng.integers(2, 9))
    Vc = _rows_for(rng, MAC_BUDGET // 2, B * H, lo=1, hi=30_000)
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(9700 + case, 6, (Vc, H), 0.02))
    cand = syn.sorted_subset(9700 + case, 2, 248_320, Vc)
    x = syn.normal_bf16(9800 + case, 3, (B, H), 1.0)
    ids, ml = vh.mtp_draft_head_argmax_nvfp4(to_torch_bf16(x), to_torch(q), to_torch(s), g, to_torch(cand))
    torch.cuda.synchronize()
    o_ids, o_ml, o_sec = orc.draft_argmax_nvfp4(x, q, s, g, cand)

    def score_of(r, gid):
        c = int(np.searchsorted(cand, gid))
        return float(orc.scores_nvfp4(x[r], q[c:c + 1], s[c:c + 1], g, nthreads=1)[0])

    check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec, score_of, TOL_4BIT)

    k = int(rng.integers(1, 8))
    Bv = max(1, 8 // (k + 1))
    X = syn.normal_bf16(9900 + case, 4, (Bv * (k + 1), H), 1.0)
    draft = rng.integers(0, Vc, size=(Bv, k)).astype(np.int32)
    acc, nid, vml = vh.spec_verify_greedy_nvfp4(to_torch_bf16(X), to_torch(q), to_torch(s), g, to_torch(draft), Bv, k)
    torch.cuda.synchronize()
    _, v_nid, v_ml, v_sec = orc.verify_greedy_nvfp4(X, q, s, g, None, Bv, k)
    nid = nid.cpu().numpy()
    check_ids(nid, vml.cpu().numpy(), v_nid, v_ml, v_sec,
              lambda r, v: float(orc.scores_nvfp4(X[r], q[v:v + 1], s[v:v + 1], g, nthreads=1)[0]), TOL_4BIT)
    np.testing.assert_array_equal(acc.cpu().numpy(), accept_scan(nid, draft, Bv, k))


@pytest.mark.parametrize("case", range(8 * SCALE))
def test_fuzz_nvfp4_tiled(vh, orc, syn, case):
    """The tiled 4-bit layout: random B (1..40, several 16-row passes), width
    (every multiple of 256 up to 6144), table size and, every other case, a
    verify with its acceptance scan instead of a draft."""
    import torch
    rng = np.random.default_rng(1700 + case)
    H = 256 * int(rng.integers(1, 25))
    q_rows = _rows_for(rng, MAC_BUDGET // 2, 16 * H, hi=20_000)
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(7000 + case, 6, (q_rows, H), 0.02))
    P = vh.nvfp4_pack(to_torch(q), to_torch(s))
    if case % 2 == 0:
        B = int(rng.choice([1, 2, 7, 8, 9, 16, 17, 33, 40]))
        cand = syn.sorted_subset(7000 + case, 2, 248_320, q_rows)
        x = syn.normal_bf16(8000 + case, 3, (B, H), 1.0)
        ids, ml = vh.mtp_draft_head_argmax_nvfp4_packed(to_torch_bf16(x), P, g, to_torch(cand))
        torch.cuda.synchronize()
        o_ids, o_ml, o_sec = orc.draft_argmax_nvfp4(x, q, s, g, cand)

        def score_of(r, gid):
            c = int(np.searchsorted(cand, gid))
            return float(orc.scores_nvfp4(x[r], q[c:c + 1], s[c:c + 1], g, nthreads=1)[0])

        check_ids(ids.cpu().numpy(), ml.cpu().numpy(), o_ids, o_ml, o_sec, score_of, TOL_4BIT)
    else:
        B, k = int(rng.choice([1, 2, 4, 5, 9])), int(rng.choice([1, 3, 7]))
        X = syn.normal_bf16(8000 + case, 4, (B * (k + 1), H), 1.0)
        d = rng.integers(0, q_rows, size=(B, k)).astype(np.int32)
        acc, nid, ml = vh.spec_verify_greedy_nvfp4_packed(to_torch_bf16(X), P, g, to_torch(d), B, k, q_rows)
        torch.cuda.synchronize()
        _, o_nid, o_ml, o_sec = orc.verify_greedy_nvfp4(X, q, s, g, None, B, k)
        check_ids(nid.cpu().numpy(), ml.cpu().numpy(), o_nid, o_ml, o_sec,
                  lambda r, v: float(orc.scores_nvfp4(X[r], q[v:v + 1], s[v:v + 1], g, nthreads=1)[0]), TOL_4BIT)
        np.testing.assert_array_equal(acc.cpu().numpy(), accept_scan(nid.cpu().numpy(), d, B, k))
