"""Exact ties on every kernel family: the lowest global id must win.

The rule (lowest id among equal scores) matters wherever the head holds
duplicate rows.  Ties only stay ties if both copies score bit for bit the same,
so every input here is small integers (or half-integers for the 4-bit head):
every product and partial sum is exact in fp32 and the summation order of a
kernel cannot split a tie.  The expected ids are then unique and come from an
exact int64/float64 brute force, which the oracle must match too.

Planted copies of a hidden row's winning head row sit on the structural seams
of the kernels: inside one warp's 32 rows, across the epilogue warps of a
128-row tile, across 128-row tiles, across the two CTAs of a 256-row pair tile,
across pair tiles, on tiles owned by different persistent CTAs, and in the last
partial tile.  The greedy rule is "少读一张大表，草稿路径才真正快起来" (global id after
the per-rank argmax, full-vocabulary verify) with the lowest-id tie-break of
the method's statement.
"""
import numpy as np
import pytest

from parity_util import accept_scan, to_torch, to_torch_bf16

pytestmark = pytest.mark.gpu

BF16 = {-2: 0xC000, -1: 0xBF80, 0: 0x0000, 1: 0x3F80, 2: 0x4000}


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


def bf16_of_ints(a):
    out = np.zeros(a.shape, np.uint16)
    for v, bits in BF16.items():
        out[a == v] = bits
    return out


def seam_positions(V, n):
    """n disjoint tuples of head rows that straddle the kernels' seams; the
    expected winner of each tuple is its smallest row."""
    kinds = [
        lambda m: (32 * m + 20, 32 * m + 3),                # one warp: ballot picks the lower lane
        lambda m: (128 * m + 32, 128 * m + 31),             # epilogue warps of one 128-row tile
        lambda m: (128 * m + 128, 128 * m + 127),           # consecutive 128-row tiles
        lambda m: (256 * m + 128, 256 * m + 127),           # the two CTAs of a pair tile
        lambda m: (256 * m + 256, 256 * m + 255),           # consecutive pair tiles
        lambda m: (128 * (m + 152) + 5, 128 * m + 5),       # tiles i and i + 152 (another pass of the grid)
        lambda m: (256 * (m + 76) + 9, 256 * m + 9, 256 * (m + 40) + 200),  # pair tiles of different pairs
        lambda m: (16 * m + 15, 16 * m + 16, 16 * m + 47),  # 16-row blocks of the 4-bit kernels
        lambda m: (V - 1 - (m % 50), 64 * m + 1),           # the last partial tile against an early one
    ]
    rng = np.random.default_rng(V + n)
    used, out = set(), []
    turn = 0
    while len(out) < n:
        for attempt in range(50_000):  # a kind with no room left hands over to the next one
            kind = kinds[(turn + attempt // 2000) % len(kinds)]
            pos = tuple(int(p) for p in kind(int(rng.integers(0, max(1, V // 16)))))
            if all(0 <= p < V for p in pos) and not (set(pos) & used):
                break
        else:
            raise RuntimeError("no room for the planted rows")
        turn += 1
        used |= set(pos)
        out.append(pos)
    return out


def int_problem(seed, V, H, R, zero_rows=()):
    """Integer head (entries -1/0/1, winners 2 * sign(x)) and hidden rows
    (entries -1/0/1); returns (W ints, X ints, planted tuples)."""
    rng = np.random.default_rng(seed)
    W = rng.integers(-1, 2, size=(V, H)).astype(np.int64)
    X = rng.integers(-1, 2, size=(R, H)).astype(np.int64)
    for r in zero_rows:
        X[r] = 0
    planted = seam_positions(V, R)
    for r, pos in enumerate(planted):
        for p in pos:
            W[p] = 2 * np.sign(X[r])
    return W, X, planted


def expected_argmax(X, W, gid=None):
    S = X @ W.T  # exact integers
    best = S.max(axis=1)
    if gid is None:
        ids = np.argmax(S, axis=1)  # first maximum = lowest row = lowest id
    else:
        ids = np.array([gid[S[r] == best[r]].min() for r in range(S.shape[0])])
    return ids.astype(np.int32), best.astype(np.float64)


def draft_ids_for(exp_nid, B, k, V):
    """Draft ids that accept b % (k+1) tokens of sequence b."""
    nid = exp_nid.reshape(B, k + 1)
    d = np.zeros((B, k), np.int32)
    for b in range(B):
        a = b % (k + 1)
        for j in range(k):
            d[b, j] = nid[b, j] if j < a else (nid[b, j] + 1 + b) % V
    return d


@pytest.mark.parametrize("B,k,path", [(4, 3, 2), (32, 3, 2), (33, 3, 2), (64, 3, 2), (5, 3, 1), (3, 15, 2)])
def test_verify_ties_bf16(vh, orc, B, k, path):
    """bf16 verify: R <= 128 rows run the one-CTA tcgen05 kernel, 129..256 the
    CTA pair; path 1 is the CUDA-core GEMV.  V = 40,000 gives every CTA (and
    pair) more than one tile and a 64-row last tile."""
    import torch
    V, H = 40_000, 256
    R = B * (k + 1)
    W, X, planted = int_problem(1000 + R, V, H, R, zero_rows=(1,))
    exp_nid, exp_ml = expected_argmax(X, W)
    for r, pos in enumerate(planted):
        if r != 1:
            assert exp_nid[r] == min(pos), "construction: the planted copies are the unique maximum"
    assert exp_nid[1] == 0 and exp_ml[1] == 0  # a zero hidden row ties every row: id 0
    draft = draft_ids_for(exp_nid, B, k, V)
    Wb, Xb = bf16_of_ints(W), bf16_of_ints(X)
    o_acc, o_nid, o_ml, _ = orc.verify_greedy(Xb, Wb, draft, B, k)
    np.testing.assert_array_equal(o_nid, exp_nid)
    np.testing.assert_array_equal(o_ml.astype(np.float64), exp_ml)
    acc, nid, ml = vh.spec_verify_greedy(to_torch_bf16(Xb), to_torch_bf16(Wb), to_torch(draft), B, k, path=path)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(nid.cpu().numpy(), exp_nid)
    np.testing.assert_array_equal(ml.cpu().numpy().astype(np.float64), exp_ml)
    np.testing.assert_array_equal(acc.cpu().numpy(), accept_scan(exp_nid, draft, B, k))
    np.testing.assert_array_equal(acc.cpu().numpy(), o_acc)


def test_verify_ties_all_zero_head(vh):
    """Every score is 0: every next id is 0 and a sequence accepts exactly its
    leading zero draft ids (one-CTA kernel, CTA pair and CUDA cores)."""
    import torch
    V, H = 3000, 128
    for B in (8, 64):
        k = 3
        W = torch.zeros(V, H, dtype=torch.bfloat16, device="cuda")
        X = torch.randn(B * (k + 1), H, device="cuda").to(torch.bfloat16)
        d = np.full((B, k), 5, np.int32)
        for b in range(B):
            d[b, : b % (k + 1)] = 0
        for path in (1, 2):
            acc, nid, ml = vh.spec_verify_greedy(X, W, to_torch(d), B, k, path=path)
            torch.cuda.synchronize()
            assert int(nid.abs().sum()) == 0 and float(ml.abs().sum()) == 0.0
            assert list(acc.cpu().numpy()) == [b % (k + 1) for b in range(B)]


def test_verify_ties_more_than_256_rows(vh, orc):
    """300 rows: a 256-row pair launch, then a 44-row one-CTA launch that also
    runs the acceptance scan over all sequences."""
    import torch
    B, k, V, H = 75, 3, 20_000, 256
    R = B * (k + 1)
    W, X, _ = int_problem(77, V, H, R)
    exp_nid, exp_ml = expected_argmax(X, W)
    draft = draft_ids_for(exp_nid, B, k, V)
    Wb, Xb = bf16_of_ints(W), bf16_of_ints(X)
    acc, nid, ml = vh.spec_verify_greedy(to_torch_bf16(Xb), to_torch_bf16(Wb), to_torch(draft), B, k, path=2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(nid.cpu().numpy(), exp_nid)
    np.testing.assert_array_equal(ml.cpu().numpy().astype(np.float64), exp_ml)
    np.testing.assert_array_equal(acc.cpu().numpy(), accept_scan(exp_nid, draft, B, k))


# ----------------------------------------------------------------------------
# 4-bit head: codes of -1/-0.5/0/0.5/1 (planted winners 6 * sign(x)), block
# scales 0.5 / 1 / 2 (winners 1), tensor scale 1 -- every score a multiple of
# 1/4, exact in fp32 in every kernel.

E2M1_OF = {0.0: 0x0, 0.5: 0x1, 1.0: 0x2, 6.0: 0x7, -0.5: 0x9, -1.0: 0xA, -6.0: 0xF}
SCALES = np.array([0x30, 0x38, 0x40], np.uint8)  # E4M3 0.5, 1, 2


def nvfp4_int_problem(seed, V, H, R):
    rng = np.random.default_rng(seed)
    w = rng.choice(np.array([-1.0, -0.5, 0.0, 0.5, 1.0]), size=(V, H))
    sc = rng.choice(SCALES, size=(V, H // 16))
    X = rng.integers(-1, 2, size=(R, H)).astype(np.int64)
    planted = seam_positions(V, R)
    for r, pos in enumerate(planted):
        for p in pos:
            w[p] = 6.0 * np.sign(X[r])
            sc[p] = 0x38
    codes = np.zeros((V, H), np.uint8)
    for v, c in E2M1_OF.items():
        codes[w == v] = c
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)  # element 2i in the low nibble
    scale_val = {0x30: 0.5, 0x38: 1.0, 0x40: 2.0}
    wv = w * np.repeat(np.vectorize(scale_val.get)(sc), 16, axis=1)  # exact decoded weights
    return q, sc.astype(np.uint8), wv, X, planted


def expected_argmax_f(X, Wv, gid=None):
    S = X.astype(np.float64) @ Wv.T  # multiples of 1/4 far below 2^53: exact
    best = S.max(axis=1)
    if gid is None:
        ids = np.argmax(S, axis=1)
    else:
        ids = np.array([gid[S[r] == best[r]].min() for r in range(S.shape[0])])
    return ids.astype(np.int32), best


# 1 / 2 sequences: <= 8 rows (warp-level MMA kernel); 3 / 4 sequences: 9..16
# rows (one tcgen05 pass); 5 / 64 sequences: the CTA-pair kernel
@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 64])
def test_verify_ties_nvfp4(vh, orc, B):
    import torch
    k, V, H = 3, 30_000, 512
    R = B * (k + 1)
    q, s, wv, X, planted = nvfp4_int_problem(500 + B, V, H, R)
    exp_nid, exp_ml = expected_argmax_f(X, wv)
    for r, pos in enumerate(planted):
        assert exp_nid[r] == min(pos)
    draft = draft_ids_for(exp_nid, B, k, V)
    Xb = bf16_of_ints(X)
    o_acc, o_nid, o_ml, _ = orc.verify_greedy_nvfp4(Xb, q, s, 1.0, draft, B, k)
    np.testing.assert_array_equal(o_nid, exp_nid)
    np.testing.assert_array_equal(o_ml.astype(np.float64), exp_ml)
    acc, nid, ml = vh.spec_verify_greedy_nvfp4(to_torch_bf16(Xb), to_torch(q), to_torch(s), 1.0, to_torch(draft),
                                               B, k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(nid.cpu().numpy(), exp_nid)
    np.testing.assert_array_equal(ml.cpu().numpy().astype(np.float64), exp_ml)
    np.testing.assert_array_equal(acc.cpu().numpy(), o_acc)


# B = 1: CUDA-core streaming kernel; 8: warp-level MMA; 12 / 16: tcgen05;
# 20: a 16-row pass and a 4-row pass
@pytest.mark.parametrize("B", [1, 8, 12, 16, 20])
def test_draft_ties_nvfp4(vh, orc, B):
    import torch
    Vc, H = 30_000, 512
    q, s, wv, X, planted = nvfp4_int_problem(900 + B, Vc, H, B)
    cand = (np.arange(Vc, dtype=np.int32) * 7 + 3)  # sorted: the lowest row is the lowest id
    exp_row, exp_ml = expected_argmax_f(X, wv)
    Xb = bf16_of_ints(X)
    o_ids, o_ml, _ = orc.draft_argmax_nvfp4(Xb, q, s, 1.0, cand)
    np.testing.assert_array_equal(o_ids, cand[exp_row])
    ids, ml = vh.mtp_draft_head_argmax_nvfp4(to_torch_bf16(Xb), to_torch(q), to_torch(s), 1.0, to_torch(cand))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), cand[exp_row])
    np.testing.assert_array_equal(ml.cpu().numpy().astype(np.float64), exp_ml)


@pytest.mark.parametrize("B", [1, 3, 9])
def test_draft_ties_bf16_seams(vh, orc, B):
    """bf16 candidate table: planted copies on the GEMV's warp and CTA seams."""
    import torch
    Vc, H = 50_000, 256
    W, X, planted = int_problem(40 + B, Vc, H, B)
    cand = (np.arange(Vc, dtype=np.int32) * 4 + 1)
    exp_row, exp_ml = expected_argmax(X, W)
    Wb, Xb = bf16_of_ints(W), bf16_of_ints(X)
    ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(Xb), to_torch_bf16(Wb), to_torch(cand))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), cand[exp_row])
    np.testing.assert_array_equal(ml.cpu().numpy().astype(np.float64), exp_ml)


# ----------------------------------------------------------------------------
# gather: the lowest ROW ID wins, whatever the order of the list


def test_gather_ties_lowest_row_id_in_any_list_order(vh, orc):
    import torch
    V, H, B = 60_000, 256, 4
    rng = np.random.default_rng(5)
    W = rng.integers(-1, 2, size=(V, H)).astype(np.int64)
    X = rng.integers(-1, 2, size=(B, H)).astype(np.int64)
    # hidden row b: equal winners at two distinct ids, the higher id listed first
    placements = [(10, 11), (100, 29_000), (0, 29_999), (5000, 5031)]  # list positions: adjacent / far apart
    winners = [(59_000 - 1000 * b, 300 + 77 * b) for b in range(B)]
    others = np.setdiff1d(np.arange(V), np.array(winners).ravel())
    rows = rng.permutation(others)[:30_000].astype(np.int32)
    want = []
    for b, (pa, pb) in enumerate(placements):
        hi_id, lo_id = winners[b]
        rows[pa], rows[pb] = hi_id, lo_id
        W[hi_id] = W[lo_id] = 2 * np.sign(X[b])
        want.append(lo_id)
    assert len(set(rows.tolist())) == rows.size
    Wb, Xb = bf16_of_ints(W), bf16_of_ints(X)
    exp_ids, exp_ml = expected_argmax(X, W[rows], gid=rows)
    assert list(exp_ids) == want
    o_ids, o_ml, _ = orc.draft_argmax_gather(Xb, Wb, rows)
    np.testing.assert_array_equal(o_ids, exp_ids)
    ids, ml = vh.mtp_draft_head_argmax_gather(to_torch_bf16(Xb), to_torch_bf16(Wb), to_torch(rows))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), exp_ids)
    np.testing.assert_array_equal(ml.cpu().numpy().astype(np.float64), exp_ml)
    # the same row listed twice ties with itself
    rows2 = np.array([rows[5], 12, 12, 7, 12], np.int32)
    W[12] = 3 * np.sign(X[0])
    Wb = bf16_of_ints(np.clip(W, -2, 2))
    ids, _ = vh.mtp_draft_head_argmax_gather(to_torch_bf16(Xb[:1]), to_torch_bf16(Wb), to_torch(rows2))
    torch.cuda.synchronize()
    assert int(ids[0]) == 12
