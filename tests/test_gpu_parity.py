"""CUDA path vs the CPU oracle, element by element, through the C ABI."""
import os

import numpy as np
import pytest

from parity_util import (TOL_4BIT, TOL_BF16, accept_scan, check_accept, check_ids, to_torch, to_torch_bf16)

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


def run_draft(vh, x_bits, W_bits, cand, ws=None):
    import torch
    ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(x_bits), to_torch_bf16(W_bits), to_torch(cand), ws=ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), ml.cpu().numpy()


def draft_score_of(orc, x_bits, W_bits, cand):
    def f(r, gid):
        c = int(np.searchsorted(cand, gid))
        assert cand[c] == gid, "GPU returned an id outside the candidate set"
        return orc.dot_bf16(x_bits[r], W_bits[c])
    return f


def check_draft(vh, orc, x, W, cand):
    g_ids, g_ml = run_draft(vh, x, W, cand)
    o_ids, o_ml, o_sec = orc.draft_argmax(x, W, cand)
    check_ids(g_ids, g_ml, o_ids, o_ml, o_sec, draft_score_of(orc, x, W, cand), TOL_BF16)
    return g_ids, g_ml


# ----------------------------------------------------------------------------
# bf16 draft head


def test_tiny_workload(vh, orc, syn):
    draft, verify, W_full = syn.tiny_case()
    for x in draft.hidden:  # 3 sequential draft steps
        check_draft(vh, orc, x, draft.W, draft.cand_ids)


@pytest.mark.parametrize("Vc,H,B", [(1, 16, 1), (7, 64, 1), (1023, 256, 1), (1024, 256, 2), (1025, 272, 3),
                                    (5000, 2048, 1), (3001, 2080, 5), (2500, 4096, 8), (700, 6144, 9),
                                    (4099, 128, 17), (33, 4096, 1), (100_003, 2048, 1), (9000, 1040, 1),
                                    (500, 8192, 1)])
def test_draft_shapes(vh, orc, syn, Vc, H, B):
    cand = syn.sorted_subset(Vc + H, 2, 300_000, Vc)
    W = syn.normal_bf16(Vc + 7, 1, (Vc, H), 0.02)
    x = syn.normal_bf16(B + 11, 3, (B, H), 1.0)
    check_draft(vh, orc, x, W, cand)


def test_draft_full_size_65536x2048(vh, orc, syn):
    """The single-stream decode workload: 65,536 candidates x 2048, B=1, 3 steps."""
    case = syn.draft_case(Vc=65_536, H=2048, B=1, steps=3, seed=2)
    for x in case.hidden:
        check_draft(vh, orc, x, case.W, case.cand_ids)


@pytest.mark.parametrize("Vc", [248_320, 65_536, 32_768])
def test_head_size_sweep(vh, orc, syn, Vc):
    case = syn.draft_case(Vc=Vc, H=2048, B=1, steps=1, seed=2, cand_seed=3)
    check_draft(vh, orc, case.hidden[0], case.W, case.cand_ids)


def test_zero_head_ties_to_lowest_id(vh, orc):
    W = np.zeros((3000, 64), np.uint16)
    cand = (np.arange(3000, dtype=np.int32) * 3 + 5)
    x = np.full((2, 64), 0x3F80, np.uint16)
    g_ids, g_ml = run_draft(vh, x, W, cand)
    assert list(g_ids) == [5, 5] and list(g_ml) == [0.0, 0.0]


def test_duplicate_rows_tie_to_lowest_id(vh, syn):
    W = syn.normal_bf16(3, 1, (4096, 128), 0.02)
    x = syn.normal_bf16(3, 3, (1, 128), 1.0)
    xf = (x[0].astype(np.uint32) << 16).view(np.float32)
    best = np.where(xf > 0, 0x3F00, 0xBF00).astype(np.uint16)  # +-0.5: the clear winner
    for r in (100, 2000, 4000):  # same row three times, in different CTAs
        W[r] = best
    cand = np.arange(4096, dtype=np.int32)
    g_ids, _ = run_draft(vh, x, W, cand)
    assert g_ids[0] == 100


def test_single_candidate(vh, syn):
    W = syn.normal_bf16(4, 1, (1, 256), 0.02)
    x = syn.normal_bf16(4, 3, (4, 256), 1.0)
    g_ids, _ = run_draft(vh, x, W, np.array([123456], np.int32))
    assert list(g_ids) == [123456] * 4


def test_workspace_reused_and_left_zero(vh, syn):
    import torch
    case = syn.draft_case(Vc=20_000, H=512, B=3, steps=2, seed=9)
    ws = vh.workspace(3)
    Wd, cd = to_torch_bf16(case.W), to_torch(case.cand_ids)
    outs = []
    for x in case.hidden + case.hidden:
        ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(x), Wd, cd, ws=ws)
        outs.append((ids.cpu().numpy(), ml.cpu().numpy()))
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    for a, b in zip(outs[:2], outs[2:]):  # deterministic: same inputs, same bits
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_restricted_equals_full_when_top1_is_candidate(vh, syn):
    """Invariant on the GPU: with W_cand = W_full[cand], the restricted argmax
    equals the full argmax whenever the full top-1 is a candidate."""
    V, H = 50_000, 512
    W_full = syn.normal_bf16(21, 1, (V, H), 0.02)
    all_ids = np.arange(V, dtype=np.int32)
    cand = syn.sorted_subset(21, 2, V, 10_000)
    for t in range(6):
        x = syn.normal_bf16(40 + t, 3, (1, H), 1.0)
        f_ids, f_ml = run_draft(vh, x, W_full, all_ids)
        c = np.union1d(cand, f_ids).astype(np.int32) if t % 2 == 0 else cand
        r_ids, r_ml = run_draft(vh, x, np.ascontiguousarray(W_full[c]), c)
        if f_ids[0] in c:
            assert r_ids[0] == f_ids[0] and r_ml[0] == f_ml[0]
        else:
            assert r_ml[0] <= f_ml[0]


# ----------------------------------------------------------------------------
# gathered (dynamic) candidate rows, read in place from the full head


def run_gather(vh, x, W_full, rows):
    import torch
    ids, ml = vh.mtp_draft_head_argmax_gather(to_torch_bf16(x), to_torch_bf16(W_full), to_torch(rows))
    torch.cuda.synchronize()
    return ids.cpu().numpy(), ml.cpu().numpy()


def check_gather(vh, orc, x, W_full, rows):
    g_ids, g_ml = run_gather(vh, x, W_full, rows)
    o_ids, o_ml, o_sec = orc.draft_argmax_gather(x, W_full, rows)
    valid = set(int(r) for r in rows if 0 <= r < W_full.shape[0])

    def score_of(r, gid):
        assert int(gid) in valid, "GPU returned an id outside the gathered set"
        return orc.dot_bf16(x[r], W_full[gid])

    check_ids(g_ids, g_ml, o_ids, o_ml, o_sec, score_of, TOL_BF16)


@pytest.mark.parametrize("V,H,B,n", [(5000, 256, 1, 1), (5000, 256, 2, 777), (20_000, 2048, 1, 9000),
                                     (3000, 4096, 3, 2999), (7000, 6144, 1, 500)])
def test_gather_shapes(vh, orc, syn, V, H, B, n):
    W = syn.normal_bf16(V + 1, 1, (V, H), 0.02)
    x = syn.normal_bf16(B + 2, 3, (B, H), 1.0)
    rng = np.random.default_rng(V + n)
    rows = rng.integers(-5, V + 5, size=n).astype(np.int32)  # unsorted, repeats, a few out of range
    rows[0] = 17
    check_gather(vh, orc, x, W, rows)


def test_gather_fixed_plus_dynamic_full_head(vh, orc, syn):
    """32,768 fixed + 16,384 per-step dynamic candidate rows read in place
    from the 248,320 x 2048 head, B = 1, three steps."""
    W_full = syn.full_head(2, syn.V_FULL, 2048)
    for step in range(3):
        rows = syn.gather_row_ids(6, syn.V_FULL, step=step)
        x = syn.normal_bf16(2, syn.STREAM_HIDDEN, (1, 2048), 1.0, offset=step * 2048)
        check_gather(vh, orc, x, W_full, rows)


def test_gather_matches_candidate_table_kernel(vh, syn):
    """Same candidate set as a sorted copied table: same ids and maxima.  One
    hidden row runs the same streaming GEMV on both sides (bit-identical
    maxima); four rows run the table on warp-level MMAs, which sum in another
    fp32 order (ids identical, maxima within 1e-4)."""
    V, H = 30_000, 1024
    W = syn.normal_bf16(5, 1, (V, H), 0.02)
    cand = syn.sorted_subset(5, 2, V, 6000)
    x = syn.normal_bf16(6, 3, (4, H), 1.0)
    perm = np.random.default_rng(0).permutation(cand).astype(np.int32)
    table = np.ascontiguousarray(W[cand])
    g_ids, g_ml = run_gather(vh, x[:1], W, perm)
    t_ids, t_ml = run_draft(vh, x[:1], table, cand)
    np.testing.assert_array_equal(g_ids, t_ids)
    np.testing.assert_array_equal(g_ml, t_ml)
    g_ids, g_ml = run_gather(vh, x, W, perm)
    t_ids, t_ml = run_draft(vh, x, table, cand)
    np.testing.assert_array_equal(g_ids, t_ids)
    np.testing.assert_allclose(g_ml, t_ml, rtol=0, atol=1e-4)


# ----------------------------------------------------------------------------
# 4-bit draft head


def run_nvfp4(vh, x, q, s, g, cand):
    import torch
    ids, ml = vh.mtp_draft_head_argmax_nvfp4(to_torch_bf16(x), to_torch(q), to_torch(s), g, to_torch(cand))
    torch.cuda.synchronize()
    return ids.cpu().numpy(), ml.cpu().numpy()


def check_nvfp4(vh, orc, x, q, s, g, cand):
    g_ids, g_ml = run_nvfp4(vh, x, q, s, g, cand)
    o_ids, o_ml, o_sec = orc.draft_argmax_nvfp4(x, q, s, g, cand)

    def score_of(r, gid):
        c = int(np.searchsorted(cand, gid))
        assert cand[c] == gid
        return float(orc.scores_nvfp4(x[r], q[c:c + 1], s[c:c + 1], g, nthreads=1)[0])

    check_ids(g_ids, g_ml, o_ids, o_ml, o_sec, score_of, TOL_4BIT)
    return g_ids, g_ml


def test_nvfp4_hand_worked_rows(vh):
    """The hand-worked 4-bit rows of tests/golden/nvfp4_cases.txt, padded to
    H = 64: checks nibble order, scale order and the tensor scale on the GPU."""
    rows = {}
    argmaxes = []
    with open(os.path.join(HERE, "golden", "nvfp4_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [p.strip() for p in line.split("|")]
            if parts[0].startswith("row"):
                rows[int(parts[0].split()[1])] = (bytes.fromhex(parts[1]), bytes.fromhex(parts[2]))
            elif parts[0] == "argmax":
                hid = {int(t.split(":")[0]): float(t.split(":")[1]) for t in parts[1].split()}
                argmaxes.append((hid, int(parts[2])))
    H = 64
    q = np.zeros((3, H // 2), np.uint8)
    s = np.zeros((3, H // 16), np.uint8)
    for r, (qb, sb) in rows.items():
        q[r, :16] = list(qb)
        s[r, :2] = list(sb)
    cand = np.array([10, 20, 30], np.int32)
    for hid, want in argmaxes:
        x = np.zeros((1, H), np.float32)
        for h, v in hid.items():
            x[0, h] = v
        xb = (x.view(np.uint32) >> 16).astype(np.uint16)
        g_ids, _ = run_nvfp4(vh, xb, q, s, 0.5, cand)
        assert g_ids[0] == want


@pytest.mark.parametrize("Vc,H,B", [(1, 64, 1), (777, 128, 1), (4097, 256, 2), (3000, 4096, 8), (1500, 1024, 11),
                                    (1, 256, 1), (5003, 256, 1), (3001, 1024, 1), (999, 8192, 1), (40_000, 4096, 1),
                                    (2000, 512, 16), (1000, 512, 17), (300, 1536, 2)])
def test_nvfp4_shapes(vh, orc, syn, Vc, H, B):
    cand = syn.sorted_subset(Vc, 2, 248_320, Vc)
    w = syn.normal_f32(Vc, 6, (Vc, H), 0.02)
    q, s, g = syn.nvfp4_quantize(w)
    x = syn.normal_bf16(B, 3, (B, H), 1.0)
    check_nvfp4(vh, orc, x, q, s, g, cand)


# the warp-level-MMA kernel (2..8 hidden rows per launch, H = 256 * 2^i <= 4096):
# one partial block, a last block with a single valid row, fewer blocks than
# SMs, every slice count from 1 to 16, groups of 8 rows with a ragged last group
@pytest.mark.parametrize("Vc,H,B", [(5, 4096, 3), (17, 2048, 2), (100, 1024, 8), (2049, 512, 9), (33, 256, 24),
                                    (70_001, 4096, 2)])
def test_nvfp4_mma_shapes(vh, orc, syn, Vc, H, B):
    cand = syn.sorted_subset(Vc + 1, 2, 248_320, Vc)
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(Vc + 2, 6, (Vc, H), 0.02))
    x = syn.normal_bf16(B + 3, 3, (B, H), 1.0)
    check_nvfp4(vh, orc, x, q, s, g, cand)


def test_nvfp4_mma_ties_lowest_id(vh, orc, syn):
    """Identical top rows in different blocks, row halves and CTAs score
    exactly alike: every hidden row gets the lowest candidate id among them."""
    Vc, H, B = 20_000, 1024, 4
    q, s, g = syn.nvfp4_quantize(syn.normal_f32(11, 6, (Vc, H), 0.02))
    top = [7000, 39, 19_999, 2048, 47]
    q[top] = 0x77  # +6 in every element
    s[top] = 0x7E  # scale 448
    cand = syn.sorted_subset(12, 2, 248_320, Vc)
    x = np.full((B, H), 0x3F80, np.uint16)  # +1.0
    ids, ml = run_nvfp4(vh, x, q, s, g, cand)
    assert list(ids) == [int(cand[min(top)])] * B
    o_ids, o_ml, _ = orc.draft_argmax_nvfp4(x, q, s, g, cand)
    assert list(o_ids) == list(ids)
    np.testing.assert_allclose(ml, o_ml, rtol=0, atol=TOL_4BIT)


@pytest.mark.parametrize("B", [1, 8])
def test_nvfp4_full_size_65536x4096(vh, orc, syn, B):
    case = syn.nvfp4_case(Vc=65_536, H=4096, B=B, steps=3 if B == 1 else 1, seed=5)
    for x in case.hidden:
        check_nvfp4(vh, orc, x, case.q, case.s, case.g, case.cand_ids)


def test_nvfp4_equals_bf16_kernel_on_representable_head(vh, orc, syn):
    """g = 1: decoded 4-bit weights are exact bf16 values, so both kernels see
    the same head; their ids agree outside the near-tie band."""
    Vc, H = 6000, 512
    rng = np.random.default_rng(3)
    q = rng.integers(0, 256, size=(Vc, H // 2), dtype=np.uint8)
    s = rng.integers(0x20, 0x40, size=(Vc, H // 16), dtype=np.uint8)
    Wb = (orc.decode_nvfp4(q, s, 1.0).view(np.uint32) >> 16).astype(np.uint16)
    cand = np.arange(Vc, dtype=np.int32) * 2
    x = syn.normal_bf16(5, 3, (4, H), 1.0)
    a_ids, a_ml = run_nvfp4(vh, x, q, s, 1.0, cand)
    b_ids, b_ml = run_draft(vh, x, Wb, cand)
    o_ids, o_ml, o_sec = orc.draft_argmax(x, Wb, cand)
    for r in range(4):
        if o_ml[r] - o_sec[r] > 1e-2:
            assert a_ids[r] == b_ids[r] == o_ids[r]
    assert np.max(np.abs(a_ml - b_ml)) < 2e-2


# ----------------------------------------------------------------------------
# greedy verify


def run_verify(vh, X, W, draft, B, k, path):
    import torch
    acc, nid, ml = vh.spec_verify_greedy(to_torch_bf16(X), to_torch_bf16(W), to_torch(draft), B, k, path=path)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nid.cpu().numpy(), ml.cpu().numpy()


def check_verify(vh, orc, X, W, B, k, path, draft=None, seed=0, syn=None):
    _, o_nid, o_ml, o_sec = orc.verify_greedy(X, W, None, B, k)
    if draft is None:
        draft = syn.corrupt_ids(seed, syn.STREAM_CORRUPT, o_nid.reshape(B, k + 1)[:, :k].copy(), W.shape[0], 0.45)
    o_acc = np.array([orc.accept_len(o_nid[b * (k + 1): b * (k + 1) + k], draft[b]) for b in range(B)], np.int32)
    g_acc, g_nid, g_ml = run_verify(vh, X, W, draft, B, k, path)

    def score_of(r, v):
        return orc.dot_bf16(X[r], W[v])

    check_ids(g_nid, g_ml, o_nid, o_ml, o_sec, score_of, TOL_BF16)
    check_accept(g_acc, g_nid, o_acc, o_ml, o_sec, draft, B, k)
    return g_acc, g_nid


@pytest.mark.parametrize("path", [1, 2])
def test_verify_tiny_workload(vh, orc, syn, path):
    _, verify, W_full = syn.tiny_case()
    check_verify(vh, orc, verify.X, W_full, 1, 3, path, seed=1, syn=syn)


@pytest.mark.parametrize("path", [0, 1, 2])
# 8 / 9 rows split the CUDA-core groups; 128 / 129 switch from one CTA to the CTA pair
@pytest.mark.parametrize("B,k,V,H", [(1, 1, 1000, 64), (5, 3, 1000, 128), (3, 2, 129, 192), (64, 3, 3000, 256),
                                     (40, 3, 2049, 512), (20, 5, 700, 128), (1, 15, 517, 64), (2, 3, 1000, 128),
                                     (32, 3, 1300, 192), (43, 2, 900, 128)])
def test_verify_shapes(vh, orc, syn, path, B, k, V, H):
    W = syn.normal_bf16(V + H, 1, (V, H), 0.02)
    X = syn.normal_bf16(B + k, 4, (B * (k + 1), H), 1.0)
    check_verify(vh, orc, X, W, B, k, path, seed=B * 100 + k, syn=syn)


def test_verify_more_than_256_rows(vh, orc, syn):
    B, k, V, H = 100, 3, 1500, 128  # 400 rows: two tensor-core launches
    W = syn.normal_bf16(77, 1, (V, H), 0.02)
    X = syn.normal_bf16(78, 4, (B * (k + 1), H), 1.0)
    check_verify(vh, orc, X, W, B, k, 2, seed=79, syn=syn)


def test_verify_accept_cases(vh):
    """Hand-built acceptance fixtures through the GPU (one-hot head)."""
    cases = []
    with open(os.path.join(HERE, "golden", "accept_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, nxt, dr, a, _ = [p.split() for p in line.split("|")]
                if int(k[0]) == 3:
                    cases.append(([int(v) for v in nxt], [int(v) for v in dr], int(a[0])))
    B, k, H = len(cases), 3, 64
    W = np.zeros((16, H), np.uint16)
    for v in range(16):
        W[v, v] = 0x3F80  # one-hot head
    X = np.full((B * (k + 1), H), 0xBF80, np.uint16)  # -1 everywhere
    draft = np.zeros((B, k), np.int32)
    for b, (nxt, dr, _) in enumerate(cases):
        for j, t in enumerate(nxt):
            X[b * (k + 1) + j, t] = 0x4000  # 2.0 at the target id
        draft[b] = dr
    for path in (1, 2):
        acc, nid, _ = run_verify(vh, X, W, draft, B, k, path)
        assert list(acc) == [c[2] for c in cases]
        assert list(nid) == [t for c in cases for t in c[0]]


def _load_verify_golden():
    path = os.path.join(HERE, "golden", "verify_b64_k3_248320x2048.txt")
    rows, seqs, meta = {}, {}, {}
    with open(path) as f:
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


@pytest.mark.parametrize("path", [2, 1])
def test_verify_full_size_256x248320(vh, orc, syn, path):
    """Batched verify at full size (64 x 4 rows against the 248,320 x 2048 head)
    against the stored oracle results, plus the live oracle on sampled rows."""
    rows, seqs, meta = _load_verify_golden()
    case = syn.verify_case(B=64, k=3, H=2048, V=syn.V_FULL, seed_w=2, seed=4, with_head=True)
    assert syn.fingerprint(case.X) == int(meta["fingerprint_x"][0])
    sample = [int(v) for v in meta["fingerprint_w_rows"][:-1]]
    assert syn.fingerprint(np.ascontiguousarray(case.W[sample])) == int(meta["fingerprint_w_rows"][-1])
    draft = np.array([seqs[b][0] for b in range(64)], np.int32)
    o_nid = np.array([rows[r][0] for r in range(256)], np.int32)
    o_ml = np.array([rows[r][1] for r in range(256)])
    o_sec = np.array([rows[r][2] for r in range(256)])
    o_acc = np.array([seqs[b][1] for b in range(64)], np.int32)
    g_acc, g_nid, g_ml = run_verify(vh, case.X, case.W, draft, 64, 3, path)
    check_ids(g_nid, g_ml, o_nid, o_ml, o_sec, lambda r, v: orc.dot_bf16(case.X[r], case.W[v]), TOL_BF16)
    check_accept(g_acc, g_nid, o_acc, o_ml, o_sec, draft, 64, 3)
    # live oracle on a few rows (independent of the stored file)
    sample_rows = np.array([0, 37, 130, 255], np.int32)
    _, l_nid, l_ml, _ = orc.verify_greedy(case.X, case.W, None, 64, 3, rows=sample_rows)
    for r in sample_rows:
        assert l_nid[r] == o_nid[r] and l_ml[r] == np.float32(o_ml[r])


def test_cross_kernel_identity(vh, syn):
    """Draft kernel over the identity candidate set == verify's next_ids."""
    import torch
    V, H, B, k = 5000, 256, 8, 3
    W = syn.normal_bf16(31, 1, (V, H), 0.02)
    X = syn.normal_bf16(32, 4, (B * (k + 1), H), 1.0)
    draft = np.zeros((B, k), np.int32)
    ids, ml = vh.mtp_draft_head_argmax(to_torch_bf16(X), to_torch_bf16(W), torch.arange(V, dtype=torch.int32,
                                                                                          device="cuda"))
    for path in (1, 2):
        _, nid, vml = run_verify(vh, X, W, draft, B, k, path)
        mism = np.nonzero(nid != ids.cpu().numpy())[0]
        # the two kernels sum in different orders: ids may differ only on near-ties
        for r in mism:
            assert abs(float(vml[r]) - float(ml.cpu().numpy()[r])) < 1e-2


def test_verify_graph_capture_replays(vh, syn):
    """Calls are capture-safe: a CUDA graph of draft x3 + verify replays to the
    same results as direct calls."""
    import torch
    case = syn.draft_case(Vc=8192, H=512, B=1, steps=3, seed=12)
    V, B, k = 3000, 16, 3
    Wf = to_torch_bf16(syn.normal_bf16(13, 1, (V, 512), 0.02))
    X = to_torch_bf16(syn.normal_bf16(14, 4, (B * (k + 1), 512), 1.0))
    d = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    Wc, cc = to_torch_bf16(case.W), to_torch(case.cand_ids)
    xs = [to_torch_bf16(h) for h in case.hidden]
    ws_d, ws_v = vh.workspace(1), vh.workspace(B * (k + 1))
    ids = [torch.empty(1, dtype=torch.int32, device="cuda") for _ in range(3)]
    mls = [torch.empty(1, dtype=torch.float32, device="cuda") for _ in range(3)]
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nid = torch.empty(B * (k + 1), dtype=torch.int32, device="cuda")

    def step():
        for i in range(3):
            vh.mtp_draft_head_argmax(xs[i], Wc, cc, ids=ids[i], maxlogit=mls[i], ws=ws_d)
        vh.spec_verify_greedy(X, Wf, d, B, k, accept_len=acc, next_ids=nid, ws=ws_v, want_maxlogit=False)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    want = [t.clone() for t in ids + [acc, nid]]
    for t in ids + [acc, nid]:
        t.fill_(-7)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        for t in ids + [acc, nid]:
            t.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(ids + [acc, nid], want):
            assert torch.equal(a, b)
    assert int(ws_d.count_nonzero()) == 0 and int(ws_v.count_nonzero()) == 0


def test_error_status_on_gpu(vh):
    import torch
    x = torch.zeros(1, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(10, 64, dtype=torch.bfloat16, device="cuda")
    c = torch.arange(10, dtype=torch.int32, device="cuda")
    with pytest.raises(vh.VHError) as e:
        vh.mtp_draft_head_argmax(x, W, c, ws=torch.zeros(8, dtype=torch.uint8, device="cuda"))
    assert e.value.status == vh.VH_ERR_WORKSPACE
    flat = torch.zeros(10 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vh.VHError) as e:
        vh.mtp_draft_head_argmax(x, flat[8:].view(10, 64), c)  # W 16 bytes off a 32-byte boundary
    assert e.value.status == vh.VH_ERR_ALIGN
    with pytest.raises(vh.VHError) as e:
        vh.spec_verify_greedy(torch.zeros(4, 80, dtype=torch.bfloat16, device="cuda"),
                              torch.zeros(10, 80, dtype=torch.bfloat16, device="cuda"),
                              torch.zeros(1, 3, dtype=torch.int32, device="cuda"), 1, 3, path=vh.VH_PATH_TENSOR)
    assert e.value.status == vh.VH_ERR_SHAPE  # tensor path needs H % 64 == 0


# ----------------------------------------------------------------------------
# greedy verify over a 4-bit head


def run_verify_nvfp4(vh, X, q, s, g, draft, B, k):
    import torch
    acc, nid, ml = vh.spec_verify_greedy_nvfp4(to_torch_bf16(X), to_torch(q), to_torch(s), g, to_torch(draft), B, k)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nid.cpu().numpy(), ml.cpu().numpy()


def check_verify_nvfp4(vh, orc, syn, X, q, s, g, B, k, seed):
    V = q.shape[0]
    _, o_nid, o_ml, o_sec = orc.verify_greedy_nvfp4(X, q, s, g, None, B, k)
    draft = syn.corrupt_ids(seed, syn.STREAM_CORRUPT, o_nid.reshape(B, k + 1)[:, :k].copy(), V, 0.45)
    o_acc = np.array([orc.accept_len(o_nid[b * (k + 1): b * (k + 1) + k], draft[b]) for b in range(B)], np.int32)
    g_acc, g_nid, g_ml = run_verify_nvfp4(vh, X, q, s, g, draft, B, k)

    def score_of(r, v):
        return float(orc.scores_nvfp4(X[r], q[v:v + 1], s[v:v + 1], g, nthreads=1)[0])

    check_ids(g_nid, g_ml, o_nid, o_ml, o_sec, score_of, TOL_4BIT)
    check_accept(g_acc, g_nid, o_acc, o_ml, o_sec, draft, B, k)


# rows <= 16: warp-level MMAs in groups of 8 (H = 256 * 2^i <= 4096) or one
# k_nvfp4_tc pass (other H % 512 == 0); 17..128 rows: CTA pair with N = 128; 129..256:
# N = 256; > 256 rows: groups of 256; H = 2048 wraps the raw-code ring along K;
# V = 40,000 gives every CTA pair several tiles (accumulator double buffering)
@pytest.mark.parametrize("B,k,V,H", [(1, 3, 1000, 512), (4, 3, 3000, 1024), (5, 3, 2000, 512), (3, 2, 700, 256),
                                     (2, 1, 129, 64), (16, 3, 1500, 512), (33, 3, 2500, 512), (64, 3, 1100, 1024),
                                     (75, 3, 900, 512), (16, 3, 3000, 2048), (20, 3, 40_000, 512),
                                     (7, 15, 1300, 512), (9, 1, 800, 512), (32, 3, 1300, 512), (43, 2, 900, 1024),
                                     (2, 3, 17, 2048), (1, 3, 3001, 1536), (3, 3, 1000, 4096)])
def test_verify_nvfp4_shapes(vh, orc, syn, B, k, V, H):
    w = syn.normal_f32(V + H, 6, (V, H), 0.02)
    q, s, g = syn.nvfp4_quantize(w)
    X = syn.normal_bf16(B + k, 4, (B * (k + 1), H), 1.0)
    check_verify_nvfp4(vh, orc, syn, X, q, s, g, B, k, seed=V)


def test_verify_nvfp4_full_head_65536x4096(vh, orc, syn):
    """4 sequences x 4 positions against the 65,536 x 4096 4-bit head."""
    c = syn.nvfp4_case(Vc=65_536, H=4096, B=1, steps=1, seed=5)
    X = syn.normal_bf16(7, syn.STREAM_VHIDDEN, (16, 4096), 1.0)
    check_verify_nvfp4(vh, orc, syn, X, c.q, c.s, c.g, 4, 3, seed=7)


def test_verify_nvfp4_full_head_248320x2048(vh, orc, syn):
    """64 sequences x 4 positions against the full 248,320 x 2048 4-bit head
    (the CTA-pair kernel's launch in the bench).  The live oracle scores the
    rows of three sequences; their draft ids are the oracle's greedy ids
    corrupted w.p. 0.45, the other sequences' draft ids are uniform ids."""
    B, k, V = 64, 3, syn.V_FULL
    q, s, g = syn.nvfp4_head(seed=2, V=V, H=2048)
    X = syn.verify_case(B=B, k=k, H=2048, V=V, seed=4, with_head=False).X
    seqs = [0, 29, 63]
    rows = np.array([b * (k + 1) + j for b in seqs for j in range(k + 1)], np.int32)
    _, o_nid, o_ml, o_sec = orc.verify_greedy_nvfp4(X, q, s, g, None, B, k, rows=rows)
    draft = syn.corrupt_ids(11, syn.STREAM_CORRUPT, np.zeros((B, k), np.int32), V, 1.0)  # uniform ids != 0
    truth = np.stack([o_nid[b * (k + 1): b * (k + 1) + k] for b in seqs])
    draft[seqs] = syn.corrupt_ids(12, syn.STREAM_CORRUPT, truth, V, 0.45)
    g_acc, g_nid, g_ml = run_verify_nvfp4(vh, X, q, s, g, draft, B, k)
    np.testing.assert_array_equal(g_acc, accept_scan(g_nid, draft, B, k))
    assert np.all((g_nid >= 0) & (g_nid < V))

    def score_of(r, v):
        return float(orc.scores_nvfp4(X[rows[r]], q[v:v + 1], s[v:v + 1], g, nthreads=1)[0])

    check_ids(g_nid[rows], g_ml[rows], o_nid[rows], o_ml[rows], o_sec[rows], score_of, TOL_4BIT)
    for i, b in enumerate(seqs):
        o_acc = orc.accept_len(o_nid[b * (k + 1): b * (k + 1) + k], draft[b])
        r = rows[i * (k + 1): i * (k + 1) + min(o_acc, k - 1) + 1]
        if all(float(o_ml[x]) - float(o_sec[x]) > 1e-2 for x in r):
            assert g_acc[b] == o_acc, (b, g_acc[b], o_acc)


def test_verify_nvfp4_accept_cases(vh):
    cases = []
    with open(os.path.join(HERE, "golden", "accept_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, nxt, dr, a, _ = [p.split() for p in line.split("|")]
                if int(k[0]) == 3:
                    cases.append(([int(v) for v in nxt], [int(v) for v in dr], int(a[0])))
    V = H = 512
    q = np.zeros((V, H // 2), np.uint8)
    for v in range(V):
        q[v, v // 2] = 0x02 if v % 2 == 0 else 0x20  # one-hot 4-bit head: weight 1.0 at h == v
    s = np.full((V, H // 16), 0x38, np.uint8)
    B, k = len(cases), 3
    X = np.full((B * (k + 1), H), 0xBF80, np.uint16)
    draft = np.zeros((B, k), np.int32)
    for b, (nxt, dr, _) in enumerate(cases):
        for j, t in enumerate(nxt):
            X[b * (k + 1) + j, t] = 0x4000
        draft[b] = dr
    acc, nid, _ = run_verify_nvfp4(vh, X, q, s, 1.0, draft, B, k)
    assert list(acc) == [c[2] for c in cases]
    assert list(nid) == [t for c in cases for t in c[0]]


def _load_golden(name):
    rows, seqs, meta = {}, {}, {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            p = line.split()
            if not p or p[0].startswith("#"):
                continue
            if p[0] == "row":
                rows[int(p[1])] = (int(p[2]), float.fromhex(p[3]), float.fromhex(p[4]))
            elif p[0] == "seq":
                seqs[int(p[1])] = ([int(v) for v in p[2:-1]], int(p[-1]))
            else:
                meta[p[0]] = p[1:]
    return rows, seqs, meta


def test_verify_nvfp4_full_size_all_rows_golden(vh, orc, syn):
    """64 x 4 rows against the full 248,320 x 2048 4-bit head: all 256 rows
    and all 64 accept lengths against the stored oracle results
    (tests/golden/make_verify_nvfp4_golden.py), plus the live oracle on a few
    sampled rows."""
    rows, seqs, meta = _load_golden("verify_nvfp4_b64_k3_248320x2048.txt")
    B, k, V = 64, 3, syn.V_FULL
    q, s, g = syn.nvfp4_head(seed=2, V=V, H=2048)
    X = syn.verify_case(B=B, k=k, H=2048, V=V, seed=4, with_head=False).X
    assert float.fromhex(meta["tensor_scale"][0]) == float(g)
    assert syn.fingerprint(X) == int(meta["fingerprint_x"][0])
    sample = [int(v) for v in meta["fingerprint_q_rows"][:-1]]
    assert syn.fingerprint(np.ascontiguousarray(q[sample])) == int(meta["fingerprint_q_rows"][-1])
    assert syn.fingerprint(np.ascontiguousarray(s[sample])) == int(meta["fingerprint_s_rows"][-1])
    draft = np.array([seqs[b][0] for b in range(B)], np.int32)
    o_nid = np.array([rows[r][0] for r in range(256)], np.int32)
    o_ml = np.array([rows[r][1] for r in range(256)])
    o_sec = np.array([rows[r][2] for r in range(256)])
    o_acc = np.array([seqs[b][1] for b in range(B)], np.int32)
    g_acc, g_nid, g_ml = run_verify_nvfp4(vh, X, q, s, g, draft, B, k)

    def score_of(r, v):
        return float(orc.scores_nvfp4(X[r], q[v:v + 1], s[v:v + 1], g, nthreads=1)[0])

    n_exact = check_ids(g_nid, g_ml, o_nid, o_ml, o_sec, score_of, TOL_4BIT)
    assert n_exact >= 200  # most rows have a clear winner
    check_accept(g_acc, g_nid, o_acc, o_ml, o_sec, draft, B, k)
    sample_rows = np.array([3, 100, 254], np.int32)
    _, l_nid, l_ml, _ = orc.verify_greedy_nvfp4(X, q, s, g, None, B, k, rows=sample_rows)
    for r in sample_rows:
        assert l_nid[r] == o_nid[r] and l_ml[r] == np.float32(o_ml[r])
