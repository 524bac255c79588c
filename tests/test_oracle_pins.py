"""Pins for the CPU oracle: each test checks it against something other than
itself (exact integer arithmetic, fp64 brute force, closed forms, a library
routine, hand-worked fixtures, invariants).  CPU only."""
import os
from fractions import Fraction

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


def bf16_bits(values):
    """Exact bf16 bit patterns of values that bf16 represents exactly."""
    f = np.asarray(values, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)


def f32_of(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# bf16 widening

def test_bf16_widening_exhaustive(oracle_mod):
    # every finite bf16 pattern widens to the float32 whose upper half it is
    for b in list(range(0, 0x7F80, 97)) + [0x0001, 0x007F, 0x3F80, 0x4049, 0x7F7F, 0x8000, 0xBF80, 0xFF7F]:
        want = float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])
        assert oracle_mod.bf16_to_f32(b) == want


# --------------------------------------------------------------------------
# Exact-integer brute force: small integer inputs make every fp32 sum exact,
# so scores, argmax and the lowest-id tie rule must match integer arithmetic.

@pytest.mark.parametrize("seed", range(12))
def test_draft_exact_integers(oracle_mod, seed):
    rng = np.random.default_rng(1000 + seed)
    B, H, Vc = int(rng.integers(1, 4)), int(rng.integers(1, 17)), int(rng.integers(1, 65))
    xi = rng.integers(-3, 4, size=(B, H))
    Wi = rng.integers(-2, 3, size=(Vc, H))
    cand = np.sort(rng.choice(5000, size=Vc, replace=False)).astype(np.int32)
    ids, ml, sec = oracle_mod.draft_argmax(bf16_bits(xi), bf16_bits(Wi), cand)
    for b in range(B):
        s = [int(sum(int(xi[b, h]) * int(Wi[c, h]) for h in range(H))) for c in range(Vc)]
        best = max(s)
        cstar = s.index(best)  # first (lowest index, hence lowest id) maximum
        assert ids[b] == cand[cstar]
        assert ml[b] == best
        others = [v for i, v in enumerate(s) if i != cstar]
        if others:
            assert sec[b] == max(others)


@pytest.mark.parametrize("seed", range(8))
def test_verify_exact_integers(oracle_mod, seed):
    rng = np.random.default_rng(2000 + seed)
    B, k = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    H, V = int(rng.integers(1, 13)), int(rng.integers(2, 50))
    R = B * (k + 1)
    Xi = rng.integers(-2, 3, size=(R, H))
    Wi = rng.integers(-2, 3, size=(V, H))
    S = [[sum(int(Xi[r, h]) * int(Wi[v, h]) for h in range(H)) for v in range(V)] for r in range(R)]
    nxt = np.array([row.index(max(row)) for row in S], dtype=np.int32)
    # draft: the true ids with some positions changed, so every accept length occurs
    draft = nxt.reshape(B, k + 1)[:, :k].copy()
    for b in range(B):
        j = int(rng.integers(0, k + 1))
        if j < k:
            draft[b, j] = (draft[b, j] + 1 + int(rng.integers(0, V - 1))) % V
    acc, got, ml, _ = oracle_mod.verify_greedy(bf16_bits(Xi), bf16_bits(Wi), draft, B, k)
    np.testing.assert_array_equal(got, nxt)
    np.testing.assert_array_equal(ml, [max(row) for row in S])
    for b in range(B):
        a = 0
        while a < k and nxt[b * (k + 1) + a] == draft[b, a]:
            a += 1
        assert acc[b] == a


def test_ties_take_lowest_global_id(oracle_mod):
    H = 8
    W = np.zeros((6, H), np.float32)
    W[[1, 3, 4]] = 1.0  # three equal best rows
    x = np.ones((1, H), np.float32)
    cand = np.array([3, 9, 11, 40, 41, 100], np.int32)
    ids, ml, sec = oracle_mod.draft_argmax(bf16_bits(x), bf16_bits(W), cand)
    assert ids[0] == 9 and ml[0] == 8.0 and sec[0] == 8.0


# --------------------------------------------------------------------------
# fp64 brute force on random normal inputs: the fp32 sequential sum stays
# within a rounding bound of the exact (fp64) score.

@pytest.mark.parametrize("seed", range(6))
def test_draft_fp64_bruteforce(oracle_mod, seed):
    rng = np.random.default_rng(3000 + seed)
    B, H, Vc = 2, 16, 64
    xb = (rng.standard_normal((B, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    Wb = ((0.02 * rng.standard_normal((Vc, H))).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    cand = np.arange(Vc, dtype=np.int32) * 3 + 1
    ids, ml, sec = oracle_mod.draft_argmax(xb, Wb, cand)
    xf, Wf = f32_of(xb).astype(np.float64), f32_of(Wb).astype(np.float64)
    for b in range(B):
        s = [sum(xf[b, h] * Wf[c, h] for h in range(H)) for c in range(Vc)]
        order = np.argsort(s)[::-1]
        best = order[0]
        assert abs(ml[b] - s[best]) < 1e-5
        if s[order[0]] - s[order[1]] > 1e-4:
            assert ids[b] == cand[best]


def test_tiny_workload_against_fp64_matmul(oracle_mod, synth_mod):
    """Tiny workload (4096 x 256 head, 1,024 candidates): oracle vs numpy's
    fp64 matmul; ids must agree wherever the fp64 top-2 gap exceeds 1e-3."""
    draft, verify, W_full = synth_mod.tiny_case()
    Wc = f32_of(draft.W).astype(np.float64)
    for x in draft.hidden:
        ids, ml, _ = oracle_mod.draft_argmax(x, draft.W, draft.cand_ids)
        s = Wc @ f32_of(x[0]).astype(np.float64)
        order = np.argsort(-s, kind="stable")
        assert abs(ml[0] - s[order[0]]) < 1e-4
        if s[order[0]] - s[order[1]] > 1e-3:
            assert ids[0] == draft.cand_ids[order[0]]
    _, nid, ml, _ = oracle_mod.verify_greedy(verify.X, W_full, None, verify.B, verify.k)
    S = f32_of(verify.X).astype(np.float64) @ f32_of(W_full).astype(np.float64).T
    for r in range(S.shape[0]):
        order = np.argsort(-S[r], kind="stable")
        assert abs(ml[r] - S[r, order[0]]) < 1e-4
        if S[r, order[0]] - S[r, order[1]] > 1e-3:
            assert nid[r] == order[0]


# --------------------------------------------------------------------------
# Invariant: restricted argmax vs full argmax (W_cand = W_full[cand]).

def test_restricted_matches_full_when_top1_in_candidates(oracle_mod, synth_mod):
    draft, verify, W_full = synth_mod.tiny_case()
    V = W_full.shape[0]
    all_ids = np.arange(V, dtype=np.int32)
    hits = 0
    for t in range(12):
        x = synth_mod.normal_bf16(100 + t, synth_mod.STREAM_HIDDEN, (1, W_full.shape[1]), 1.0)
        fid, fml, _ = oracle_mod.draft_argmax(x, W_full, all_ids)
        # half of the trials force the full top-1 into the candidate set
        cand = draft.cand_ids
        if t % 2 == 0 and fid[0] not in cand:
            cand = np.sort(np.concatenate([cand[:-1], [fid[0]]])).astype(np.int32)
            cand = np.unique(cand)
        Wc = np.ascontiguousarray(W_full[cand])
        rid, rml, _ = oracle_mod.draft_argmax(x, Wc, cand)
        if fid[0] in cand:
            hits += 1
            assert rid[0] == fid[0] and rml[0] == fml[0]
        else:
            assert rml[0] <= fml[0] and rid[0] != fid[0]
    assert hits >= 6


def test_verify_equals_draft_over_identity_candidates(oracle_mod, synth_mod):
    _, verify, W_full = synth_mod.tiny_case()
    _, nid, ml, _ = oracle_mod.verify_greedy(verify.X, W_full, None, verify.B, verify.k)
    ids, dml, _ = oracle_mod.draft_argmax(verify.X, W_full, np.arange(W_full.shape[0], dtype=np.int32))
    np.testing.assert_array_equal(ids, nid)
    np.testing.assert_array_equal(dml, ml)


# --------------------------------------------------------------------------
# Closed-form special cases.

def test_single_candidate(oracle_mod):
    rng = np.random.default_rng(5)
    x = bf16_bits(rng.integers(-3, 4, size=(3, 8)))
    W = bf16_bits(rng.integers(-3, 4, size=(1, 8)))
    ids, ml, _ = oracle_mod.draft_argmax(x, W, np.array([777], np.int32))
    assert list(ids) == [777] * 3
    want = [sum(float(a) * float(b) for a, b in zip(f32_of(x)[i], f32_of(W)[0])) for i in range(3)]
    assert list(ml) == want  # small integers: exact


def test_zero_head_ties_to_first_candidate(oracle_mod):
    x = bf16_bits(np.arange(1, 17, dtype=np.float32).reshape(2, 8))
    W = np.zeros((5, 8), np.uint16)
    cand = np.array([2, 4, 6, 8, 10], np.int32)
    ids, ml, sec = oracle_mod.draft_argmax(x, W, cand)
    assert list(ids) == [2, 2] and list(ml) == [0.0, 0.0] and list(sec) == [0.0, 0.0]


def test_negative_zero_equals_positive_zero(oracle_mod):
    # candidate 0 scores -0 (negative x against +w), candidate 1 scores +0
    x = bf16_bits([[-1.0, 0.0]])
    W = bf16_bits([[0.0, 0.0], [0.0, 0.0]])
    W[0, 0] = 0x0000  # +0 * -1 = -0
    ids, ml, _ = oracle_mod.draft_argmax(x, W, np.array([5, 6], np.int32))
    assert ids[0] == 5 and ml[0] == 0.0 and not np.signbit(ml[0])


def test_one_hot_head(oracle_mod):
    # W[c, h] = alpha if h == c mod H: the winner is the lowest-id candidate
    # sitting on the largest hidden coordinate
    H, Vc, alpha = 16, 48, 0.5
    W = np.zeros((Vc, H), np.float32)
    for c in range(Vc):
        W[c, c % H] = alpha
    x = np.zeros((1, H), np.float32)
    x[0, 5] = 3.0
    x[0, 9] = 2.0
    cand = np.arange(Vc, dtype=np.int32) * 2 + 100
    ids, ml, sec = oracle_mod.draft_argmax(bf16_bits(x), bf16_bits(W), cand)
    assert ids[0] == cand[5] and ml[0] == 1.5 and sec[0] == 1.5  # c = 5, 21, 37 tie


def test_duplicate_rows_take_lowest_id(oracle_mod, synth_mod):
    W = synth_mod.normal_bf16(9, 1, (10, 32), 0.02)
    W[7] = W[2]
    x = synth_mod.normal_bf16(9, 3, (1, 32), 1.0)
    s = f32_of(W).astype(np.float64) @ f32_of(x[0]).astype(np.float64)
    # make row 2 (and its duplicate, row 7) the clear winner
    if np.argmax(s) not in (2, 7):
        W[2] = W[7] = bf16_bits(np.where(f32_of(x[0]) > 0, 0.5, -0.5).astype(np.float32))
    cand = np.arange(10, dtype=np.int32) + 50
    ids, ml, sec = oracle_mod.draft_argmax(x, W, cand)
    assert ids[0] == 52 and sec[0] == ml[0]


# --------------------------------------------------------------------------
# Hand-built acceptance cases.

def _parse_accept_cases():
    cases = []
    with open(os.path.join(GOLDEN, "accept_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, nxt, dr, a, em = [p.split() for p in line.split("|")]
            cases.append((int(k[0]), [int(v) for v in nxt], [int(v) for v in dr], int(a[0]), [int(v) for v in em]))
    return cases


def test_acceptance_fixtures(oracle_mod):
    cases = _parse_accept_cases()
    assert len(cases) >= 8
    V = H = 8
    W = bf16_bits(np.eye(V, H, dtype=np.float32))  # one-hot head: score[v] = X[r, v]
    for k, nxt, draft, want, emitted in cases:
        X = np.full((k + 1, H), -1.0, np.float32)
        for j, t in enumerate(nxt):
            X[j, t] = 2.0
        acc, got, _, _ = oracle_mod.verify_greedy(bf16_bits(X), W, np.array([draft], np.int32), 1, k)
        assert list(got) == nxt
        assert acc[0] == want
        assert oracle_mod.accept_len(got, draft) == want
        # emitted tokens: accepted draft prefix, then the target's own id
        assert draft[:want] + [int(got[want])] == emitted


def test_acceptance_multi_sequence_layout(oracle_mod):
    # rows are [b][j]: sequence b owns rows b*(k+1) .. b*(k+1)+k
    cases = [c for c in _parse_accept_cases() if c[0] == 3]
    B, k, V = len(cases), 3, 8
    W = bf16_bits(np.eye(V, dtype=np.float32))
    X = np.full((B * (k + 1), V), -1.0, np.float32)
    draft = np.zeros((B, k), np.int32)
    for b, (_, nxt, dr, _, _) in enumerate(cases):
        for j, t in enumerate(nxt):
            X[b * (k + 1) + j, t] = 2.0
        draft[b] = dr
    acc, _, _, _ = oracle_mod.verify_greedy(bf16_bits(X), W, draft, B, k)
    assert list(acc) == [c[3] for c in cases]


# --------------------------------------------------------------------------
# 4-bit formats: exhaustive tables against closed forms and a library routine.

def _e2m1_closed(code):
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return -v if s else v


def _e4m3_closed(code):
    s, e, m = (code >> 7) & 1, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return None
    v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else Fraction(2) ** (e - 7) * (1 + Fraction(m, 8))
    return -v if s else v


def test_e2m1_exhaustive(oracle_mod):
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # the OCP FP4 (E2M1) magnitudes
    for code in range(16):
        got = oracle_mod.e2m1_value(code)
        assert got == float(_e2m1_closed(code))
        assert abs(got) == table[code & 7]
        assert np.signbit(got) == bool(code & 8)


def test_e4m3_exhaustive(oracle_mod):
    import torch
    lib_vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for code in range(256):
        got = oracle_mod.e4m3_value(code)
        want = _e4m3_closed(code)
        if want is None:
            assert np.isnan(got) and np.isnan(lib_vals[code])
            continue
        assert got == float(want)
        assert got == lib_vals[code]
    assert oracle_mod.e4m3_value(0x7E) == 448.0 and oracle_mod.e4m3_value(0x01) == 2.0 ** -9


def _parse_nvfp4_cases():
    rows, scores, argmaxes = {}, [], []
    with open(os.path.join(GOLDEN, "nvfp4_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [p.strip() for p in line.split("|")]
            head = parts[0].split()

            def hidden(spec):
                out = {}
                for tok in spec.split():
                    h, v = tok.split(":")
                    out[int(h)] = float(v)
                return out

            if head[0] == "row":
                rows[int(head[1])] = (bytes.fromhex(parts[1]), bytes.fromhex(parts[2]))
            elif head[0] == "score":
                scores.append((int(head[1]), hidden(parts[1]), float(parts[2])))
            elif head[0] == "argmax":
                argmaxes.append((hidden(parts[1]), int(parts[2])))
    return rows, scores, argmaxes


def test_nvfp4_hand_worked_rows(oracle_mod):
    rows, scores, argmaxes = _parse_nvfp4_cases()
    H, g = 32, 0.5
    q = np.array([list(rows[r][0]) for r in sorted(rows)], np.uint8)
    s = np.array([list(rows[r][1]) for r in sorted(rows)], np.uint8)
    for r, hid, want in scores:
        x = np.zeros((1, H), np.float32)
        for h, v in hid.items():
            x[0, h] = v
        got = oracle_mod.scores_nvfp4(bf16_bits(x)[0], q, s, g)
        assert got[r] == want, (r, hid, got[r], want)
    cand = np.array([10, 20, 30], np.int32)
    for hid, want in argmaxes:
        x = np.zeros((1, H), np.float32)
        for h, v in hid.items():
            x[0, h] = v
        ids, _, _ = oracle_mod.draft_argmax_nvfp4(bf16_bits(x), q, s, g, cand)
        assert ids[0] == want


@pytest.mark.parametrize("seed", range(4))
def test_nvfp4_fp64_bruteforce(oracle_mod, seed):
    """Random codes and scales, g != 1: oracle scores vs exact rational decode
    summed in fp64."""
    rng = np.random.default_rng(4000 + seed)
    Vc, H, g = 12, 48, 0.0003
    q = rng.integers(0, 256, size=(Vc, H // 2), dtype=np.uint8)
    s = rng.integers(0, 0x7F, size=(Vc, H // 16), dtype=np.uint8)  # positive, finite scales
    xb = (rng.standard_normal((1, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x = f32_of(xb[0]).astype(np.float64)
    got = oracle_mod.scores_nvfp4(xb[0], q, s, g)
    dec = oracle_mod.decode_nvfp4(q, s, g)
    for c in range(Vc):
        exact = 0.0
        for h in range(H):
            byte = int(q[c, h // 2])
            code = (byte >> 4) if h % 2 else (byte & 15)
            w = float(_e2m1_closed(code) * _e4m3_closed(int(s[c, h // 16])) * Fraction(g))
            assert abs(dec[c, h] - w) <= abs(w) * 2 ** -23  # one fp32 rounding
            exact += x[h] * w
        assert abs(got[c] - exact) < 1e-6 + 1e-5 * abs(exact)


def test_nvfp4_equals_bf16_on_representable_head(oracle_mod):
    """With g = 1 every decoded weight (<= 6 significant bits) is a bf16
    value, so the 4-bit oracle must equal the bf16 oracle on the decoded head."""
    rng = np.random.default_rng(11)
    Vc, H = 40, 64
    q = rng.integers(0, 256, size=(Vc, H // 2), dtype=np.uint8)
    s = rng.integers(0x20, 0x48, size=(Vc, H // 16), dtype=np.uint8)
    dec = oracle_mod.decode_nvfp4(q, s, 1.0)
    Wb = bf16_bits(dec)
    xb = (rng.standard_normal((3, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    cand = np.arange(Vc, dtype=np.int32) * 7
    a = oracle_mod.draft_argmax_nvfp4(xb, q, s, 1.0, cand)
    b = oracle_mod.draft_argmax(xb, Wb, cand)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


# --------------------------------------------------------------------------
# Gathered candidate rows (ids in any order, repeats, out-of-range entries).

@pytest.mark.parametrize("seed", range(8))
def test_gather_exact_integers(oracle_mod, seed):
    rng = np.random.default_rng(5000 + seed)
    V, H, B = int(rng.integers(2, 40)), int(rng.integers(1, 12)), int(rng.integers(1, 4))
    Wi = rng.integers(-2, 3, size=(V, H))
    xi = rng.integers(-2, 3, size=(B, H))
    n = int(rng.integers(1, 60))
    rows = rng.integers(-3, V + 3, size=n).astype(np.int32)  # includes out-of-range entries
    rows[0] = int(rng.integers(0, V))                        # at least one valid entry
    ids, ml, _ = oracle_mod.draft_argmax_gather(bf16_bits(xi), bf16_bits(Wi), rows)
    for b in range(B):
        valid = [int(r) for r in rows if 0 <= r < V]
        s = {r: sum(int(xi[b, h]) * int(Wi[r, h]) for h in range(H)) for r in valid}
        best = max(s.values())
        assert ml[b] == best
        assert ids[b] == min(r for r, v in s.items() if v == best)  # lowest id on ties, any list order


def test_gather_equals_sorted_candidate_table(oracle_mod, synth_mod):
    _, verify, W_full = synth_mod.tiny_case()
    rng = np.random.default_rng(3)
    rows = rng.integers(0, W_full.shape[0], size=700).astype(np.int32)
    uniq = np.unique(rows).astype(np.int32)
    x = synth_mod.normal_bf16(8, synth_mod.STREAM_HIDDEN, (3, W_full.shape[1]), 1.0)
    a = oracle_mod.draft_argmax_gather(x, W_full, rows)
    b = oracle_mod.draft_argmax(x, np.ascontiguousarray(W_full[uniq]), uniq)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_nvfp4_verify_equals_bf16_verify_on_representable_head(oracle_mod):
    rng = np.random.default_rng(21)
    V, H, B, k = 300, 64, 3, 3
    q = rng.integers(0, 256, size=(V, H // 2), dtype=np.uint8)
    s = rng.integers(0x20, 0x48, size=(V, H // 16), dtype=np.uint8)
    Wb = bf16_bits(oracle_mod.decode_nvfp4(q, s, 1.0))
    X = (rng.standard_normal((B * (k + 1), H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    draft = rng.integers(0, V, size=(B, k)).astype(np.int32)
    a = oracle_mod.verify_greedy_nvfp4(X, q, s, 1.0, draft, B, k)
    b = oracle_mod.verify_greedy(X, Wb, draft, B, k)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_nvfp4_verify_acceptance_fixtures(oracle_mod):
    """One-hot 4-bit head (code 2 = 1.0, scale 0x38 = 1.0): row j's greedy id is
    the position of its peak; the hand-built acceptance cases must hold."""
    cases = [c for c in _parse_accept_cases() if c[0] == 3]
    V = H = 64
    q = np.zeros((V, H // 2), np.uint8)
    for v in range(V):
        q[v, v // 2] = 0x02 if v % 2 == 0 else 0x20
    s = np.full((V, H // 16), 0x38, np.uint8)
    B, k = len(cases), 3
    X = np.full((B * (k + 1), H), -1.0, np.float32)
    draft = np.zeros((B, k), np.int32)
    for b, (_, nxt, dr, _, _) in enumerate(cases):
        for j, t in enumerate(nxt):
            X[b * (k + 1) + j, t] = 2.0
        draft[b] = dr
    acc, nid, _, _ = oracle_mod.verify_greedy_nvfp4(bf16_bits(X), q, s, 1.0, draft, B, k)
    assert list(acc) == [c[3] for c in cases]
    assert list(nid) == [t for c in cases for t in c[1]]
