"""Seeded input generators: determinism, structure and distributions (CPU)."""
import numpy as np


def f32_of(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def test_normal_is_counter_based(synth_mod):
    a = synth_mod.normal_bf16(3, 1, (64, 32), 0.02)
    b = synth_mod.normal_bf16(3, 1, (64, 32), 0.02)
    np.testing.assert_array_equal(a, b)
    # any slice regenerates from its offset alone
    c = synth_mod.normal_bf16(3, 1, (10, 32), 0.02, offset=20 * 32)
    np.testing.assert_array_equal(a[20:30], c)
    rows = np.array([63, 0, 17], np.int32)
    np.testing.assert_array_equal(synth_mod.normal_bf16_rows(3, 1, rows, 32, 0.02), a[rows])
    # other seeds / streams differ
    assert not np.array_equal(a, synth_mod.normal_bf16(4, 1, (64, 32), 0.02))
    assert not np.array_equal(a, synth_mod.normal_bf16(3, 2, (64, 32), 0.02))


def test_normal_moments(synth_mod):
    z = f32_of(synth_mod.normal_bf16(1, 1, (1 << 20,), 1.0)).astype(np.float64)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    assert abs(np.mean(np.abs(z) > 1.96) - 0.05) < 2e-3  # two-sided 5% tail
    w = f32_of(synth_mod.normal_bf16(1, 1, (1 << 18,), 0.02)).astype(np.float64)
    assert abs(w.std() - 0.02) < 2e-4


def test_sorted_subset(synth_mod):
    for n, k in [(10, 10), (4096, 1024), (248_320, 65_536), (248_320, 1)]:
        s = synth_mod.sorted_subset(2, synth_mod.STREAM_CAND, n, k)
        assert s.size == k and s.dtype == np.int32
        assert np.all(np.diff(s) > 0) and s[0] >= 0 and s[-1] < n
    s1 = synth_mod.sorted_subset(2, 2, 248_320, 65_536)
    s2 = synth_mod.sorted_subset(3, 2, 248_320, 65_536)
    assert not np.array_equal(s1, s2)
    # roughly uniform over the range
    assert abs(np.mean(s1) / 248_320 - 0.5) < 0.01


def test_corruption(synth_mod):
    V = 248_320
    truth = np.arange(0, 64 * 3 * 200, dtype=np.int32) % V
    out = synth_mod.corrupt_ids(4, synth_mod.STREAM_CORRUPT, truth, V, 0.45)
    changed = out != truth
    assert abs(changed.mean() - 0.45) < 0.02
    assert np.all((out >= 0) & (out < V))
    # p = 1 always changes the id, p = 0 never does
    assert np.all(synth_mod.corrupt_ids(1, 5, truth, V, 1.0) != truth)
    np.testing.assert_array_equal(synth_mod.corrupt_ids(1, 5, truth, V, 0.0), truth)


def test_accept_length_distribution(synth_mod):
    # with independent corruption p = 0.45 and k = 3: P(a = j) = 0.45 * 0.55^j, P(a = 3) = 0.55^3
    k, n = 3, 20000
    truth = np.zeros(n * k, np.int32)
    d = synth_mod.corrupt_ids(8, 5, truth, 1000, 0.45).reshape(n, k)
    a = np.argmax(np.concatenate([d != 0, np.ones((n, 1), bool)], axis=1), axis=1)  # first mismatch
    hist = np.bincount(a, minlength=4) / n
    want = [0.45, 0.45 * 0.55, 0.45 * 0.55 ** 2, 0.55 ** 3]
    assert np.max(np.abs(hist - want)) < 0.015
    assert abs(a.mean() - sum(j * p for j, p in enumerate(want))) < 0.03


def test_nvfp4_encoder_round_trip(synth_mod, oracle_mod):
    w = synth_mod.normal_f32(5, synth_mod.STREAM_W4, (64, 256), 0.02)
    q, s, g = synth_mod.nvfp4_quantize(w)
    assert q.shape == (64, 128) and s.shape == (64, 16)
    assert abs(g - np.abs(w).max() / (6 * 448)) < 1e-9
    dec = oracle_mod.decode_nvfp4(q, s, g).astype(np.float64)
    # per block: error at most half an E2M1 step at the block's scale (step <= 2 * scale
    # for magnitudes in [4, 6]), plus the scale's own rounding
    for r in range(64):
        for b in range(16):
            blk = slice(b * 16, b * 16 + 16)
            scale = oracle_mod.e4m3_value(int(s[r, b])) * g
            err = np.abs(dec[r, blk] - w[r, blk])
            assert np.all(err <= scale * 1.0 + 1e-12)
    rel = np.linalg.norm(dec - w) / np.linalg.norm(w)
    assert rel < 0.12
    assert np.all(s < 0x7F)  # no NaN scale code


def test_tiny_case_shapes(synth_mod):
    draft, verify, W_full = synth_mod.tiny_case()
    assert W_full.shape == (4096, 256)
    assert draft.W.shape == (1024, 256) and draft.cand_ids.shape == (1024,)
    np.testing.assert_array_equal(draft.W, W_full[draft.cand_ids])
    assert len(draft.hidden) == 3 and draft.hidden[0].shape == (1, 256)
    assert verify.X.shape == (4, 256) and verify.B == 1 and verify.k == 3
