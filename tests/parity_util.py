"""Comparison rules between the CUDA path and the oracle.

Ids: bit-exact wherever the oracle's top-1 / top-2 score gap exceeds 1e-2;
inside that band any id whose ORACLE score is within 1e-2 of the oracle
maximum is accepted (several answers are correct there).
Max logit: within 2e-2 absolute for bf16 heads, 5e-2 for the 4-bit head.
Accept lengths: equal to the oracle's when every row up to the first mismatch
has a clear gap; always equal to the scan recomputed from the GPU's own
next_ids (self-consistency).
"""
import numpy as np

GAP = 1e-2
TOL_BF16 = 2e-2
TOL_4BIT = 5e-2


def to_torch_bf16(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def to_torch(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def check_ids(gpu_ids, gpu_ml, o_ids, o_ml, o_sec, score_of, tol):
    """score_of(row, id) -> oracle score of that id for that row."""
    gpu_ids = np.asarray(gpu_ids)
    gpu_ml = np.asarray(gpu_ml, dtype=np.float64)
    n_exact = 0
    for r in range(len(o_ids)):
        gap = float(o_ml[r]) - float(o_sec[r])
        if gap > GAP:
            assert gpu_ids[r] == o_ids[r], f"row {r}: id {gpu_ids[r]} != oracle {o_ids[r]} (gap {gap:.3g})"
            n_exact += 1
        else:
            s = score_of(r, int(gpu_ids[r]))
            assert s >= float(o_ml[r]) - GAP, f"row {r}: near-tie id {gpu_ids[r]} scores {s} < {o_ml[r]} - {GAP}"
        assert abs(gpu_ml[r] - float(o_ml[r])) <= tol, f"row {r}: maxlogit {gpu_ml[r]} vs oracle {o_ml[r]}"
    return n_exact


def accept_scan(next_ids, draft, B, k):
    nid = np.asarray(next_ids).reshape(B, k + 1)
    d = np.asarray(draft).reshape(B, k)
    out = np.zeros(B, np.int32)
    for b in range(B):
        a = 0
        while a < k and nid[b, a] == d[b, a]:
            a += 1
        out[b] = a
    return out


def check_accept(gpu_acc, gpu_nid, o_acc, o_ml, o_sec, draft, B, k):
    gpu_acc = np.asarray(gpu_acc)
    # self-consistency: the fused scan agrees with the GPU's own next_ids
    np.testing.assert_array_equal(gpu_acc, accept_scan(gpu_nid, draft, B, k))
    assert np.all((gpu_acc >= 0) & (gpu_acc <= k))
    # exactness where every row up to the first mismatching one is clear
    for b in range(B):
        rows = range(b * (k + 1), b * (k + 1) + min(int(o_acc[b]), k - 1) + 1)
        if all(float(o_ml[r]) - float(o_sec[r]) > GAP for r in rows):
            assert gpu_acc[b] == o_acc[b], f"seq {b}: accept {gpu_acc[b]} != oracle {o_acc[b]}"
