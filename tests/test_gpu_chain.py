"""The fused 3-step draft chain against the oracle.

An MTP3 round runs the draft head three times in a row (one fresh hidden
vector per step, "少读一张大表，草稿路径才真正快起来"; MTP, "Qwen3.8-Flash-Next" §2).
The library launches every draft kernel as a programmatic dependent launch, so
step i+1 starts its prologue while step i drains, and the whole chain can be
captured once as a CUDA graph and replayed (CUDA Graph, same page §3).  These
tests issue the three calls back to back with no host synchronisation between
them (sharing one workspace, as a decode loop does), and replay the captured
chain, and check every step's ids and max logits against the oracle.
"""
import numpy as np
import pytest

from parity_util import TOL_4BIT, TOL_BF16, check_ids, to_torch, to_torch_bf16

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


def run_chain(calls, outs, replays=0):
    """calls(): enqueue the chain.  Eager once; then, with replays > 0, capture
    it as a graph and replay it `replays` times.  Returns one list of host
    copies of `outs` per run (eager first)."""
    import torch
    runs = []
    for t in outs:
        t.fill_(-7)
    calls()
    torch.cuda.synchronize()
    runs.append([t.cpu().numpy().copy() for t in outs])
    if replays:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            calls()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for _ in range(replays):
            for t in outs:
                t.fill_(-7)
            g.replay()
            torch.cuda.synchronize()
            runs.append([t.cpu().numpy().copy() for t in outs])
    return runs


def test_chain_draft_65536x2048(vh, orc, syn):
    """The single-stream decode chain: 65,536 candidate rows x 2048, B = 1,
    three steps back to back, then the same chain as a graph replayed twice."""
    import torch
    case = syn.draft_case(Vc=65_536, H=2048, B=1, steps=3, seed=2)
    Wd, cd = to_torch_bf16(case.W), to_torch(case.cand_ids)
    xs = [to_torch_bf16(h) for h in case.hidden]
    ws = vh.workspace(1)
    ids = [torch.empty(1, dtype=torch.int32, device="cuda") for _ in range(3)]
    mls = [torch.empty(1, dtype=torch.float32, device="cuda") for _ in range(3)]

    def calls():
        for i in range(3):
            vh.mtp_draft_head_argmax(xs[i], Wd, cd, ids=ids[i], maxlogit=mls[i], ws=ws)

    runs = run_chain(calls, ids + mls, replays=2)
    want = [orc.draft_argmax(x, case.W, case.cand_ids) for x in case.hidden]

    def score_of_step(i):
        def f(r, gid):
            c = int(np.searchsorted(case.cand_ids, gid))
            assert case.cand_ids[c] == gid
            return orc.dot_bf16(case.hidden[i][r], case.W[c])
        return f

    for run in runs:
        for i in range(3):
            o_ids, o_ml, o_sec = want[i]
            check_ids(run[i], run[3 + i], o_ids, o_ml, o_sec, score_of_step(i), TOL_BF16)
    assert int(ws.count_nonzero()) == 0


def test_chain_gather_fixed_plus_dynamic(vh, orc, syn):
    """Dynamic candidate rows: 32,768 fixed + 16,384 per-step rows of the
    248,320 x 2048 head, a different row list per step, chained and replayed."""
    import torch
    W_full = syn.full_head(2, syn.V_FULL, 2048)
    Wd = to_torch_bf16(W_full)
    rows = [syn.gather_row_ids(6, syn.V_FULL, step=i) for i in range(3)]
    xh = [syn.normal_bf16(2, syn.STREAM_HIDDEN, (1, 2048), 1.0, offset=i * 2048) for i in range(3)]
    rd = [to_torch(r) for r in rows]
    xs = [to_torch_bf16(h) for h in xh]
    ws = vh.workspace(1)
    ids = [torch.empty(1, dtype=torch.int32, device="cuda") for _ in range(3)]
    mls = [torch.empty(1, dtype=torch.float32, device="cuda") for _ in range(3)]

    def calls():
        for i in range(3):
            vh.mtp_draft_head_argmax_gather(xs[i], Wd, rd[i], ids=ids[i], maxlogit=mls[i], ws=ws)

    runs = run_chain(calls, ids + mls, replays=1)
    for i in range(3):
        o_ids, o_ml, o_sec = orc.draft_argmax_gather(xh[i], W_full, rows[i])
        for run in runs:
            check_ids(run[i], run[3 + i], o_ids, o_ml, o_sec,
                      lambda r, gid, i=i: orc.dot_bf16(xh[i][r], W_full[gid]), TOL_BF16)


@pytest.mark.parametrize("B", [1, 8])
def test_chain_nvfp4_65536x4096(vh, orc, syn, B):
    """The 4-bit draft head (65,536 x 4096), three steps chained and replayed."""
    import torch
    case = syn.nvfp4_case(Vc=65_536, H=4096, B=B, steps=3, seed=5)
    qd, sd, cd = to_torch(case.q), to_torch(case.s), to_torch(case.cand_ids)
    xs = [to_torch_bf16(h) for h in case.hidden]
    ws = vh.workspace(B)
    ids = [torch.empty(B, dtype=torch.int32, device="cuda") for _ in range(3)]
    mls = [torch.empty(B, dtype=torch.float32, device="cuda") for _ in range(3)]

    def calls():
        for i in range(3):
            vh.mtp_draft_head_argmax_nvfp4(xs[i], qd, sd, case.g, cd, ids=ids[i], maxlogit=mls[i], ws=ws)

    runs = run_chain(calls, ids + mls, replays=1)
    for i in range(3):
        x = case.hidden[i]
        o_ids, o_ml, o_sec = orc.draft_argmax_nvfp4(x, case.q, case.s, case.g, case.cand_ids)

        def score_of(r, gid, x=x):
            c = int(np.searchsorted(case.cand_ids, gid))
            assert case.cand_ids[c] == gid
            return float(orc.scores_nvfp4(x[r], case.q[c:c + 1], case.s[c:c + 1], case.g, nthreads=1)[0])

        for run in runs:
            check_ids(run[i], run[3 + i], o_ids, o_ml, o_sec, score_of, TOL_4BIT)


def test_chain_draft_then_verify_round(vh, orc, syn):
    """One speculative round on one stream: three draft steps, then the
    verify of 16 sequences x 4 positions against the full head, chained and
    replayed; draft and verify results both against the oracle."""
    import torch
    from parity_util import check_accept
    V, H, B, k = 30_000, 512, 16, 3
    case = syn.draft_case(Vc=8192, H=H, B=1, steps=3, seed=12, V=V)
    Wf = syn.normal_bf16(13, 1, (V, H), 0.02)
    X = syn.normal_bf16(14, 4, (B * (k + 1), H), 1.0)
    _, o_nid, o_ml, o_sec = orc.verify_greedy(X, Wf, None, B, k)
    draft = syn.corrupt_ids(15, syn.STREAM_CORRUPT, o_nid.reshape(B, k + 1)[:, :k].copy(), V, 0.45)
    o_acc = np.array([orc.accept_len(o_nid[b * (k + 1): b * (k + 1) + k], draft[b]) for b in range(B)], np.int32)
    Wc, cc = to_torch_bf16(case.W), to_torch(case.cand_ids)
    xs = [to_torch_bf16(h) for h in case.hidden]
    Wfd, Xd, dd = to_torch_bf16(Wf), to_torch_bf16(X), to_torch(draft)
    ws_d, ws_v = vh.workspace(1), vh.workspace(B * (k + 1))
    ids = [torch.empty(1, dtype=torch.int32, device="cuda") for _ in range(3)]
    mls = [torch.empty(1, dtype=torch.float32, device="cuda") for _ in range(3)]
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nid = torch.empty(B * (k + 1), dtype=torch.int32, device="cuda")
    vml = torch.empty(B * (k + 1), dtype=torch.float32, device="cuda")

    def calls():
        for i in range(3):
            vh.mtp_draft_head_argmax(xs[i], Wc, cc, ids=ids[i], maxlogit=mls[i], ws=ws_d)
        vh.spec_verify_greedy(Xd, Wfd, dd, B, k, accept_len=acc, next_ids=nid, row_maxlogit=vml, ws=ws_v)

    runs = run_chain(calls, ids + mls + [acc, nid, vml], replays=2)
    want = [orc.draft_argmax(x, case.W, case.cand_ids) for x in case.hidden]
    for run in runs:
        for i in range(3):
            o_ids, d_ml, d_sec = want[i]
            check_ids(run[i], run[3 + i], o_ids, d_ml, d_sec,
                      lambda r, gid, i=i: orc.dot_bf16(case.hidden[i][r],
                                                       case.W[int(np.searchsorted(case.cand_ids, gid))]), TOL_BF16)
        check_ids(run[7], run[8], o_nid, o_ml, o_sec, lambda r, v: orc.dot_bf16(X[r], Wf[v]), TOL_BF16)
        check_accept(run[6], run[7], o_acc, o_ml, o_sec, draft, B, k)
