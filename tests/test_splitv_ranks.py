"""Split-V draft head on fake CPU ranks (gloo): every rank scores its shard of
the candidate table (with the oracle, so no GPU is needed), the ranks
all-gather (score, id) and merge; the merged result must equal the
single-table argmax, including ties that straddle ranks.  CPU only."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from verify_head_gb300.splitv import merge_rank_argmax, shard_rows, split_v_draft_argmax


def test_merge_rule():
    ml = torch.tensor([[1.0, 2.0, 5.0, float("nan")], [3.0, 2.0, 5.0, -1.0], [0.5, 2.0, 4.0, -2.0]])
    ids = torch.tensor([[10, 7, 9, 1], [11, 3, 8, 2], [12, 5, 1, 3]], dtype=torch.int32)
    win, best = merge_rank_argmax(ml, ids)
    assert win.tolist() == [11, 3, 8, 2]  # max; tie -> lowest id; NaN loses
    assert best.tolist() == [3.0, 2.0, 5.0, -1.0]
    # -0 and +0 tie -> lowest id
    win, _ = merge_rank_argmax(torch.tensor([[-0.0], [0.0]]), torch.tensor([[9], [4]], dtype=torch.int32))
    assert win.tolist() == [4]


def test_shard_rows_cover():
    for n, w in [(65_536, 2), (1000, 3), (7, 8)]:
        spans = [shard_rows(n, r, w) for r in range(w)]
        assert spans[0][0] == 0 and spans[-1][1] == n
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))


@pytest.mark.parametrize("world", [2, 3, 4, 5, 8])
def test_merge_of_shard_argmaxes_equals_global(world):
    """The oracle's head split into `world` contiguous shards: merging the
    per-shard (max, global id) pairs gives the single-table argmax, including
    an exact tie planted across every shard boundary."""
    import oracle
    import synth
    oracle.build()
    synth.build()
    draft, _, _ = synth.tiny_case()
    W, cand = draft.W.copy(), draft.cand_ids
    x = draft.hidden[0]
    xf = (x[0].astype(np.uint32) << 16).view(np.float32)
    win = np.where(xf > 0, 0x3F00, 0xBF00).astype(np.uint16)
    for r in range(1, world):  # same winning row at the first row of every shard but the first
        W[shard_rows(cand.size, r, world)[0]] = win
    W[shard_rows(cand.size, 1, world)[0] - 1] = win  # and at the last row of shard 0
    ml_r, ids_r = [], []
    for r in range(world):
        lo, hi = shard_rows(cand.size, r, world)
        ids, ml, _ = oracle.draft_argmax(x, W[lo:hi], cand[lo:hi], nthreads=1)
        ids_r.append(ids)
        ml_r.append(ml)
    win_ids, best = merge_rank_argmax(torch.from_numpy(np.stack(ml_r)), torch.from_numpy(np.stack(ids_r)))
    want_ids, want_ml, _ = oracle.draft_argmax(x, W, cand, nthreads=1)
    assert int(win_ids[0]) == int(want_ids[0]) == int(cand[shard_rows(cand.size, 1, world)[0] - 1])
    assert float(best[0]) == float(want_ml[0])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    import oracle
    import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        draft, _, W_full = synth.tiny_case()
        W, cand = draft.W.copy(), draft.cand_ids
        # plant a tie across the shard boundary: the last row of shard 0 and the
        # first row of shard 1 become the same clear winner; shard 0 holds the lower id
        lo1, _ = shard_rows(cand.size, 1, world)
        x = draft.hidden[0]
        xf = (x[0].astype(np.uint32) << 16).view(np.float32)
        win = np.where(xf > 0, 0x3F00, 0xBF00).astype(np.uint16)
        W[lo1 - 1] = win
        W[lo1] = win
        lo, hi = shard_rows(cand.size, rank, world)

        def local():
            ids, ml, _ = oracle.draft_argmax(x, W[lo:hi], cand[lo:hi], nthreads=1)
            return torch.from_numpy(ids), torch.from_numpy(ml)

        ids, ml = split_v_draft_argmax(local)
        want_ids, want_ml, _ = oracle.draft_argmax(x, W, cand, nthreads=1)
        np.save(os.path.join(out_dir, f"r{rank}.npy"),
                np.array([int(ids[0]), float(ml[0]), int(want_ids[0]), float(want_ml[0]), int(cand[lo1 - 1])]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_split_v_on_cpu_ranks(tmp_path, world):
    import oracle
    import synth
    oracle.build()
    synth.build()
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    res = [np.load(os.path.join(tmp_path, f"r{r}.npy")) for r in range(world)]
    for r in res:
        assert r[0] == r[2] and r[1] == r[3]  # merged == single-table argmax
        assert r[0] == r[4]                   # the tie across ranks went to the lower id
    assert all(np.array_equal(res[0], r) for r in res)


def _dead_rank_main(rank, world, port, out_dir):
    import datetime

    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        return  # this rank dies before the exchange: no all-gather, no clean shutdown
    outcome = "returned"
    try:
        split_v_draft_argmax(lambda: (torch.zeros(1, dtype=torch.int32), torch.zeros(1)))
    except Exception as e:  # the surviving rank must see an error, not hang
        outcome = "raised " + type(e).__name__
    with open(os.path.join(out_dir, "r0.txt"), "w") as f:
        f.write(outcome)


def test_split_v_dead_rank_raises(tmp_path):
    """A rank that exits before the exchange: the surviving rank's merge raises
    (peer closed or process-group timeout) instead of waiting forever."""
    import time
    port = _free_port()
    t0 = time.time()
    ctx = mp.start_processes(_dead_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=False,
                             start_method="spawn")
    while not ctx.join(timeout=60):
        assert time.time() - t0 < 120, "ranks did not finish"
    out = open(os.path.join(tmp_path, "r0.txt")).read()
    assert out.startswith("raised"), out
