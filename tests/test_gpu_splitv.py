"""Split-V draft head with the CUDA kernel on every rank.

"少读一张大表，草稿路径才真正快起来" splits the 65,536-row candidate head over two
ranks (32,768 rows each): each rank takes the argmax over its rows, then the
ranks exchange the best score and the global token id.  Here two processes
share cuda:0; each runs mtp_draft_head_argmax on its shard, and the (id, max)
pairs are all-gathered over gloo (host copies, 8 bytes per hidden row per
rank) and merged with the kernel's rule.  The merged result must equal the
oracle over the whole table, including an exact tie planted across the shard
boundary.  The kernels of the two ranks never wait on each other: the only
exchange is on the host, after each rank's kernel has finished.
"""
import os
import socket

import numpy as np
import pytest

from parity_util import TOL_BF16, check_ids

pytestmark = pytest.mark.gpu

VC, H, B = 65_536, 2048, 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _case():
    """The 65,536 x 2048 candidate head; hidden row 0 meets a clear winner
    planted at the last row of shard 0 and the first row of shard 1."""
    import synth
    case = synth.draft_case(Vc=VC, H=H, B=B, steps=1, seed=2)
    W = case.W.copy()
    x = case.hidden[0]
    xf = (x[0].astype(np.uint32) << 16).view(np.float32)
    win = np.where(xf > 0, 0x3F00, 0xBF00).astype(np.uint16)  # +-0.5 against +-~1: far above N(0,0.02) rows
    W[VC // 2 - 1] = win
    W[VC // 2] = win
    return x, W, case.cand_ids


def _shard(rank, world, split):
    if split == "contiguous":
        lo, hi = VC * rank // world, VC * (rank + 1) // world
        return np.arange(lo, hi)
    return np.arange(rank, VC, world)  # interleaved: a rank's rows are not one range of ids


def _rank_main(rank, world, port, out_dir, split):
    import datetime

    import torch
    import torch.distributed as dist

    import verify_head_gb300 as vh
    from verify_head_gb300.splitv import split_v_draft_argmax
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    # a rank that fails makes the other one raise within a minute instead of waiting forever
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        torch.cuda.set_device(0)
        x, W, cand = _case()
        rows = _shard(rank, world, split)
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        Wd = torch.from_numpy(np.ascontiguousarray(W[rows]).view(np.int16)).cuda().view(torch.bfloat16)
        cd = torch.from_numpy(np.ascontiguousarray(cand[rows])).cuda()

        def local():
            ids, ml = vh.mtp_draft_head_argmax(xd, Wd, cd)
            return ids.cpu(), ml.cpu()  # gloo exchanges host tensors

        ids, ml = split_v_draft_argmax(local)
        np.savez(os.path.join(out_dir, f"r{rank}.npz"), ids=ids.numpy(), ml=ml.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("split", ["contiguous", "interleaved"])
def test_split_v_two_ranks_on_gpu(tmp_path, split):
    import torch
    import torch.multiprocessing as mp
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    import synth
    import verify_head_gb300 as vh
    oracle.build()
    synth.build()
    vh.build()
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), split), nprocs=world, join=True,
                       start_method="spawn")
    res = [np.load(os.path.join(tmp_path, f"r{r}.npz")) for r in range(world)]
    for r in res[1:]:  # every rank holds the same merged answer
        np.testing.assert_array_equal(r["ids"], res[0]["ids"])
        np.testing.assert_array_equal(r["ml"], res[0]["ml"])
    x, W, cand = _case()
    o_ids, o_ml, o_sec = oracle.draft_argmax(x, W, cand)
    assert int(o_ids[0]) == int(cand[VC // 2 - 1])  # the tie goes to the lower global id
    assert int(res[0]["ids"][0]) == int(cand[VC // 2 - 1])

    def score_of(r, gid):
        c = int(np.searchsorted(cand, gid))
        assert cand[c] == gid
        return oracle.dot_bf16(x[r], W[c])

    check_ids(res[0]["ids"], res[0]["ml"], o_ids, o_ml, o_sec, score_of, TOL_BF16)
