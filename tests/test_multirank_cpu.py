"""Multi-rank host logic on CPU (gloo, world size 2): request sharding, per-rank oracle
work on its shard, and the max-over-ranks timing / summed-token reduction that the
benchmark uses under torchrun."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from diffusion_speculative_verify_gb300.sharding import shard_requests


def test_shard_requests_covers_every_request_once_and_balances():
    rng = np.random.default_rng(0)
    plen = rng.integers(128, 8193, 256)
    for ws in (1, 2, 3, 8):
        shards = shard_requests(plen, ws)
        flat = sorted(r for s in shards for r in s)
        assert flat == list(range(256))
        loads = [sum(int(plen[r]) + 1 for r in s) for s in shards]
        assert max(loads) - min(loads) <= int(plen.max()) + 1   # LPT bound
    assert shard_requests([5, -1, 0], 2) in ([[0], [1, 2]], [[1, 2], [0]])
    with pytest.raises(ValueError):
        shard_requests([1], 0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import workloads
        w = workloads.WORKLOADS["tiny_fp32"].with_(batch=6, V=64)
        lay = workloads.make_layout_inputs(w, seed=3)
        shards = shard_requests(lay["prompt_len"].tolist(), world)
        mine = shards[rank]
        acc = workloads.make_accept_inputs(w, seed=3)
        _, labels, err = oracle.build_layout(lay["tau"].numpy(), lay["prompt_len"].numpy())
        res = oracle.accept(acc["target_logits"].numpy(), acc["draft_logits"].numpy(),
                            acc["draft_tokens"].numpy(), labels, w.gamma, 1.0,
                            acc["philox_seed"], 0, requests=mine)
        committed = torch.tensor([int(sum(res["n_commit"][r] for r in mine))], dtype=torch.int64)
        elapsed = torch.tensor([0.5 + rank], dtype=torch.float64)   # stand-in per-rank time
        dist.all_reduce(committed, op=dist.ReduceOp.SUM)
        dist.all_reduce(elapsed, op=dist.ReduceOp.MAX)
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        if rank == 0:
            out.put((int(committed.item()), float(elapsed.item()), gathered))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_shards_reduce_like_the_benchmark():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    committed, elapsed, gathered = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert elapsed == 1.5                       # max over ranks
    assert sorted(gathered[0] + gathered[1]) == list(range(6))
    # the same total as one process computing every request
    import oracle
    import workloads
    w = workloads.WORKLOADS["tiny_fp32"].with_(batch=6, V=64)
    lay = workloads.make_layout_inputs(w, seed=3)
    acc = workloads.make_accept_inputs(w, seed=3)
    _, labels, _ = oracle.build_layout(lay["tau"].numpy(), lay["prompt_len"].numpy())
    res = oracle.accept(acc["target_logits"].numpy(), acc["draft_logits"].numpy(),
                        acc["draft_tokens"].numpy(), labels, w.gamma, 1.0, acc["philox_seed"], 0)
    assert committed == int(res["n_commit"].sum())
