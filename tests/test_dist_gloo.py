"""The multi-rank path on CPU (gloo, world size 2): the timing reduction the benchmark uses
takes the slowest rank, and splitting a batch by tokens across ranks gives the same layer
output as the whole batch (tokens are independent units, so the path shards without any
exchange)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from oracle import moe_oracle as o
    from routing_dispatch_grouped_gb300 import synth

    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method=f"tcp://127.0.0.1:{port}")
    try:
        slow = bench.reduce_max(10.0 + 5.0 * rank, "cpu")
        cfg = synth.CONFIGS["tiny_fp32"]
        inp = synth.make_inputs(cfg)
        a, b = bench.shard_tokens(cfg.T, rank, world)
        wgu = inp["w_gate_up"].double().numpy()
        wd = inp["w_down"].double().numpy()
        part = o.forward(inp["x"][a:b].double().numpy(), inp["logits"][a:b].numpy(), wgu, wd,
                         cfg.k, round_h=False)["out"]
        parts = [None] * world
        dist.all_gather_object(parts, part)
        if rank == 0:
            whole = o.forward(inp["x"].double().numpy(), inp["logits"].numpy(), wgu, wd, cfg.k,
                              round_h=False)["out"]
            results.put((slow, float(np.max(np.abs(np.concatenate(parts) - whole)))))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_max_and_token_sharding():
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    slow, diff = results.get(timeout=10)
    assert slow == 15.0
    assert diff == 0.0


@pytest.mark.parametrize("T,world", [(256, 2), (255, 2), (7, 4), (0, 2)])
def test_shard_tokens_covers_batch(T, world):
    import bench
    got = [bench.shard_tokens(T, r, world) for r in range(world)]
    assert got[0][0] == 0 and got[-1][1] == T
    assert all(got[i][1] == got[i + 1][0] for i in range(world - 1))
