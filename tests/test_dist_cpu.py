"""Host-side logic of bench.py's multi-rank run, on two gloo ranks on the CPU.

Each rank runs the layer on its own tokens with identical weights; the timed region is the
max over ranks.  No GPU is used.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from mixture_experts_layer_pft_gb300 import workloads

        ws, r, lr = bench.dist_env()
        assert (ws, r, lr) == (world, rank, rank)
        bench.barrier(world)
        m = bench.max_over_ranks(10.0 + rank, world, device="cpu")
        w = workloads.WORKLOADS[0]
        inp = workloads.make_inputs(w, "cpu", T=8, token_seed=w.seed + 7919 * rank)
        gathered_x = [torch.empty_like(inp["x"]) for _ in range(world)]
        gathered_w = [torch.empty_like(inp["W1"]) for _ in range(world)]
        dist.all_gather(gathered_x, inp["x"])
        dist.all_gather(gathered_w, inp["W1"])
        out[rank] = (m, not torch.equal(gathered_x[0], gathered_x[1]),
                     torch.equal(gathered_w[0], gathered_w[1]))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_max_timing_and_token_sharding():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    for r in range(world):
        m, x_differs, w_same = out[r]
        assert m == 11.0  # the max over ranks
        assert x_differs and w_same
