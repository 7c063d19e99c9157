"""SmallEP algebra across two processes on the CPU (gloo), with the oracle
as each rank's compute: the CPU-GPU hybrid inference article's SmallEP
section splits the routed experts over expert-parallel ranks; each rank
combines its own experts (rank 0 also the shared expert) and the partial
outputs are reduced.  Rank p here evaluates its partial with the oracle
(gate weights of other ranks' slots set to zero, fp64 sums), the partials are
all-gathered over gloo and added in rank order, and the result must equal
the single-process fp64 layer.  The expert partition is the one
moe_forward_smallep uses (smallep_groups)."""
import os

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth


def _partition(E, P):
    from moe_expert_ffn_02_gb300 import smallep_groups
    return smallep_groups(E, P)


def test_partition_covers_each_expert_once():
    for E in (1, 7, 8, 256, 384):
        for P in (1, 2, 3, 5, min(E, 16), E):
            if P > E:
                continue
            g = _partition(E, P)
            assert g[0][0] == 0 and g[-1][1] == E
            assert all(g[i][1] == g[i + 1][0] for i in range(P - 1))
            sizes = [hi - lo for lo, hi in g]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1


def _rank_partial(rank, P, inp, k, ids, w):
    lo, hi = _partition(inp["w_gate"].shape[0], P)[rank]
    mine = (ids >= lo) & (ids < hi)
    _, y = oracle.forward(inp, k, ids, np.where(mine, w, 0.0).astype(np.float32), want_f64=True)
    if rank != 0:                      # the shared expert belongs to rank 0 only
        _, y_sh = oracle.forward(inp, k, ids, np.zeros_like(w), want_f64=True)
        y = y - y_sh
    return y


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    wl = synth.Workload("gloo", 24, 256, 256, 8, 3, n_shared=1)
    inp = synth.make_inputs(wl, seed=3)
    L = oracle.logits(inp["x"], inp["router_w"], inp["router_b"])
    r = oracle.route_from_logits(L, wl.top_k)
    ids, w = r["ids"], r["w"]
    part = torch.from_numpy(_rank_partial(rank, world, inp, wl.top_k, ids, w))
    parts = [torch.empty_like(part) for _ in range(world)]
    dist.all_gather(parts, part)
    y = parts[0].clone()
    for p in range(1, world):          # fixed rank order
        y += parts[p]
    if rank == 0:
        _, ref = oracle.forward(inp, wl.top_k, ids, w, want_f64=True)
        q.put(float(np.max(np.abs(y.numpy() - ref)) / max(np.max(np.abs(ref)), 1e-300)))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_rank_partials_reduce_to_the_layer(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29000 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    err = q.get(timeout=10)
    assert err < 1e-12, err
