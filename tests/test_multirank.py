"""The multi-GPU path of the benchmark is data-parallel over tokens ("replicas":
each rank its own batch, the same experts, no exchange on the data path).
Its host logic - per-rank workloads, the max-over-ranks time and the job
throughput - runs here on two gloo ranks on the CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from mixture_experts_ffn_infer_gb300 import synthetic as syn


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = bench.rank_workload(syn.WORKLOADS["tiny"], rank)
        x, ids, w, _ = syn.make_host_inputs(wl)
        fingerprint = float(x.float().sum()) + float(ids.sum())
        # ranks report different times; every rank must see the slowest
        t_max = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        gathered = [None] * world
        dist.all_gather_object(gathered, (fingerprint, syn.bank_seed_of(wl), t_max))
        if rank == 0:
            out.put(gathered)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (f0, b0, t0), (f1, b1, t1) = res
    assert f0 != f1                       # each rank draws its own batch
    assert b0 == b1                       # ... over the same expert bank
    assert t0 == t1 == 15.0               # max over ranks
    assert bench.job_tokens_per_s(16, world, 10, t0) == pytest.approx(16 * 2 * 10 / 0.015)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    wl = syn.WORKLOADS["k2_decode"]
    assert bench.rank_workload(wl, 0).seed == wl.seed
    assert bench.rank_workload(wl, 3).bank_seed == syn.bank_seed_of(wl)
