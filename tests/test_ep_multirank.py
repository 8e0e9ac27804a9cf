"""The expert-parallel forward across real ranks: two gloo processes on the CPU.

mixture_experts_ffn_infer_gb300/ep.py runs as on GPUs (the count exchange,
the row exchange and the reverse exchange through torch.distributed
all_to_all_single), with the oracle's local steps (tests/ep_cpu_ops.py) in
place of the device kernels.  Each rank's result must equal the single-rank
oracle on the whole expert bank bit for bit, with the pages' exact split
sizes and with fixed-capacity splits, under uniform and skewed routing."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out_dir, capacity, routing):
    import oracle
    from mixture_experts_ffn_infer_gb300 import ep as mep
    from mixture_experts_ffn_infer_gb300 import synthetic as syn
    from tests.ep_cpu_ops import OracleOps

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        d, dff, E, k, n = 256, 128, 8, 3, 11
        bank = syn.expert_bank(E, d, dff, 21, "cpu")          # the same bank on every rank
        wl = syn.Workload("ep", n, d, dff, E, k, routing=routing, seed=40 + rank)
        x, ids, w, _ = syn.make_host_inputs(wl)
        local = mep.shard_bank(bank, rank, WORLD)
        cap = n * k if capacity else 0
        y = mep.moe_infer_ep(x, ids, w, local, E, capacity=cap, ops=OracleOps(d, E, k))
        ref = oracle.moe_infer(x, ids, w, bank)
        np.save(os.path.join(out_dir, f"y{rank}.npy"), y.numpy())
        np.save(os.path.join(out_dir, f"ref{rank}.npy"), ref)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("capacity,routing", [(False, "uniform"), (True, "uniform"), (False, "zipf"),
                                              (True, "zipf")])
def test_ep_two_gloo_ranks_equal_single_rank(tmp_path, capacity, routing):
    mp.start_processes(_worker, args=(_free_port(), str(tmp_path), capacity, routing), nprocs=WORLD, join=True,
                       start_method="spawn")
    for r in range(WORLD):
        y = np.load(tmp_path / f"y{r}.npy")
        ref = np.load(tmp_path / f"ref{r}.npy")
        assert np.array_equal(y, ref), r
