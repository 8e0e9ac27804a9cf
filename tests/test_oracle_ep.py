"""Pins of the expert-parallel oracle (oracle/ep.py) - CPU only.

"Mixture of experts" page, moe_infer, ep_size > 1 branch; "Input features"
page, expert construction (rank r holds experts r E/ep .. (r + 1) E/ep - 1).

* A worked example small enough to follow by hand: every split, the
  source-major counts each rank receives, the regroup order and the counts
  per local expert are written out below from the routing alone.
* The multi-rank forward equals the single-rank routed sum bit for bit (the
  exchanges only move rows; every row meets the same expert arithmetic and
  each token sums its slots in the same order), for 1, 2 and 4 ranks.
* Moving any exchange piece to the wrong rank, or dropping the regroup,
  breaks that equality (checked on planted copies of the plan).
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import ep as oep
from mixture_experts_ffn_infer_gb300 import synthetic as syn


def test_plan_worked_example():
    # E = 4 experts on 2 ranks (rank 0: experts 0, 1; rank 1: experts 2, 3), k = 2
    ids0 = np.array([[0, 3], [2, 1], [3, 2]], np.int32)   # flat 0 3 2 1 3 2
    ids1 = np.array([[1, 2], [0, 1], [2, 3]], np.int32)   # flat 1 2 0 1 2 3
    p0, p1 = oep.ep_plan([ids0, ids1], 4, 2)
    # rank 0: one entry for expert 0, one for 1, two each for 2 and 3
    assert p0["tokens_per_expert"].tolist() == [1, 1, 2, 2]
    assert p0["idxs"].tolist() == [0, 3, 2, 5, 1, 4]        # expert order, ties by flat index
    assert p0["input_split_sizes"].tolist() == [2, 4]       # 2 rows to rank 0, 4 to rank 1
    assert p1["tokens_per_expert"].tolist() == [1, 2, 2, 1]
    assert p1["idxs"].tolist() == [2, 0, 3, 1, 4, 5]
    assert p1["input_split_sizes"].tolist() == [3, 3]
    # rank 0 receives counts of experts 0, 1 from rank 0 (1, 1) then from rank 1 (1, 2)
    assert p0["tokens_per_expert_group"].tolist() == [1, 1, 1, 2]
    assert p0["output_splits"].tolist() == [2, 3]
    # received rows labelled by local expert: 0 | 1 | 0 | 1 1  ->  expert 0 rows first
    assert p0["gatherd_idxs"].tolist() == [0, 2, 1, 3, 4]
    assert p0["tokens_per_expert_post_gather"].tolist() == [2, 3]
    # rank 1: experts 2, 3 from rank 0 (2, 2) and from rank 1 (2, 1)
    assert p1["tokens_per_expert_group"].tolist() == [2, 2, 2, 1]
    assert p1["output_splits"].tolist() == [4, 3]
    # labels 0 0 | 1 1 | 0 0 | 1
    assert p1["gatherd_idxs"].tolist() == [0, 1, 4, 5, 2, 3, 6]
    assert p1["tokens_per_expert_post_gather"].tolist() == [4, 3]


def _ranks(ep, n_per_rank=9, d=256, dff=128, E=8, k=2, seed=5):
    wl = syn.Workload("ep", n_per_rank, d, dff, E, k, seed=seed)
    bank = syn.expert_bank(E, d, dff, seed, "cpu")
    xs, ids, ws = [], [], []
    for r in range(ep):
        x, i, w, _ = syn.make_host_inputs(syn.Workload(**{**wl.__dict__, "seed": seed + 100 * r}))
        xs.append(x)
        ids.append(i)
        ws.append(w)
    return xs, ids, ws, bank


@pytest.mark.parametrize("ep", [1, 2, 4])
def test_ep_forward_equals_single_rank_bit_for_bit(ep):
    xs, ids, ws, bank = _ranks(ep)
    ys = oep.moe_infer_ep(xs, ids, ws, bank, ep)
    for r in range(ep):
        ref = oracle.moe_infer(xs[r], ids[r], ws[r], bank)
        assert np.array_equal(ys[r], ref), r


def test_plan_invariants_skewed_routing():
    ep, E, k = 4, 16, 4
    g = torch.Generator().manual_seed(3)
    ids = [syn.routing_zipf(40, E, k, 1.2, g) for _ in range(ep)]
    plans = oep.ep_plan(ids, E, ep)
    epr = E // ep
    for r, p in enumerate(plans):
        assert p["input_split_sizes"].sum() == ids[r].numel()                       # every entry is sent once
        assert sorted(p["idxs"].tolist()) == list(range(ids[r].numel()))            # a permutation
        assert p["gatherd_idxs"].size == p["output_splits"].sum()
        assert sorted(p["gatherd_idxs"].tolist()) == list(range(p["gatherd_idxs"].size))
        # what r receives from s is what s sends to r
        for s in range(ep):
            assert p["output_splits"][s] == plans[s]["input_split_sizes"][r]
        # the regroup orders received rows by local expert, ties by received position
        group = p["tokens_per_expert_group"]
        labels = np.repeat(np.arange(group.size) % epr, group)
        lab = labels[p["gatherd_idxs"]]
        assert np.all(np.diff(lab) >= 0)
        for e in range(epr):
            pos = p["gatherd_idxs"][lab == e]
            assert np.all(np.diff(pos) > 0)
        assert p["tokens_per_expert_post_gather"].sum() == group.sum()


def test_planted_exchange_mistakes_are_caught():
    ep = 2
    xs, ids, ws, bank = _ranks(ep, seed=9)
    good = oep.moe_infer_ep(xs, ids, ws, bank, ep)
    real_plan = oep.ep_plan

    def plan_swapped_sources(ids_, E_, ep_):
        plans = real_plan(ids_, E_, ep_)
        for p in plans:  # receive the pieces in the wrong source order
            p["output_splits"] = p["output_splits"][::-1].copy()
        return plans

    def plan_no_regroup(ids_, E_, ep_):
        plans = real_plan(ids_, E_, ep_)
        for p in plans:
            p["gatherd_idxs"] = np.arange(p["gatherd_idxs"].size)
        return plans

    for bad in (plan_swapped_sources, plan_no_regroup):
        oep.ep_plan = bad
        try:
            try:
                ys = oep.moe_infer_ep(xs, ids, ws, bank, ep)
            except (ValueError, IndexError):
                continue  # a shape mismatch is also a caught mistake
            assert any(not np.array_equal(y, g) for y, g in zip(ys, good)), bad.__name__
        finally:
            oep.ep_plan = real_plan
