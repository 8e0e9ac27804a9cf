"""The routing plan on the GPU (moe_permute) against the oracle's counting sort:
counts, offsets, sorted_pos and inv_pos must be identical, bit for bit."""

import numpy as np
import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
import oracle
from mixture_experts_ffn_infer_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _run(ids_host, E, validate=False):
    ids = ids_host.cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    counts, offsets, sp, ip = mx.permute(ids, E, ws=ws, validate=validate)
    err = mx.moe_get_error(ws)
    return counts.cpu().numpy(), offsets.cpu().numpy(), sp.cpu().numpy(), ip.cpu().numpy(), err


def _check(ids_host, E):
    c, o, sp, ip, err = _run(ids_host, E)
    rc, ro, rsp, rip, bad = oracle.permute(ids_host, E)
    assert np.array_equal(c, rc)
    assert np.array_equal(o, ro)
    assert np.array_equal(sp, rsp)
    assert np.array_equal(ip, rip)
    assert err == (mx.MOE_OK if bad == 0 else 4)


@pytest.mark.parametrize("name", list(syn.WORKLOADS))
def test_permute_workloads_bit_exact(name):
    wl = syn.WORKLOADS[name]
    _, ids, _, _ = syn.make_host_inputs(wl)
    _check(ids, wl.num_experts)


@pytest.mark.parametrize("n,k,E", [(1, 8, 384), (1, 1, 1), (3, 5, 33), (37, 8, 384), (1000, 7, 1024),
                                   (777, 3, 64), (4097, 8, 384)])
def test_permute_ragged_shapes(n, k, E):
    ids = syn.routing_uniform(n, E, k, torch.Generator().manual_seed(n * 31 + k))
    _check(ids, E)


def test_permute_all_tokens_one_expert():
    ids = torch.full((5000, 1), 17, dtype=torch.int32)
    _check(ids, 384)


def test_permute_forced_empty_experts():
    g = torch.Generator().manual_seed(5)
    subset = torch.randperm(384, generator=g)[:16].tolist()
    ids = syn.routing_subset(2048, subset, 8, g)
    c, *_ = _run(ids, 384)
    assert (c == 0).sum() == 384 - 16
    _check(ids, 384)


def test_permute_out_of_range_ids_flagged_and_skipped():
    ids = torch.tensor([[3, 1], [1, 7], [-1, 3], [9, 1], [2, 2]], dtype=torch.int32)
    _check(ids, 8)


def test_permute_duplicates_flagged_only_when_validating():
    ids = torch.tensor([[3, 1], [5, 5], [0, 2]], dtype=torch.int32)
    *_, err = _run(ids, 8, validate=False)
    assert err == mx.MOE_OK
    *_, err = _run(ids, 8, validate=True)
    assert err == 4
    _check(ids, 8)   # histogram semantics: a duplicated id counts twice, as in the oracle
