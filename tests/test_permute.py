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
    nbytes = mx.moe_permute_workspace_size(mx.dims(128, 128, E, ids.shape[1]), ids.shape[0])
    assert nbytes >= 256
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
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


# one CTA plans up to 8192 entries; larger batches run in chunks of 2048 entries over many CTAs
@pytest.mark.parametrize("n,k,E", [(1, 8, 384), (1, 1, 1), (3, 5, 33), (37, 8, 384), (1000, 7, 1024),
                                   (777, 3, 64), (1024, 8, 16), (1025, 8, 16), (2049, 5, 1024), (4097, 8, 384)])
def test_permute_ragged_shapes(n, k, E):
    ids = syn.routing_uniform(n, E, k, torch.Generator().manual_seed(n * 31 + k))
    _check(ids, E)


@pytest.mark.parametrize("n", [5000, 20000])
def test_permute_all_tokens_one_expert(n):
    ids = torch.full((n, 1), 17, dtype=torch.int32)
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


def test_permute_errors_in_chunked_plan():
    # 3000 x 8 entries: the chunked path; bad ids in several chunks, one duplicate
    g = torch.Generator().manual_seed(11)
    ids = syn.routing_uniform(3000, 64, 8, g)
    ids[5, 2] = 64
    ids[1500, 0] = -3
    ids[2999, 7] = 1000
    _check(ids, 64)
    ids = syn.routing_uniform(3000, 64, 8, g)
    ids[2100, 3] = ids[2100, 4]
    *_, err = _run(ids, 64, validate=False)
    assert err == mx.MOE_OK
    *_, err = _run(ids, 64, validate=True)
    assert err == 4
    _check(ids, 64)
