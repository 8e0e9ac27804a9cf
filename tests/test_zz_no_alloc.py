"""moe_infer_static: the routed-expert forward on the library's built-in scratch.

Some callers cannot allocate device memory themselves (a plugin or embedded
runtime that only hands over input and output buffers, code running inside
another library's allocator hooks, paths where a cudaMalloc could synchronise
the device).  For them the library offers moe_infer_static, which needs no
workspace.  These tests call it through the C ABI on two calls in a row and
compare each result with moe_infer (caller-provided workspace): both run the
same deterministic kernels on the same inputs, so the outputs must be equal
bit for bit (leftover or partly overwritten scratch would show up here), and
both must lie within the parity tolerance of the oracle.  The file sorts last
so that a run stopping at its first failure has run every other test; it also
passes on its own.
"""

import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
import oracle
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu


def _static(c, x, ids, w):
    n, d = x.shape
    E, d_ff, _ = c.bank.w_gate.shape[0], c.bank.w_gate.shape[1], d
    dm = mx.dims(d, d_ff, E, ids.shape[1])
    out = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    mx.moe_infer_static(dm, n, x, ids, w, mx.weights(c.bank), out)
    return out


def _check_same(a, b):
    assert torch.equal(a, b)


def test_static_matches_workspace_entry_two_calls_tiny():
    c = cases.workload("tiny")
    # second call: another seeded batch of a different size
    x2 = torch.randn(77, c.x.shape[1], generator=torch.Generator().manual_seed(123)).to(torch.bfloat16).cuda()
    ids2 = syn.routing_uniform(77, c.inp.wl.num_experts, c.inp.wl.top_k, torch.Generator().manual_seed(124)).cuda()
    w2 = syn.router_weights(77, c.inp.wl.top_k, torch.Generator().manual_seed(125)).cuda()
    a1 = _static(c, c.x, c.ids, c.w)
    a2 = _static(c, x2, ids2, w2)
    torch.cuda.synchronize()
    _check_same(a1, mx.infer(c.x, c.ids, c.w, c.bank))
    _check_same(a2, mx.infer(x2, ids2, w2, c.bank))
    # and both against the oracle, under the parity tolerance
    ref1 = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank)
    ref2 = oracle.moe_infer(x2.cpu(), ids2.cpu(), w2.cpu(), c.inp.bank)
    for y, ref in ((a1, ref1), (a2, ref2)):
        rep = oracle.parity_report(y, ref, bf16_output=True)
        assert rep["ok"], rep


def test_static_matches_workspace_entry_two_calls_k2_decode():
    c = cases.workload("k2_decode")
    a1 = _static(c, c.x, c.ids, c.w)
    x2, ids2, w2 = c.x[:9].flip(0).contiguous(), c.ids[:9].contiguous(), c.w[:9].contiguous()
    a2 = _static(c, x2, ids2, w2)
    torch.cuda.synchronize()
    _check_same(a1, mx.infer(c.x, c.ids, c.w, c.bank))
    _check_same(a2, mx.infer(x2, ids2, w2, c.bank))


def test_static_k2_largest_batch_that_fits():
    # 24 tokens is the largest K2 batch whose workspace fits the built-in scratch
    dm = mx.dims(7168, 2048, 384, 8)
    assert mx.moe_workspace_size(dm, 24) <= mx.MOE_STATIC_SCRATCH_BYTES
    c = cases.workload("k2_decode", n_tokens=24)
    a = _static(c, c.x, c.ids, c.w)
    torch.cuda.synchronize()
    _check_same(a, mx.infer(c.x, c.ids, c.w, c.bank))


def test_static_rejects_problems_larger_than_its_scratch():
    dm = mx.dims(7168, 2048, 384, 8)
    assert mx.moe_workspace_size(dm, 25) > mx.MOE_STATIC_SCRATCH_BYTES
    t = torch.empty(1, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MoeError) as e:
        mx.moe_infer_static(dm, 25, t, t, t, mx.moe_weights(), t)
    assert e.value.status == 3   # MOE_ERR_WORKSPACE, nothing launched
