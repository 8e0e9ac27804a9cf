"""Error behaviour of the C ABI on the GPU, without faulting it: device-detected
routing errors, f16 overflow, a pipeline wait that runs out, and host-side
argument errors.  After every error the context stays usable."""

import numpy as np
import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
import oracle
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu

MOE_ERR_WORKSPACE, MOE_ERR_ROUTING, MOE_ERR_TIMEOUT, MOE_ERR_RANGE = 3, 4, 5, 6


def _tiny_call(c, ids, x=None):
    n, d = c.x.shape
    dm = mx.dims(d, c.inp.wl.d_ff, c.inp.wl.num_experts, ids.shape[1])
    ws = mx.workspace(dm, n)
    out = torch.empty(n, d, dtype=torch.float32, device="cuda")
    mx.moe_infer(dm, n, c.x if x is None else x, ids, c.w, mx.weights(c.bank), out, ws, out_is_fp32=True)
    return out, ws


def test_out_of_range_ids_are_reported_and_skipped():
    c = cases.workload("tiny")
    ids = c.inp.topk_ids.clone()
    ids[3, 1] = 16          # E = 16: out of range
    ids[40, 0] = -5
    out, ws = _tiny_call(c, ids.cuda())
    assert mx.moe_get_error(ws) == MOE_ERR_ROUTING
    assert mx.moe_get_error(ws) == mx.MOE_OK          # reading clears the word
    good = [t for t in range(c.x.shape[0]) if t not in (3, 40)]
    ref = oracle.moe_infer(c.inp.x, ids, c.inp.topk_weight, c.inp.bank, tokens=good)
    rep = oracle.parity_report(out[good], ref, bf16_output=False)
    assert rep["ok"], rep
    # a clean call afterwards reports nothing
    out2, ws2 = _tiny_call(c, c.ids)
    assert mx.moe_get_error(ws2) == mx.MOE_OK


def test_f16_overflow_is_reported():
    c = cases.workload("tiny")
    big = (c.inp.x.float() * 3000.0).to(torch.bfloat16).cuda()
    out, ws = _tiny_call(c, c.ids, x=big)
    assert mx.moe_get_error(ws) == MOE_ERR_RANGE


def test_pipeline_wait_that_runs_out_returns_timeout_and_gpu_stays_usable():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    mx.moe_check_bounded_wait(ws)
    assert mx.moe_get_error(ws) == MOE_ERR_TIMEOUT
    c = cases.workload("tiny")
    y = mx.infer(c.x, c.ids, c.w, c.bank)
    ref = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank)
    assert oracle.parity_report(y, ref)["ok"]


def test_host_side_errors():
    c = cases.workload("tiny")
    n, d = c.x.shape
    dm = mx.dims(d, c.inp.wl.d_ff, c.inp.wl.num_experts, c.inp.wl.top_k)
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    out = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.MoeError) as e:
        mx.moe_infer(dm, n, c.x, c.ids, c.w, mx.weights(c.bank), out, small)
    assert e.value.status == MOE_ERR_WORKSPACE
    with pytest.raises(mx.MoeError) as e:
        mx.moe_infer(mx.dims(1000, 256, 16, 4), n, c.x, c.ids, c.w, mx.weights(c.bank), out, small)
    assert e.value.status == 2
