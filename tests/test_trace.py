"""moe_trace: the per-kernel events a call records, in both modes, and the
count of kernels it launched (what bench.py reports as gpu_launches)."""

import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu


def _trace(gemms_only):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    t = mx.moe_trace()
    s = torch.cuda.current_stream()
    for i, e in enumerate(evs):
        e.record(s)
        t.events[i] = e.cuda_event
    t.n_events = len(evs)
    t.gemms_only = gemms_only
    return t, evs


@pytest.mark.parametrize("name,routing_kernels", [("tiny", 1), ("k2_prefill", 3)])
def test_trace_events_and_launch_count(name, routing_kernels):
    c = cases.workload(name)
    n, d = c.x.shape
    k = c.ids.shape[1]
    E, d_ff, _ = mx.bank_sizes(c.bank)
    dm = mx.dims(d, d_ff, E, k)
    ws = mx.workspace(dm, n)
    out = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    ref = mx.infer(c.x, c.ids, c.w, c.bank)
    for gemms_only in (0, 1):
        t, evs = _trace(gemms_only)
        mx.moe_infer(dm, n, c.x, c.ids, c.w, mx.weights(c.bank), out, ws, trace=t)
        torch.cuda.synchronize()
        labels = [t.labels[i].decode() for i in range(t.n_recorded - 1)]
        if gemms_only:
            assert labels == ["gateup_swiglu", "down_scatter"]
        else:
            assert labels == ["route_permute", "gather_rows", "gateup_swiglu", "down_scatter", "combine"]
        assert t.n_launched == routing_kernels + 4
        times = [evs[i].elapsed_time(evs[i + 1]) for i in range(t.n_recorded - 1)]
        assert all(x >= 0 for x in times)
        assert torch.equal(out, ref)   # tracing changes nothing in the result
