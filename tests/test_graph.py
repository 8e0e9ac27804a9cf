"""The calls are asynchronous on the caller's stream with no host synchronisation,
so a whole forward can be captured in a CUDA graph and replayed: the replay must
give the eager result bit for bit, for both tile widths and the fused layer."""

import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "k2_decode", syn.Workload("g16", 40, 512, 256, 32, 4, seed=21)])
def test_infer_graph_replay_matches_eager(name):
    c = cases.workload(name)
    n, d = c.x.shape
    k = c.ids.shape[1]
    E, d_ff, _ = mx.bank_sizes(c.bank)
    dm = mx.dims(d, d_ff, E, k)
    bank = mx.pack_bank(c.bank)
    W = mx.weights(bank)
    ws = mx.workspace(dm, n)
    x, ids, w = c.x.clone(), c.ids.clone(), c.w.clone()
    out = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()   # packing and copies ran on the default stream; the calls below use their own
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mx.moe_infer(dm, n, x, ids, w, W, out, ws, stream=s)   # first call outside the capture
    s.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mx.moe_infer(dm, n, x, ids, w, W, out, ws, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    # new inputs in the same buffers: the graph reads them
    x.copy_(torch.flip(c.x, dims=[0]))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, mx.infer(x, ids, w, c.bank))
    assert mx.moe_get_error(ws) == mx.MOE_OK


def test_layer_graph_replay_matches_eager():
    wl = syn.Workload("blkg", 300, 384, 256, 3, 2, full_block=True, d_ff_shared=256, seed=11)
    c = cases.workload(wl)
    n, d = c.x.shape
    dm = mx.dims(d, 256, 3, 2)
    ws = mx.workspace(dm, n, 256)
    out = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    W, WS = mx.weights(c.bank), mx.weights(c.shared)
    with torch.cuda.stream(s):
        mx.moe_layer_forward(dm, n, c.x, c.gain, c.inp.eps, c.ids, c.w, W, WS, 256, out, ws, stream=s)
    s.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mx.moe_layer_forward(dm, n, c.x, c.gain, c.inp.eps, c.ids, c.w, W, WS, 256, out, ws, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


@pytest.mark.parametrize("act", [mx.MOE_ACT_EXACT, mx.MOE_ACT_FP8_DYNAMIC])
def test_mlp_and_fp8_infer_graph_replay_matches_eager(act):
    # the dense MLP entry point (wide tiles) and moe_infer in either activation scheme, in one graph
    c = cases.workload(syn.Workload("gf", 200, 512, 256, 8, 2, seed=23))
    n, d = c.x.shape
    dm = mx.dims(d, 256, 8, 2, act)
    dm1 = mx.dims(d, 256, 1, 1, act)
    mlp_bank = syn.ExpertBank(*(t[:1].contiguous() for t in (c.bank.w_gate, c.bank.w_up, c.bank.w_down,
                                                              c.bank.s_gate, c.bank.s_up, c.bank.s_down)))
    ws, ws1 = mx.workspace(dm, n), mx.workspace(dm1, n)
    W, W1 = mx.weights(c.bank), mx.weights(mlp_bank)
    out = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    out1 = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()

    def body():
        mx.moe_infer(dm, n, c.x, c.ids, c.w, W, out, ws, stream=s)
        mx.moe_mlp_forward(dm1, n, c.x, W1, out1, ws1, stream=s)

    with torch.cuda.stream(s):
        body()
    s.synchronize()
    eager, eager1 = out.clone(), out1.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        body()
    out.zero_()
    out1.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager) and torch.equal(out1, eager1)
    assert mx.moe_get_error(ws) == mx.MOE_OK and mx.moe_get_error(ws1) == mx.MOE_OK


@pytest.mark.parametrize("act", [mx.MOE_ACT_EXACT, mx.MOE_ACT_FP8_DYNAMIC])
def test_weights_written_just_before_the_call_are_the_ones_used(act):
    # Every kernel of a call is a dependent launch of the one before, and the GEMMs stream weights
    # without waiting; a bank overwritten in place by the kernel right before the call must still be
    # read only after that kernel has finished (decode-sized: 16-token tiles; and wide tiles).
    for wl in (syn.Workload("pd16", 16, 512, 256, 32, 4, seed=31), syn.Workload("pdw", 200, 512, 256, 8, 2, seed=32)):
        c = cases.workload(wl)
        other = cases.bank_to(syn.expert_bank(wl.num_experts, wl.d, wl.d_ff, 77), "cuda")
        ref = mx.infer(c.x, c.ids, c.w, other, act_scheme=act)
        tiled, tiled_other = mx.pack_bank(c.bank), mx.pack_bank(other)
        torch.cuda.synchronize()
        mx.infer(c.x, c.ids, c.w, tiled, act_scheme=act)            # the bank as it was
        tiled.w_gate.copy_(tiled_other.w_gate)                       # then overwritten in place ...
        tiled.w_down.copy_(tiled_other.w_down)
        for nm in ("s_gate", "s_up", "s_down"):
            getattr(tiled, nm).copy_(getattr(tiled_other, nm))
        y = mx.infer(c.x, c.ids, c.w, tiled, act_scheme=act)         # ... and used at once
        assert torch.equal(y, ref)
        # the dense MLP entry point and the fused layer's path start with other kernels
        one = syn.ExpertBank(*(t[:1].contiguous() for t in (c.bank.w_gate, c.bank.w_up, c.bank.w_down,
                                                            c.bank.s_gate, c.bank.s_up, c.bank.s_down)))
        one_other = syn.ExpertBank(*(t[:1].contiguous() for t in (other.w_gate, other.w_up, other.w_down,
                                                                  other.s_gate, other.s_up, other.s_down)))
        ref1 = mx.mlp_forward(c.x, one_other, act_scheme=act)
        mx.mlp_forward(c.x, one, act_scheme=act)
        for nm in ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down"):
            getattr(one, nm).copy_(getattr(one_other, nm))
        assert torch.equal(mx.mlp_forward(c.x, one, act_scheme=act), ref1)
