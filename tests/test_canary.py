"""Out-of-bounds writes, without a sanitizer: every buffer a call writes sits
inside a larger allocation whose surrounding bytes hold a fixed pattern, and the
pattern must be intact after the call.  Covers the workspace and the outputs of
moe_permute, moe_experts_forward, moe_combine, moe_infer, moe_layer_forward and
moe_mlp_forward, on both tile widths and both activation schemes, including a
ragged batch whose last tile is partial and a 16-token batch whose down units
are single row blocks."""

import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu

PAD = 4096          # guard bytes on each side
PATTERN = 0xA5


class Guarded:
    """A device buffer of `nbytes` (256-byte aligned) with PAD pattern bytes on each side."""

    def __init__(self, nbytes):
        self.nbytes = nbytes
        self.raw = torch.full((PAD + nbytes + PAD,), PATTERN, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        n = 1
        for s in shape:
            n *= s
        return self.raw[PAD:PAD + n * torch.empty(0, dtype=dtype).element_size()].view(dtype).view(*shape)

    def bytes(self):
        return self.raw[PAD:PAD + self.nbytes]

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.raw[:PAD] == PATTERN).all()) and bool((self.raw[PAD + self.nbytes:] == PATTERN).all())


def _ws(dm, n, dff_sh=0):
    g = Guarded(mx.moe_workspace_size(dm, n, dff_sh))
    g.bytes().zero_()
    return g


@pytest.mark.parametrize("wl", [syn.Workload("c16", 37, 384, 256, 5, 3, seed=41),     # 16-token tiles, ragged
                                syn.Workload("c16s", 37, 512, 256, 5, 3, seed=44),    # down units cut into single blocks
                                syn.Workload("cw", 300, 256, 384, 3, 2, seed=42)])    # wide tiles, partial last tile
@pytest.mark.parametrize("act", [mx.MOE_ACT_EXACT, mx.MOE_ACT_FP8_DYNAMIC])
def test_routed_calls_write_only_their_buffers(wl, act):
    c = cases.workload(wl)
    n, d, k, E, dff = wl.n_tokens, wl.d, wl.top_k, wl.num_experts, wl.d_ff
    dm = mx.dims(d, dff, E, k, act)
    bank_t = mx.pack_bank(c.bank)   # kept alive: the moe_weights struct holds raw device pointers
    W = mx.weights(bank_t)
    torch.cuda.synchronize()
    # moe_infer
    ws = _ws(dm, n)
    out = Guarded(n * d * 2)
    mx.moe_infer(dm, n, c.x, c.ids, c.w, W, out.view(torch.bfloat16, (n, d)), ws.bytes())
    assert out.intact() and ws.intact()
    assert mx.moe_get_error(ws.bytes()) == mx.MOE_OK
    # moe_permute + moe_experts_forward + moe_combine
    ws2 = _ws(dm, n)
    counts, offsets = Guarded(E * 4), Guarded((E + 1) * 4)
    sp, ip = Guarded(n * k * 4), Guarded(n * k * 4)
    mx.moe_permute(dm, n, c.ids, counts.view(torch.int32, (E,)), offsets.view(torch.int32, (E + 1,)),
                   sp.view(torch.int32, (n * k,)), ip.view(torch.int32, (n * k,)), ws2.bytes())
    rows = Guarded(n * k * d * 2)
    mx.moe_experts_forward(dm, n, c.x, c.w, offsets.view(torch.int32, (E + 1,)), sp.view(torch.int32, (n * k,)), W,
                           rows.view(torch.float16, (n, k, d)), ws2.bytes())
    out2 = Guarded(n * d * 4)
    mx.moe_combine(dm, n, rows.view(torch.float16, (n, k, d)), None, None, out2.view(torch.float32, (n, d)),
                   out_is_fp32=True)
    for g in (counts, offsets, sp, ip, rows, out2, ws2):
        assert g.intact()
    # the pieces give the one-call result
    assert torch.equal(out2.view(torch.float32, (n, d)).to(torch.bfloat16), out.view(torch.bfloat16, (n, d)))


@pytest.mark.parametrize("act", [mx.MOE_ACT_EXACT, mx.MOE_ACT_FP8_DYNAMIC])
def test_layer_and_mlp_write_only_their_buffers(act):
    wl = syn.Workload("cl", 96, 512, 256, 12, 4, full_block=True, d_ff_shared=384, seed=43)
    c = cases.workload(wl)
    n, d = wl.n_tokens, wl.d
    dm = mx.dims(d, wl.d_ff, wl.num_experts, wl.top_k, act)
    ws = _ws(dm, n, 384)
    out = Guarded(n * d * 2)
    mx.moe_layer_forward(dm, n, c.x, c.gain, c.inp.eps, c.ids, c.w, mx.weights(c.bank), mx.weights(c.shared), 384,
                         out.view(torch.bfloat16, (n, d)), ws.bytes())
    assert out.intact() and ws.intact()
    dm1 = mx.dims(d, 384, 1, 1, act)
    ws1 = _ws(dm1, n)
    out1 = Guarded(n * d * 4)
    mx.moe_mlp_forward(dm1, n, c.x, mx.weights(c.shared), out1.view(torch.float32, (n, d)), ws1.bytes(),
                       out_is_fp32=True)
    assert out1.intact() and ws1.intact()
    assert mx.moe_get_error(ws.bytes()) == mx.MOE_OK and mx.moe_get_error(ws1.bytes()) == mx.MOE_OK
