"""moe_mlp_forward: one SwiGLU MLP on every row, against the oracle's expert.

"SwiGLU output" page, MLP class: down(silu(gate x) * up x), the module every
expert is built from and the dense feed-forward blocks use too.  The library
runs it as a single expert segment holding all rows in order; the oracle's
single-expert forward (fp64, pinned in test_oracle_pins.py) is the reference,
under the same tolerance as the routed path."""

import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
import oracle
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu


def _mlp_case(n, d, dff, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g).to(torch.bfloat16)
    bank = syn.expert_bank(1, d, dff, seed)
    return x, bank


def _ref(x, bank, rows=None, fp8=False):
    xs = x if rows is None else x[rows]
    b = bank
    return oracle.expert_forward(xs.double().numpy(), b.w_gate[0], b.s_gate[0], b.w_up[0], b.s_up[0],
                                 b.w_down[0], b.s_down[0], fp8_act=fp8)


def _ok(y, ref, bf16=True):
    rep = oracle.parity_report(y, ref, bf16)
    assert rep["ok"], rep


@pytest.mark.parametrize("n,d,dff,seed", [
    (5, 256, 384, 1),       # 16-token tiles, ragged
    (1, 1024, 256, 2),      # one row
    (300, 384, 512, 3),     # wide tiles of 128, 128 and 44 rows
    (64, 1152, 256, 4),     # nine down row blocks: the last pair has one
])
def test_mlp_matches_oracle(n, d, dff, seed):
    x, bank = _mlp_case(n, d, dff, seed)
    ref = _ref(x, bank)
    gb = cases.bank_to(bank, "cuda")
    xd = x.cuda()
    _ok(mx.mlp_forward(xd, gb), ref)
    _ok(mx.mlp_forward(xd, gb, out_is_fp32=True), ref, bf16=False)
    # the tiled bank gives the same bytes
    assert torch.equal(mx.mlp_forward(xd, mx.pack_bank(gb)), mx.mlp_forward(xd, gb))


@pytest.mark.parametrize("n,d,dff,seed", [(7, 512, 256, 5), (200, 256, 384, 6)])
def test_mlp_fp8_matches_oracle_scheme(n, d, dff, seed):
    x, bank = _mlp_case(n, d, dff, seed)
    y = mx.mlp_forward(x.cuda(), cases.bank_to(bank, "cuda"), act_scheme=mx.MOE_ACT_FP8_DYNAMIC)
    _ok(y, _ref(x, bank, fp8=True))


def test_mlp_equals_moe_infer_with_one_expert():
    # the same rows through moe_infer with E = 1, k = 1 and router weight 1 give the same bytes
    x, bank = _mlp_case(96, 512, 256, 7)
    gb = cases.bank_to(bank, "cuda")
    xd = x.cuda()
    ids = torch.zeros(96, 1, dtype=torch.int32, device="cuda")
    w = torch.ones(96, 1, device="cuda")
    assert torch.equal(mx.mlp_forward(xd, gb), mx.infer(xd, ids, w, gb))


def test_mlp_large_width_sampled_rows():
    # a dense-block-sized MLP (d 7168, width 4096) on 512 rows, compared on a row sample
    x, bank = _mlp_case(512, 7168, 4096, 8)
    gb = cases.bank_to(bank, "cuda")
    y = mx.mlp_forward(x.cuda(), mx.pack_bank(gb))
    rows = [0, 1, 127, 128, 300, 511]
    _ok(y[rows], _ref(x, bank, rows))
    assert torch.isfinite(y.float()).all()
