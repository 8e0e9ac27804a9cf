"""Dynamic FP8 activations: the CUDA path against the oracle's same scheme.

"Input features" page, quantisation config: fmt e4m3, activation_scheme
"dynamic", weight blocks of 128 x 128.  Under MOE_ACT_FP8_DYNAMIC every row
entering a linear (x or the normalised row, and h) is quantised per group of
128 features: scale s = amax / 448 in fp32, code = nearest e4m3 of v / s.

Both sides take the x codes from the same bf16 bytes with the same fp32
arithmetic, so they agree exactly there; h differs between the two only by
fp32 accumulation order, which moves an h code by one e4m3 step in rare
boundary cases.  The comparison uses the same tolerance as the exact scheme
(per element |y - y_ref| <= 1e-2 rms(y_ref) + half a bf16 ulp, mean relative
error <= 2e-3) against the oracle run with fp8_act=True.

The scheme itself is an approximation of the exact function: on the tiny
workload the oracle's FP8 result differs from its exact one by a mean relative
error of about 4.3e-2.  That distance is the scheme's stated accuracy, checked
here to stay below 6e-2."""

import numpy as np
import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
import oracle
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu

FP8 = mx.MOE_ACT_FP8_DYNAMIC
SCHEME_MEAN_REL = 6e-2   # FP8 scheme vs the exact function (the oracle's own distance is ~4.3e-2)


def _assert_ok(y, ref, bf16=True):
    rep = oracle.parity_report(y, ref, bf16)
    assert rep["ok"], rep
    return rep


def _infer_ref(c, tokens=None, bank=None):
    return oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, bank if bank is not None else c.inp.bank,
                            tokens=tokens, fp8_act=True)


def test_fp8_wide_tiles_rows_of_8320_features():
    # 65 K blocks through the dynamic FP8 gather and the FP8 wide-tile kernel
    wl = syn.Workload("wide8320", 64, 8320, 128, 2, 1, seed=23)
    c = cases.workload(wl)
    _assert_ok(mx.infer(c.x, c.ids, c.w, c.bank, act_scheme=FP8), _infer_ref(c))


def test_tiny_fp8_matches_oracle_and_scheme_accuracy():
    c = cases.workload("tiny")   # 32 rows per expert: wide tiles
    ref = _infer_ref(c)
    y = mx.infer(c.x, c.ids, c.w, c.bank, act_scheme=FP8)
    _assert_ok(y, ref)
    y32 = mx.infer(c.x, c.ids, c.w, c.bank, out_is_fp32=True, act_scheme=FP8)
    _assert_ok(y32, ref, bf16=False)
    # the scheme changes the result by about an e4m3 step against the exact function
    exact = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank)
    err = np.abs(y32.double().cpu().numpy() - exact)
    rel = err.mean() / np.abs(exact).mean()
    assert 1e-2 < rel < SCHEME_MEAN_REL
    # and the exact scheme on the same inputs is unaffected by the option
    _assert_ok(mx.infer(c.x, c.ids, c.w, c.bank), exact)


@pytest.mark.parametrize("n,d,dff,E,k,seed", [
    (37, 256, 384, 5, 3, 1),       # 22 rows per expert: 16-token tiles, ragged
    (1, 1024, 256, 16, 4, 2),      # one token
    (300, 384, 256, 3, 1, 4),      # a hundred rows per expert: wide tiles
    (600, 256, 256, 2, 1, 6),      # tiles of 128, 128 and 44 rows
    (150, 1152, 256, 4, 2, 8),     # nine row blocks of down: the last pair has one block
    (40, 256, 128, 64, 32, 12),    # top-k 32 over 64 experts
    (64, 1024, 256, 40, 8, 22),    # 176 down units on 152 SMs: 152 pairs, then 48 single row blocks
])
def test_small_shapes_fp8(n, d, dff, E, k, seed):
    wl = syn.Workload("s", n, d, dff, E, k, seed=seed)
    c = cases.workload(wl)
    ref = _infer_ref(c)
    _assert_ok(mx.infer(c.x, c.ids, c.w, c.bank, act_scheme=FP8), ref)
    _assert_ok(mx.infer(c.x, c.ids, c.w, c.bank, out_is_fp32=True, act_scheme=FP8), ref, bf16=False)


def test_fp8_all_zero_rows_and_deterministic():
    wl = syn.Workload("z", 64, 256, 256, 4, 2, seed=3)
    c = cases.workload(wl)
    x = c.x.clone()
    x[5] = 0          # an all-zero token: every group takes scale 1 and codes 0
    x[9, :128] = 0    # one all-zero group
    xh = x.cpu()
    ref = oracle.moe_infer(xh, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank, fp8_act=True)
    a = mx.infer(x, c.ids, c.w, c.bank, act_scheme=FP8)
    b = mx.infer(x, c.ids, c.w, c.bank, act_scheme=FP8)
    assert torch.equal(a, b)
    assert not a[5].any()
    _assert_ok(a, ref)


def test_layer_forward_fp8_small_and_wide_with_shared_expert():
    for wl in (syn.Workload("blk", 96, 512, 256, 12, 4, full_block=True, d_ff_shared=384, seed=7),
               syn.Workload("blkw", 300, 384, 256, 3, 2, full_block=True, d_ff_shared=256, seed=11)):
        c = cases.workload(wl)
        ref = oracle.layer_forward(c.inp.x, c.inp.gain, c.inp.eps, c.inp.topk_ids, c.inp.topk_weight,
                                   c.inp.bank, c.inp.shared, fp8_act=True)
        _assert_ok(mx.layer_forward(c.x, c.gain, c.inp.eps, c.ids, c.w, c.bank, c.shared, act_scheme=FP8), ref)


def test_k2_decode_fp8_whole_output():
    c = cases.workload("k2_decode")   # 16-token tiles
    y = mx.infer(c.x, c.ids, c.w, c.bank, act_scheme=FP8)
    _assert_ok(y, _infer_ref(c, bank=c.bank))


@pytest.mark.parametrize("name", ["k2_prefill", "k2_skewed"])
def test_k2_large_fp8_sampled_tokens(name):
    c = cases.workload(name)          # wide tiles; skewed routing spans many tiles of its hot experts
    y = mx.infer(c.x, c.ids, c.w, c.bank, act_scheme=FP8)
    tok = cases.parity_tokens(c.inp.topk_ids, n_min=512, seed=1)
    assert len(tok) >= 512
    _assert_ok(y[tok], _infer_ref(c, tokens=tok, bank=c.bank))
    assert torch.isfinite(y.float()).all()


def test_k2_twice_the_block_batch_fp8_sampled_tokens():
    # 65,536 tokens (R = 524,288 routed rows) through the dynamic FP8 gather and wide-tile kernel
    wl = syn.Workload("k2_65536", 65536, 7168, 2048, 384, 8, seed=4, bank_seed=1)
    c = cases.workload(wl)
    y = mx.infer(c.x, c.ids, c.w, c.bank, act_scheme=FP8)
    tok = cases.parity_tokens(c.inp.topk_ids, n_min=512, seed=3)
    assert len(tok) >= 512 and tok[-1] == wl.n_tokens - 1
    _assert_ok(y[tok], _infer_ref(c, tokens=tok, bank=c.bank))
    assert torch.isfinite(y.float()).all()


def test_k2_block_fp8_sampled_tokens():
    c = cases.workload("k2_block")
    y = mx.layer_forward(c.x, c.gain, c.inp.eps, c.ids, c.w, c.bank, c.shared, act_scheme=FP8)
    tok = cases.parity_tokens(c.inp.topk_ids, n_min=512, seed=2)
    assert len(tok) >= 512
    ref = oracle.layer_forward(c.inp.x, c.inp.gain, c.inp.eps, c.inp.topk_ids, c.inp.topk_weight, c.bank,
                               c.shared, tokens=tok, fp8_act=True)
    _assert_ok(y[tok], ref)
    assert torch.isfinite(y.float()).all()


def test_k2_skewed_hot_expert_every_tile_fp8():
    from tests.test_parity import _hot_expert_rows
    c = cases.workload("k2_skewed")
    rows, hot, entries = _hot_expert_rows(c, FP8)
    b = c.bank
    W = [t[hot].cpu() for t in (b.w_gate, b.s_gate, b.w_up, b.s_up, b.w_down, b.s_down)]
    xt = torch.stack([c.inp.x[t] for t, _ in entries]).double().numpy()
    o = oracle.expert_forward(xt, *W, fp8_act=True)
    for i, (t, j) in enumerate(entries):
        ref = o[i] * float(c.inp.topk_weight[t, j])
        got = rows[t, j].double().cpu().numpy()
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.max(np.abs(got - ref) - 2.0 ** -10 * np.abs(ref)) <= 1e-2 * rms, (t, j)
