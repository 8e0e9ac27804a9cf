"""The CUDA path against the CPU oracle on the same seeded inputs.

Tolerance (stated for the routed-expert forward): per element
|y - y_ref| <= 1e-2 * rms(y_ref) (+ 2^-8 |y_ref|, half a bf16 ulp, for a bf16
output) and mean |y - y_ref| / mean |y_ref| <= 2e-3.  Small workloads are
compared element by element over the whole output (K2 decode too, which also
covers the 16-token down pass's split last round); the larger K2 workloads on
a seeded sample of at least 512 tokens that the oracle computes one by one, at
the full size and launch configuration: a token of every touched expert, the
tokens at both edge rows of every 128-row tile of the three most-loaded
experts, and uniform tokens (tests/gpu_cases.py, parity_tokens)."""

import numpy as np
import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
import oracle
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu


def _assert_ok(y, ref, bf16=True):
    rep = oracle.parity_report(y, ref, bf16)
    assert rep["ok"], rep
    return rep


# ------------------------------------------------------------------ small, whole output

def test_tiny_infer_bf16_and_fp32_outputs():
    c = cases.workload("tiny")
    ref = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank)
    y = mx.infer(c.x, c.ids, c.w, c.bank)
    _assert_ok(y, ref, bf16=True)
    y32 = mx.infer(c.x, c.ids, c.w, c.bank, out_is_fp32=True)
    _assert_ok(y32, ref, bf16=False)
    assert torch.equal(y32.to(torch.bfloat16), y)   # the bf16 output is the fp32 result rounded once


@pytest.mark.parametrize("n,d,dff,E,k,seed", [
    (37, 256, 384, 5, 3, 1),       # ragged token count, d_ff of three 128-blocks
    (1, 1024, 256, 16, 4, 2),      # one token
    (200, 512, 128, 64, 6, 3),     # many experts, most with few rows
    (300, 384, 256, 3, 1, 4),      # k = 1, a hundred rows per expert (several token tiles)
    (64, 128, 128, 1, 1, 5),       # single expert
    (600, 256, 256, 2, 1, 6),      # 300 rows per expert: tiles of 128, 128 and 44 rows
    (150, 1152, 256, 4, 2, 8),     # nine 128-row blocks of down: the last pair has one block
    (40, 256, 128, 64, 32, 12),    # the largest top-k (32): 1280 rows over 64 experts
    (24, 128, 256, 1024, 4, 13),   # the largest expert count (1024), almost every expert empty
    (200, 256, 128, 40, 32, 14),   # top-k 32 with 160 rows per expert: wide tiles
    (64, 1024, 256, 40, 8, 22),    # 176 down units on 152 SMs: 152 pairs, then 48 single row blocks
])
def test_small_shapes_infer(n, d, dff, E, k, seed):
    wl = syn.Workload("s", n, d, dff, E, k, seed=seed)
    c = cases.workload(wl)
    ref = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank)
    _assert_ok(mx.infer(c.x, c.ids, c.w, c.bank), ref)
    _assert_ok(mx.infer(c.x, c.ids, c.w, c.bank, out_is_fp32=True), ref, bf16=False)


def test_experts_forward_rows_and_combine_separately():
    c = cases.workload("tiny")
    n, k, d = c.inp.wl.n_tokens, c.inp.wl.top_k, c.inp.wl.d
    dm = mx.dims(d, c.inp.wl.d_ff, c.inp.wl.num_experts, k)
    ws = mx.workspace(dm, n)
    counts, offsets, sp, ip = mx.permute(c.ids, c.inp.wl.num_experts, ws=ws)
    rows = torch.empty(n, k, d, dtype=torch.float16, device="cuda")
    mx.moe_experts_forward(dm, n, c.x, c.w, offsets, sp, mx.weights(c.bank), rows, ws)
    # each row is topk_weight * expert(x) for its own (token, slot)
    for t, j in [(0, 0), (0, 3), (77, 1), (127, 2)]:
        e = int(c.inp.topk_ids[t, j])
        b = c.inp.bank
        o = oracle.expert_forward(c.inp.x[t:t + 1].double().numpy(), b.w_gate[e], b.s_gate[e], b.w_up[e],
                                  b.s_up[e], b.w_down[e], b.s_down[e])[0] * float(c.inp.topk_weight[t, j])
        got = rows[t, j].double().cpu().numpy()
        rms = np.sqrt(np.mean(o ** 2))
        assert np.max(np.abs(got - o) - 2.0 ** -10 * np.abs(o)) <= 1e-2 * rms
    out = torch.empty(n, d, dtype=torch.float32, device="cuda")
    mx.moe_combine(dm, n, rows, None, None, out, out_is_fp32=True)
    ref = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank)
    _assert_ok(out, ref, bf16=False)
    # combine is an ordered fp32 sum of the f16 rows
    assert torch.equal(out, rows.float().sum(dim=1)) or torch.allclose(out, rows.float().sum(dim=1), rtol=0,
                                                                        atol=1e-6)
    assert mx.moe_get_error(ws) == mx.MOE_OK


def test_combine_adds_shared_then_residual():
    n, k, d = 19, 3, 256
    g = torch.Generator().manual_seed(3)
    rows = torch.randn(n, k, d, generator=g).half().cuda()
    shared = torch.randn(n, d, generator=g).half().cuda()
    resid = torch.randn(n, d, generator=g).bfloat16().cuda()
    dm = mx.dims(d, 128, 4, k)
    out = torch.empty(n, d, dtype=torch.float32, device="cuda")
    mx.moe_combine(dm, n, rows, shared, resid, out, out_is_fp32=True)
    r = rows.double()
    ref = ((r[:, 0] + r[:, 1] + r[:, 2]) + shared.double()) + resid.double()
    assert torch.allclose(out.double(), ref, rtol=1e-6, atol=1e-6)
    outb = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    mx.moe_combine(dm, n, rows, shared, resid, outb)
    assert torch.equal(outb, out.to(torch.bfloat16))


def test_layer_forward_small_with_shared_expert():
    wl = syn.Workload("blk", 96, 512, 256, 12, 4, full_block=True, d_ff_shared=384, seed=7)
    c = cases.workload(wl)
    ref = oracle.layer_forward(c.inp.x, c.inp.gain, c.inp.eps, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank,
                               c.inp.shared)
    y = mx.layer_forward(c.x, c.gain, c.inp.eps, c.ids, c.w, c.bank, c.shared)
    _assert_ok(y, ref)
    y2 = mx.layer_forward(c.x, c.gain, c.inp.eps, c.ids, c.w, c.bank, None)
    ref2 = oracle.layer_forward(c.inp.x, c.inp.gain, c.inp.eps, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank)
    _assert_ok(y2, ref2)


def test_layer_forward_wide_tiles():
    # 200 routed rows per expert and 300 shared rows: tiles of 128 rows
    wl = syn.Workload("blkw", 300, 384, 256, 3, 2, full_block=True, d_ff_shared=256, seed=11)
    c = cases.workload(wl)
    ref = oracle.layer_forward(c.inp.x, c.inp.gain, c.inp.eps, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank,
                               c.inp.shared)
    _assert_ok(mx.layer_forward(c.x, c.gain, c.inp.eps, c.ids, c.w, c.bank, c.shared), ref)


def test_deterministic_and_zero_tokens():
    c = cases.workload("tiny")
    a = mx.infer(c.x, c.ids, c.w, c.bank)
    b = mx.infer(c.x, c.ids, c.w, c.bank)
    assert torch.equal(a, b)
    empty = mx.infer(c.x[:0], c.ids[:0], c.w[:0], c.bank)
    assert empty.shape == (0, c.x.shape[1])


def test_forced_empty_experts_and_hot_expert():
    wl = syn.Workload("s", 256, 512, 256, 64, 4, seed=9)
    g = torch.Generator().manual_seed(2)
    ids = syn.routing_subset(256, [3, 17, 40, 41, 63], 4, g)
    c = cases.workload(wl, ids=ids)
    c.ids = ids.cuda()
    ref = oracle.moe_infer(c.inp.x, ids, c.inp.topk_weight, c.inp.bank)
    _assert_ok(mx.infer(c.x, c.ids, c.w, c.bank), ref)


def test_wide_tiles_rows_wider_than_the_gather_holds():
    # d 8320 (65 K blocks): the f16 row gather keeps up to 8192 columns of a row in registers and
    # reads the rest a second time; wide tiles (64 rows over 2 experts), 130 f16 panels per row
    wl = syn.Workload("wide8320", 64, 8320, 128, 2, 1, seed=23)
    c = cases.workload(wl)
    ref = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.inp.bank)
    _assert_ok(mx.infer(c.x, c.ids, c.w, c.bank), ref)


def _tile_split_flag(counts, tile=128):
    """The stage-split rule of the wide f16 GEMM: 1 when at least 90 % of the tiles belong to
    experts cut into two or more tiles."""
    tiles = [(c + tile - 1) // tile for c in counts]
    multi = sum(t for t in tiles if t >= 2)
    return int(sum(tiles) > 0 and 10 * multi >= 9 * sum(tiles)), sum(tiles)


@pytest.mark.parametrize("counts", [
    [200, 200, 200, 200, 129, 50, 0, 0],   # 10 of 11 tiles in multi-tile experts: 2 + 5 stages
    [200, 200, 200, 200, 50, 50, 0, 0],    # 8 of 10: 3 + 4
    [100] * 8,                             # one tile per expert
    [1300, 20, 0, 0, 0, 0, 0, 0],          # a hot expert: 11 of 12
])
def test_wide_stage_split_flag_and_parity(counts):
    # Wide tiles (128 rows, d 1024: 8 K blocks per gate/up unit, so either ring wraps) with a
    # chosen number of tiles per expert.  The routing kernel writes the tile count and the
    # weight-sharing flag to the workspace words at bytes 64 and 72; both stage splits must
    # give the oracle's output.
    E, n = 8, sum(counts)
    wl = syn.Workload("split", n, 1024, 256, E, 1, seed=21)
    g = torch.Generator().manual_seed(5)
    ids = torch.cat([torch.full((c,), e, dtype=torch.int32) for e, c in enumerate(counts)])
    ids = ids[torch.randperm(n, generator=g)].reshape(n, 1).contiguous()
    c = cases.workload(wl, ids=ids)
    c.ids = ids.cuda()
    ws = mx.workspace(mx.dims(1024, 256, E, 1), n)
    y = mx.infer(c.x, c.ids, c.w, c.bank, ws=ws)
    words = ws[64:80].view(torch.int32).cpu().tolist()
    flag, n_tiles = _tile_split_flag(counts)
    assert words[0] == n_tiles and words[2] == flag, (words, n_tiles, flag)
    _assert_ok(y, oracle.moe_infer(c.inp.x, ids, c.inp.topk_weight, c.inp.bank))


# ------------------------------------------------------------------ K2 sizes

def test_k2_decode_whole_output():
    c = cases.workload("k2_decode")
    y = mx.infer(c.x, c.ids, c.w, c.bank)
    ref = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.bank)
    _assert_ok(y, ref)
    y32 = mx.infer(c.x, c.ids, c.w, c.bank, out_is_fp32=True)
    _assert_ok(y32, ref, bf16=False)


@pytest.mark.parametrize("name", ["k2_prefill", "k2_skewed"])
def test_k2_large_sampled_tokens(name):
    # at the full size and launch configuration (wide tiles, chunked unit order): at least 512 tokens,
    # covering every touched expert and both edge rows of every tile of the three most-loaded experts
    c = cases.workload(name)
    y = mx.infer(c.x, c.ids, c.w, c.bank)
    tok = cases.parity_tokens(c.inp.topk_ids, n_min=512, seed=1)
    assert len(tok) >= 512
    ref = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.bank, tokens=tok)
    _assert_ok(y[tok], ref)
    assert torch.isfinite(y.float()).all()


def test_k2_twice_the_block_batch_sampled_tokens():
    # 65,536 tokens (R = 524,288 routed rows): element offsets into the sorted rows and the expert
    # outputs pass 2^31, so any 32-bit index arithmetic on the wide-tile path would show here
    wl = syn.Workload("k2_65536", 65536, 7168, 2048, 384, 8, seed=4, bank_seed=1)
    c = cases.workload(wl)
    y = mx.infer(c.x, c.ids, c.w, c.bank)
    tok = cases.parity_tokens(c.inp.topk_ids, n_min=512, seed=3)
    assert len(tok) >= 512 and tok[-1] == wl.n_tokens - 1
    ref = oracle.moe_infer(c.inp.x, c.inp.topk_ids, c.inp.topk_weight, c.bank, tokens=tok)
    _assert_ok(y[tok], ref)
    assert torch.isfinite(y.float()).all()


def test_k2_block_sampled_tokens():
    c = cases.workload("k2_block")
    y = mx.layer_forward(c.x, c.gain, c.inp.eps, c.ids, c.w, c.bank, c.shared)
    tok = cases.parity_tokens(c.inp.topk_ids, n_min=512, seed=2)
    assert len(tok) >= 512
    ref = oracle.layer_forward(c.inp.x, c.inp.gain, c.inp.eps, c.inp.topk_ids, c.inp.topk_weight, c.bank,
                               c.shared, tokens=tok)
    _assert_ok(y[tok], ref)
    assert torch.isfinite(y.float()).all()


def _hot_expert_rows(c, act=mx.MOE_ACT_EXACT):
    """moe_permute + moe_experts_forward on the tiled bank; returns (rows f16 [n, k, d] on the GPU,
    the hottest expert, its (token, slot) entries at the first and last valid row of every 128-row tile)."""
    n, k = c.ids.shape
    E, d_ff, d = 384, 2048, 7168
    dm = mx.dims(d, d_ff, E, k, act)
    ws = mx.workspace(dm, n)
    counts, offsets, sp, ip = mx.permute(c.ids, E, ws=ws)
    bank_t = mx.pack_bank(c.bank)
    torch.cuda.synchronize()
    rows = torch.empty(n, k, d, dtype=torch.float16, device="cuda")
    mx.moe_experts_forward(dm, n, c.x, c.w, offsets, sp, mx.weights(bank_t), rows, ws)
    torch.cuda.synchronize()
    assert mx.moe_get_error(ws) == mx.MOE_OK
    del bank_t
    counts, offsets, sp = counts.cpu(), offsets.cpu(), sp.cpu()
    hot = int(counts.argmax())
    lo, cnt = int(offsets[hot]), int(counts[hot])
    picks = sorted({i for t0 in range(0, cnt, 128) for i in (t0, min(t0 + 127, cnt - 1))})
    entries = [(int(sp[lo + i]) // k, int(sp[lo + i]) % k) for i in picks]
    return rows, hot, entries


def test_k2_skewed_hot_expert_every_tile():
    # the skewed workload's hottest expert spans about sixty 128-row tiles of one expert (wide kernel,
    # several tiles per expert, a ragged last tile): its first and last row of every tile against the oracle
    c = cases.workload("k2_skewed")
    rows, hot, entries = _hot_expert_rows(c)
    assert len(entries) >= 100
    b = c.bank
    W = [t[hot].cpu() for t in (b.w_gate, b.s_gate, b.w_up, b.s_up, b.w_down, b.s_down)]
    xt = torch.stack([c.inp.x[t] for t, _ in entries]).double().numpy()
    o = oracle.expert_forward(xt, *W)
    for i, (t, j) in enumerate(entries):
        ref = o[i] * float(c.inp.topk_weight[t, j])
        got = rows[t, j].double().cpu().numpy()
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.max(np.abs(got - ref) - 2.0 ** -10 * np.abs(ref)) <= 1e-2 * rms, (t, j)
