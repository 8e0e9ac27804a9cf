"""Pins of the CPU oracle against things other than itself.

Each test ties one part of the oracle to a value printed on the Kimi K2 pages,
to a closed form, to an invariant, or to a library routine that computes the
same step exactly (``torch.float8_e4m3fn`` decoding, ``torch.bincount``,
``torch.argsort(stable=True)``, fp64 ``torch.matmul``, ``F.silu``).  They are
chosen so that a plausible slip anywhere in the oracle (a dropped term, a
transposed operand, a wrong scale index, an unstable sort, a lost router
weight) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from mixture_experts_ffn_infer_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _deq_torch(q, s):
    """Library dequantisation: torch's e4m3 decode times the block scale, in fp64."""
    v = q.view(torch.float8_e4m3fn).to(torch.float64)
    return v * s.to(torch.float64).repeat_interleave(128, 0).repeat_interleave(128, 1)


def _small_bank(E, d, dff, seed):
    return syn.expert_bank(E, d, dff, seed)


# ---------------------------------------------------------------- page values

def test_k2_parameter_counts_match_pages():
    g = json.load(open(os.path.join(GOLDEN, "k2_expert_params.json")))
    wl = syn.WORKLOADS["k2_decode"]
    assert (wl.d, wl.d_ff, wl.num_experts, wl.top_k) == (g["d"], g["d_ff"], g["num_routed_experts"], g["top_k"])
    per_proj = wl.d * wl.d_ff
    assert per_proj == g["gate_projection_params"] == g["up_projection_params"] == g["down_projection_params"]
    assert 3 * per_proj == g["params_per_expert"]
    assert 3 * per_proj * g["num_routed_experts"] * g["moe_blocks"] == g["routed_params_all_blocks"]
    # The generator's tensors have exactly those element counts (scales excluded, as the page says).
    bank = syn.ExpertBank(*(torch.empty(0) for _ in range(6)))
    shapes = [(wl.d_ff, wl.d), (wl.d_ff, wl.d), (wl.d, wl.d_ff)]
    assert sum(a * b for a, b in shapes) == g["params_per_expert"]
    del bank


# ---------------------------------------------------------------- number formats

def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == ref[~nan]).all()
    # signed zero
    assert math.copysign(1.0, oracle.e4m3_value(0x80)) == -1.0


def test_e4m3_named_points():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_points.json")))
    for p in g["points"]:
        v = oracle.e4m3_value(int(p["code"], 16))
        if p["value"] == "nan":
            assert math.isnan(v)
        else:
            assert v == p["value"] and math.copysign(1, v) == math.copysign(1, p["value"])


def test_bf16_decode_matches_torch():
    bits = torch.randint(0, 1 << 16, (4096,), dtype=torch.int32)
    bits = torch.cat([bits, torch.tensor([0, 0x8000, 0x3F80, 0x7F7F, 0x0001, 0xFF7F])])
    ref = bits.to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    ours = np.array([oracle.bf16_value(int(b) & 0xFFFF) for b in bits])
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == ref[~nan]).all()


def test_dequant_matches_library_and_scale_layout():
    torch.manual_seed(3)
    w = torch.randn(256, 384) * torch.linspace(0.01, 1.0, 384)   # block scales differ by column block
    w[:128] *= 7.0                                                # and by row block
    q, s = syn.quantize_blockwise(w)
    assert s.shape == (2, 3) and len(set(s.flatten().tolist())) == 6
    ours = oracle.dequant(q, s)
    ref = _deq_torch(q, s).numpy()
    assert (ours == ref).all()
    # The quantiser maps each block's amax to +-448 exactly (scale = amax / 448).
    deq_amax = np.abs(ref).reshape(2, 128, 3, 128).max(axis=(1, 3))
    assert (deq_amax == s.numpy().astype(np.float64) * 448.0).all()


# ---------------------------------------------------------------- activation

def test_silu_special_values_and_library():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(50.0) == pytest.approx(50.0, rel=1e-15)
    assert abs(oracle.silu(-50.0)) < 1e-19
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    xs = torch.linspace(-30, 30, 1201, dtype=torch.float64)
    ref = F.silu(xs).numpy()
    ours = np.array([oracle.silu(float(v)) for v in xs])
    assert np.allclose(ours, ref, rtol=1e-14, atol=1e-300)


# ---------------------------------------------------------------- one expert

def test_expert_matches_fp64_matmul_with_library_silu():
    d, dff = 256, 384
    b = _small_bank(1, d, dff, seed=11)
    x = torch.randn(5, d, dtype=torch.float64, generator=torch.Generator().manual_seed(5))
    Wg = _deq_torch(b.w_gate[0], b.s_gate[0])
    Wu = _deq_torch(b.w_up[0], b.s_up[0])
    Wd = _deq_torch(b.w_down[0], b.s_down[0])
    ref = (F.silu(x @ Wg.T) * (x @ Wu.T)) @ Wd.T
    ours = oracle.expert_forward(x.numpy(), b.w_gate[0], b.s_gate[0], b.w_up[0], b.s_up[0],
                                 b.w_down[0], b.s_down[0])
    assert np.allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-14)


def _perm_code_matrix(perm, code=0x38):
    """e4m3 codes of a 0/1 matrix with a one at (r, perm[r]); 0x38 encodes 1.0."""
    n = len(perm)
    q = torch.zeros(n, n, dtype=torch.uint8)
    q[torch.arange(n), torch.as_tensor(perm)] = code
    return q


def test_expert_closed_form_with_permutation_weights():
    """gate = a*P, up = b*Q, down = c*R (P, Q, R permutation matrices, one scale per matrix).
    Then expert(x)[i] = c * silu(a x[P^-1...]) ... written out by indices: a transposed or
    mis-indexed operand moves entries and fails."""
    n = 256
    rng = np.random.default_rng(7)
    P, Q, Rm = (rng.permutation(n) for _ in range(3))
    a, b_, c = 0.5, 0.25, 2.0
    sg = torch.full((2, 2), a)
    su = torch.full((2, 2), b_)
    sd = torch.full((2, 2), c)
    x = rng.standard_normal((3, n))
    ours = oracle.expert_forward(x, _perm_code_matrix(P), sg, _perm_code_matrix(Q), su,
                                 _perm_code_matrix(Rm), sd)
    g = a * x[:, P]                      # (gate x)[f] = a * x[P[f]]
    u = b_ * x[:, Q]
    h = g / (1 + np.exp(-g)) * u
    y = c * h[:, Rm]                     # (down h)[r] = c * h[R[r]]
    assert np.allclose(ours, y, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- RMSNorm

def _bf16_bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_round(a):
    """Nearest bf16 of float32 values, through torch's own conversion."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


def test_rmsnorm_constant_rows_closed_form():
    # A constant row c has mean square c^2: with eps = 0 the normalised row is
    # sign(c) exactly, and the output is bf16(gain * sign(c)) = +-gain.
    d = 512
    gain = torch.linspace(0.5, 1.5, d)
    gb = _bf16_bits(gain)
    g = gain.to(torch.bfloat16).double().numpy()
    for cval in (0.5, -3.0, 1e-3, 96.0):
        hb = _bf16_bits(torch.full((1, d), cval))
        assert np.array_equal(oracle.rmsnorm(hb, gb, 0.0)[0], np.sign(cval) * g)
    # eps enters as mean(h^2) + eps: 0.5 / sqrt(0.25 + 0.75) = 0.5 exactly
    ones = _bf16_bits(torch.ones(d))
    y = oracle.rmsnorm(_bf16_bits(torch.full((1, d), 0.5)), ones, 0.75)
    assert np.array_equal(y, np.full((1, d), 0.5))
    # and 3 / sqrt(9 + 7) = 0.75
    y = oracle.rmsnorm(_bf16_bits(torch.full((1, d), 3.0)), ones, 7.0)
    assert np.array_equal(y, np.full((1, d), 0.75))


def test_rmsnorm_invariants():
    d = 1024
    h = torch.randn(4, d, generator=torch.Generator().manual_seed(1))
    ones = torch.ones(d)
    xn = oracle.rmsnorm(_bf16_bits(h), _bf16_bits(ones), 0.0)
    # the output is a bf16 tensor, as the excerpt's cast makes it
    assert np.array_equal(xn, _bf16_round(xn))
    # unit gain, eps = 0: every output row has mean square 1 up to the bf16 rounding
    assert np.allclose((xn ** 2).mean(axis=1), 1.0, rtol=2e-3)
    # the unrounded normalised row is h / rms(h); the output is its nearest bf16
    hd = h.to(torch.bfloat16).double().numpy()
    exact = hd / np.sqrt((hd ** 2).mean(axis=1, keepdims=True))
    assert np.max(np.abs(xn - exact) / np.abs(exact)) <= 2.0 ** -8 * (1 + 1e-6)
    # scale invariance (power-of-two scale keeps the bf16 input exact)
    xn2 = oracle.rmsnorm(_bf16_bits(h * 8.0), _bf16_bits(ones), 0.0)
    assert np.array_equal(xn, xn2)
    # the gain multiplies the bf16 normalised row feature-wise, then rounds once more
    gain = torch.linspace(-2, 2, d).to(torch.bfloat16)
    yg = oracle.rmsnorm(_bf16_bits(h), _bf16_bits(gain), 0.0)
    assert np.array_equal(yg, _bf16_round(xn * gain.double().numpy()[None, :]))


# ---------------------------------------------------------------- routing plan

@pytest.mark.parametrize("n,k,E,seed", [(128, 4, 16, 0), (1, 8, 384, 1), (37, 8, 384, 2), (300, 6, 33, 3),
                                        (64, 8, 384, 4)])
def test_permute_matches_bincount_and_stable_argsort(n, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    ids = syn.routing_uniform(n, E, k, g)
    counts, offsets, sp, ip, bad = oracle.permute(ids, E)
    flat = ids.reshape(-1).long()
    assert bad == 0
    assert (counts == torch.bincount(flat, minlength=E).numpy()).all()
    assert counts.sum() == n * k
    assert (offsets == np.concatenate([[0], np.cumsum(counts)])).all()
    assert (sp == torch.argsort(flat, stable=True).numpy()).all()
    assert (np.sort(sp) == np.arange(n * k)).all()                 # bijection
    assert (ip[sp] == np.arange(n * k)).all() and (sp[ip] == np.arange(n * k)).all()


def test_permute_ties_are_by_flat_index_and_skewed_counts():
    g = torch.Generator().manual_seed(9)
    ids = syn.routing_zipf(2000, 384, 8, 1.2, g)
    counts, offsets, sp, ip, _ = oracle.permute(ids, 384)
    flat = ids.reshape(-1).numpy()
    for e in range(384):
        seg = sp[offsets[e]:offsets[e + 1]]
        assert (flat[seg] == e).all()
        assert (np.diff(seg) > 0).all()                            # ascending flat index within an expert
    assert counts.max() > 4 * counts.mean()


def test_permute_empty_experts_and_out_of_range_ids():
    ids = torch.tensor([[3, 1], [1, 7], [-1, 3], [9, 1]], dtype=torch.int32)
    counts, offsets, sp, ip, bad = oracle.permute(ids, 8)
    assert bad == 2
    assert counts.tolist() == [0, 3, 0, 2, 0, 0, 0, 1]
    assert offsets.tolist() == [0, 0, 3, 3, 5, 5, 5, 5, 6]
    assert sp.tolist() == [1, 2, 7, 0, 5, 3, -1, -1]
    assert ip.tolist() == [3, 0, 1, 5, -1, 4, -1, 2]


# ---------------------------------------------------------------- routed sum

def _restated_moe_infer_fp64(x_bf16, ids, w, bank):
    """Independent restatement of the pages' moe_infer (count, stable sort, gather, per-expert
    slices, scatter back, weighted sum) with torch library primitives in fp64."""
    n, k = ids.shape
    E = bank.w_gate.shape[0]
    x = x_bf16.to(torch.float64)
    flat = ids.reshape(-1).long()
    tokens_per_expert = torch.bincount(flat, minlength=E)
    idxs = torch.argsort(flat, stable=True)
    sorted_tokens = x[idxs // k]
    outs = []
    start = 0
    for e in range(E):
        cnt = int(tokens_per_expert[e])
        if cnt == 0:
            continue
        xe = sorted_tokens[start:start + cnt]
        Wg = _deq_torch(bank.w_gate[e], bank.s_gate[e])
        Wu = _deq_torch(bank.w_up[e], bank.s_up[e])
        Wd = _deq_torch(bank.w_down[e], bank.s_down[e])
        outs.append((F.silu(xe @ Wg.T) * (xe @ Wu.T)) @ Wd.T)
        start += cnt
    outs = torch.cat(outs)
    new_x = torch.empty_like(outs)
    new_x[idxs] = outs
    return (new_x.view(n, k, -1) * w.to(torch.float64)[:, :, None]).sum(dim=1)


def test_oracle_matches_fp64_restatement_tiny():
    inp = syn.make_inputs(syn.WORKLOADS["tiny"])
    ours = oracle.moe_infer(inp.x, inp.topk_ids, inp.topk_weight, inp.bank)
    ref = _restated_moe_infer_fp64(inp.x, inp.topk_ids, inp.topk_weight, inp.bank).numpy()
    rel = np.abs(ours - ref).max() / np.abs(ref).max()
    assert rel < 1e-12


@pytest.mark.parametrize("n,d,dff,E,k,seed", [(128, 1024, 256, 16, 4, 0), (23, 256, 128, 8, 3, 1),
                                              (9, 128, 384, 5, 5, 2)])
def test_sorted_slice_form_equals_token_loop_bitwise(n, d, dff, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g).to(torch.bfloat16)
    ids = syn.routing_uniform(n, E, k, g)
    w = syn.router_weights(n, k, g)
    bank = _small_bank(E, d, dff, seed)
    a = oracle.moe_infer(x, ids, w, bank)
    b = oracle.moe_infer_sorted(x, ids, w, bank)
    assert np.array_equal(a, b)


def test_single_expert_unit_weight_reduces_to_expert():
    d, dff, E = 256, 256, 6
    g = torch.Generator().manual_seed(4)
    x = torch.randn(7, d, generator=g).to(torch.bfloat16)
    ids = torch.tensor([[2], [5], [0], [2], [3], [1], [4]], dtype=torch.int32)
    w = torch.ones(7, 1)
    bank = _small_bank(E, d, dff, 4)
    y = oracle.moe_infer(x, ids, w, bank)
    for t in range(7):
        e = int(ids[t, 0])
        ref = oracle.expert_forward(x[t:t + 1].double().numpy(), bank.w_gate[e], bank.s_gate[e], bank.w_up[e],
                                    bank.s_up[e], bank.w_down[e], bank.s_down[e])
        assert np.array_equal(y[t], ref[0])


def test_routed_sum_is_linear_in_router_weights_and_uses_each_slot():
    inp = syn.make_inputs(syn.WORKLOADS["tiny"], n_tokens=16)
    # weights on a 2^-12 grid so that w1 + w2 is exact in fp32
    w1 = torch.round(inp.topk_weight * 4096) / 4096
    w2 = torch.round(torch.rand(w1.shape, generator=torch.Generator().manual_seed(8)) * 1024) / 1024
    y1 = oracle.moe_infer(inp.x, inp.topk_ids, w1, inp.bank)
    y2 = oracle.moe_infer(inp.x, inp.topk_ids, w2, inp.bank)
    y12 = oracle.moe_infer(inp.x, inp.topk_ids, w1 + w2, inp.bank)
    assert np.allclose(y12, y1 + y2, rtol=1e-12, atol=1e-14)
    # zeroing slot j removes exactly expert ids[t, j]'s contribution
    wz = w1.clone()
    wz[:, 1] = 0
    yz = oracle.moe_infer(inp.x, inp.topk_ids, wz, inp.bank)
    for t in range(3):
        e = int(inp.topk_ids[t, 1])
        o = oracle.expert_forward(inp.x[t:t + 1].double().numpy(), inp.bank.w_gate[e], inp.bank.s_gate[e],
                                  inp.bank.w_up[e], inp.bank.s_up[e], inp.bank.w_down[e], inp.bank.s_down[e])
        assert np.allclose(y1[t] - yz[t], float(w1[t, 1]) * o[0], rtol=1e-10, atol=1e-13)


def test_token_subset_matches_full_run():
    inp = syn.make_inputs(syn.WORKLOADS["tiny"])
    full = oracle.moe_infer(inp.x, inp.topk_ids, inp.topk_weight, inp.bank)
    sel = [0, 5, 127, 64, 5]
    sub = oracle.moe_infer(inp.x, inp.topk_ids, inp.topk_weight, inp.bank, tokens=sel)
    assert np.array_equal(sub, full[sel])


# ---------------------------------------------------------------- full block

def test_layer_forward_matches_fp64_restatement():
    wl = syn.Workload("blk", 24, 256, 128, 8, 3, full_block=True, d_ff_shared=256, seed=6)
    inp = syn.make_inputs(wl)
    y = oracle.layer_forward(inp.x, inp.gain, inp.eps, inp.topk_ids, inp.topk_weight, inp.bank, inp.shared)
    h = inp.x.double()
    # the excerpt's RMSNorm in torch: float32 row, variance (the exact mean of
    # squares rounded to float32), h * rsqrt(variance + eps), cast to bf16, times the bf16 gain
    h32 = inp.x.float()
    variance = (h * h).mean(dim=1, keepdim=True).float()
    normed = (h32 * (1.0 / torch.sqrt(variance + inp.eps))).to(torch.bfloat16)
    xn = (inp.gain.to(torch.bfloat16) * normed).double()
    # routed part via the restatement, fed with xn
    n, k = inp.topk_ids.shape
    routed = torch.zeros(n, wl.d, dtype=torch.float64)
    for t in range(n):
        for j in range(k):
            e = int(inp.topk_ids[t, j])
            Wg = _deq_torch(inp.bank.w_gate[e], inp.bank.s_gate[e])
            Wu = _deq_torch(inp.bank.w_up[e], inp.bank.s_up[e])
            Wd = _deq_torch(inp.bank.w_down[e], inp.bank.s_down[e])
            routed[t] += float(inp.topk_weight[t, j]) * ((F.silu(Wg @ xn[t]) * (Wu @ xn[t])) @ Wd.T)
    S = inp.shared
    shared = (F.silu(xn @ _deq_torch(S.w_gate[0], S.s_gate[0]).T) * (xn @ _deq_torch(S.w_up[0], S.s_up[0]).T)) \
        @ _deq_torch(S.w_down[0], S.s_down[0]).T
    ref = (h + (routed + shared)).numpy()
    assert np.allclose(y, ref, rtol=1e-11, atol=1e-12)


def test_layer_forward_zero_router_weights_no_shared_is_identity():
    wl = syn.Workload("blk", 8, 256, 128, 4, 2, full_block=True, seed=2)
    inp = syn.make_inputs(wl)
    y = oracle.layer_forward(inp.x, inp.gain, inp.eps, inp.topk_ids, torch.zeros_like(inp.topk_weight), inp.bank)
    assert np.array_equal(y, inp.x.double().numpy())


# ---------------------------------------------------------------- dynamic FP8 activations
#
# "Input features" page, quantisation config: fmt e4m3, activation_scheme
# "dynamic", weight blocks of 128 x 128.  The oracle quantises every row
# entering a linear per group of 128 features (scale amax / 448 in float32,
# code = nearest e4m3 of v / s, ties to even, saturating).


def _torch_e4m3_codes(v32):
    """torch's float32 -> float8_e4m3fn cast (round to nearest, ties to even) as code bytes."""
    return v32.to(torch.float8_e4m3fn).view(torch.uint8)


def test_e4m3_encode_matches_torch_cast_and_saturates():
    g = torch.Generator().manual_seed(21)
    vals = torch.tensor([oracle.e4m3_value(c) for c in range(0x7F)], dtype=torch.float64)
    mids = (vals[1:] + vals[:-1]) / 2              # exact ties between neighbouring codes
    pts = torch.cat([vals, mids, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20),
                     torch.rand(4000, generator=g, dtype=torch.float64) * 448,
                     torch.rand(2000, generator=g, dtype=torch.float64) * 2.0 ** -6])
    pts = torch.cat([pts, -pts]).float()
    ref = _torch_e4m3_codes(pts)
    ours = torch.tensor([oracle.e4m3_encode(float(v)) for v in pts], dtype=torch.uint8)
    assert torch.equal(ours, ref)
    # past the largest finite value the encoder saturates (torch's cast gives NaN there)
    for v, c in ((448.0, 0x7E), (460.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE)):
        assert oracle.e4m3_encode(v) == c
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def _fp8_rows():
    g = torch.Generator().manual_seed(22)
    v = torch.randn(3, 512, generator=g, dtype=torch.float64)
    v[:, 128:256] *= 1e-3        # groups of very different size in one row
    v[:, 256:384] *= 300.0
    v[1, 384:] = 0.0             # an all-zero group
    return v.float().double()    # float32 inputs


def test_fp8_dynamic_group_invariants():
    v = _fp8_rows()
    deq, codes, scales = oracle.fp8_dynamic(v.numpy())
    vn = v.numpy()
    assert scales.shape == (3, 4)
    for r in range(3):
        for gi in range(4):
            sl = slice(128 * gi, 128 * (gi + 1))
            grp, c, s = vn[r, sl], codes[r, sl], float(scales[r, gi])
            if not np.any(grp):
                assert s == 1.0 and not np.any(deq[r, sl]) and np.all((c & 0x7F) == 0)
                continue
            # the group's largest magnitude takes the largest code and nothing saturates:
            # 448 * s covers amax up to float32 rounding
            assert (c & 0x7F).max() == 0x7E
            amax = np.abs(grp).max()
            assert 448.0 * s >= amax * (1 - 2.0 ** -22) and 448.0 * s <= amax * (1 + 2.0 ** -22)
            # round to nearest: within half an e4m3 step (2^-4 relative, 2^-10 * s in the subnormals)
            err = np.abs(deq[r, sl] - grp)
            assert np.all(err <= 2.0 ** -4 * np.abs(grp) + 2.0 ** -10 * s)
            # codes times the scale are the returned values
            vals = np.array([oracle.e4m3_value(int(x)) for x in c])
            assert np.array_equal(deq[r, sl], vals * s)
            # the codes are torch's cast of v / s (float32 division)
            q = torch.from_numpy(grp.astype(np.float32)) / torch.tensor(s, dtype=torch.float32)
            assert torch.equal(_torch_e4m3_codes(q), torch.from_numpy(c.copy()))


def test_fp8_dynamic_groups_are_independent_and_scale_equivariant():
    v = _fp8_rows()
    deq, codes, scales = oracle.fp8_dynamic(v.numpy())
    w = v.clone()
    w[:, 256:384] *= 1e4                           # only group 2 changes
    deq2, codes2, scales2 = oracle.fp8_dynamic(w.numpy())
    keep = np.r_[0:256, 384:512]
    assert np.array_equal(deq[:, keep], deq2[:, keep]) and np.array_equal(scales[:, [0, 1, 3]],
                                                                          scales2[:, [0, 1, 3]])
    # a power-of-two factor moves only the scales
    deq3, codes3, scales3 = oracle.fp8_dynamic((v * 32.0).numpy())
    nz = scales != 1.0
    assert np.array_equal(codes3, codes) and np.array_equal(scales3[nz], scales[nz] * 32.0)
    assert np.array_equal(deq3, deq * 32.0)


def _torch_fp8_dynamic(v):
    """Per-128-feature dynamic quantisation restated with torch: float32 amax / 448, torch's e4m3 cast."""
    v32 = v.float()
    grp = v32.reshape(*v32.shape[:-1], -1, 128)
    s = grp.abs().amax(-1, keepdim=True) / 448.0
    s = torch.where(s > 0, s, torch.ones_like(s))
    q = (grp / s).clamp(-448, 448).to(torch.float8_e4m3fn).to(torch.float64)
    return (q * s.double()).reshape(v.shape)


def test_expert_fp8_act_matches_torch_restatement():
    d, dff = 256, 384
    b = _small_bank(1, d, dff, seed=11)
    x = torch.randn(5, d, dtype=torch.float64, generator=torch.Generator().manual_seed(5))
    Wg = _deq_torch(b.w_gate[0], b.s_gate[0])
    Wu = _deq_torch(b.w_up[0], b.s_up[0])
    Wd = _deq_torch(b.w_down[0], b.s_down[0])
    xq = _torch_fp8_dynamic(x)
    h = F.silu(xq @ Wg.T) * (xq @ Wu.T)
    ref = _torch_fp8_dynamic(h) @ Wd.T
    ours = oracle.expert_forward(x.numpy(), b.w_gate[0], b.s_gate[0], b.w_up[0], b.s_up[0],
                                 b.w_down[0], b.s_down[0], fp8_act=True)
    assert np.allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-14)
    # the scheme changes the result by about an e4m3 step, not by nothing
    exact = oracle.expert_forward(x.numpy(), b.w_gate[0], b.s_gate[0], b.w_up[0], b.s_up[0],
                                  b.w_down[0], b.s_down[0])
    rel = np.abs(ours - exact).mean() / np.abs(exact).mean()
    assert 3e-3 < rel < 1e-1


def test_moe_infer_fp8_act_matches_torch_restatement_tiny():
    inp = syn.make_inputs(syn.WORKLOADS["tiny"], n_tokens=24)
    ours = oracle.moe_infer(inp.x, inp.topk_ids, inp.topk_weight, inp.bank, fp8_act=True)
    xq = _torch_fp8_dynamic(inp.x.double())
    n, k = inp.topk_ids.shape
    ref = torch.zeros(n, inp.x.shape[1], dtype=torch.float64)
    for t in range(n):
        for j in range(k):
            e = int(inp.topk_ids[t, j])
            Wg = _deq_torch(inp.bank.w_gate[e], inp.bank.s_gate[e])
            Wu = _deq_torch(inp.bank.w_up[e], inp.bank.s_up[e])
            Wd = _deq_torch(inp.bank.w_down[e], inp.bank.s_down[e])
            h = F.silu(Wg @ xq[t]) * (Wu @ xq[t])
            ref[t] += float(inp.topk_weight[t, j]) * (Wd @ _torch_fp8_dynamic(h[None])[0])
    rel = np.abs(ours - ref.numpy()).max() / np.abs(ref.numpy()).max()
    assert rel < 1e-12
    # the sorted-slice form does the same arithmetic
    sorted_form = oracle.moe_infer_sorted(inp.x, inp.topk_ids, inp.topk_weight, inp.bank, fp8_act=True)
    assert np.array_equal(sorted_form, ours)


def test_layer_forward_fp8_act_quantises_the_normalised_row_and_shared_expert():
    wl = syn.Workload("blk", 6, 256, 128, 8, 3, full_block=True, d_ff_shared=256, seed=6)
    inp = syn.make_inputs(wl)
    y = oracle.layer_forward(inp.x, inp.gain, inp.eps, inp.topk_ids, inp.topk_weight, inp.bank, inp.shared,
                             fp8_act=True)
    xn = torch.from_numpy(oracle.rmsnorm(inp.x, inp.gain, inp.eps))
    xq = _torch_fp8_dynamic(xn)

    def expert(bank, e, row):
        Wg = _deq_torch(bank.w_gate[e], bank.s_gate[e])
        Wu = _deq_torch(bank.w_up[e], bank.s_up[e])
        Wd = _deq_torch(bank.w_down[e], bank.s_down[e])
        return Wd @ _torch_fp8_dynamic((F.silu(Wg @ row) * (Wu @ row))[None])[0]

    n, k = inp.topk_ids.shape
    ref = torch.zeros(n, wl.d, dtype=torch.float64)
    for t in range(n):
        for j in range(k):
            ref[t] += float(inp.topk_weight[t, j]) * expert(inp.bank, int(inp.topk_ids[t, j]), xq[t])
        ref[t] = inp.x[t].double() + (ref[t] + expert(inp.shared, 0, xq[t]))
    assert np.allclose(y, ref.numpy(), rtol=1e-11, atol=1e-12)
