"""Host-side arithmetic of bench.py's roofline report (no GPU): which roof bounds
each GEMM and how the fraction is formed.

A GEMM is HBM-bound when its algorithmic bytes take longer at the copy bandwidth
than its algorithmic flops at the tensor peak of its MMAs' operand type (e4m3
for 16-token tiles and the dynamic FP8 scheme, f16 for the exact scheme's wide
tiles): the decode and prefill batches are, the full block (683 rows per expert)
is not."""

import torch

import bench
from mixture_experts_ffn_infer_gb300 import synthetic as syn

HBM = 6695.5              # GB/s
E4M3 = 1720.0 * 2.0       # TFLOP/s


def _alg(name, touched):
    wl = syn.WORKLOADS[name]
    ids = torch.arange(touched, dtype=torch.int32).reshape(1, -1)   # only the touched count matters
    return wl, bench.algorithmic(wl, [ids], wl.n_tokens)


def test_algorithmic_flops_per_gemm():
    wl, a = _alg("k2_decode", 104)
    R = wl.n_tokens * wl.top_k
    assert a["gateup_flops"] == 4 * wl.d * wl.d_ff * R
    assert a["down_flops"] == 2 * wl.d * wl.d_ff * R
    assert a["gateup_flops"] + a["down_flops"] == a["step_flops"]
    # weights of the touched experts dominate the decode bytes: 2 of 3 projections in gate/up
    per_proj = wl.d * wl.d_ff + (wl.d // 128) * (wl.d_ff // 128) * 4
    assert a["gateup_bytes"] == 104 * 2 * per_proj + R * wl.d * 2 + R * wl.d_ff * 2


def test_decode_and_prefill_gemms_are_hbm_bound():
    for name, touched in (("k2_decode", 104), ("k2_prefill", 384)):
        _, a = _alg(name, touched)
        t_hbm = a["gateup_bytes"] / (HBM * 1e9) * 1e3
        r = bench.kernel_roofline("gateup_swiglu", a["gateup_bytes"], a["gateup_flops"], t_hbm * 2, HBM, "m",
                                  E4M3, "m", None)
        assert r["bound"] == "hbm" and r["unit"] == "GB/s"
        assert abs(r["frac"] - 0.5) < 1e-12          # twice the roofline time: half of the peak
        assert abs(r["t_roof_ms"] - t_hbm) < 1e-9


def test_full_block_gemms_are_tensor_bound():
    _, a = _alg("k2_block", 384)
    for kern, b, f in (("gateup_swiglu", a["gateup_bytes"], a["gateup_flops"]),
                       ("down_scatter", a["down_bytes"], a["down_flops"])):
        t_tensor = f / (E4M3 * 1e12) * 1e3
        assert t_tensor > b / (HBM * 1e9) * 1e3
        r = bench.kernel_roofline(kern, b, f, t_tensor * 4, HBM, "m", E4M3, "m", None)
        assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == E4M3
        assert abs(r["achieved"] - E4M3 / 4) < 1e-6 and abs(r["frac"] - 0.25) < 1e-12


def test_missing_kernel_time_reports_no_fraction():
    _, a = _alg("k2_decode", 104)
    r = bench.kernel_roofline("down_scatter", a["down_bytes"], a["down_flops"], None, HBM, "m", E4M3, "m", None)
    assert r["achieved"] is None and r["frac"] is None and r["bound"] == "hbm"


def test_traffic_record_is_used_only_for_its_scheme_and_unchanged_source(tmp_path, monkeypatch):
    import hashlib
    import json
    src = tmp_path / "mixture_experts_ffn_infer_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("kernel v1\n")
    (tmp_path / "profiles").mkdir()
    sha = hashlib.sha256(b"kernel v1\n").hexdigest()
    (tmp_path / "profiles" / "traffic_w.json").write_text(json.dumps(
        {"source": "k.cu", "source_sha256": sha, "gateup_swiglu": 111}))
    (tmp_path / "profiles" / "traffic_w_fp8.json").write_text(json.dumps(
        {"source": "k.cu", "source_sha256": sha, "gateup_swiglu": 222}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("w", "gateup_swiglu") == 111
    assert bench._traffic("w", "gateup_swiglu", fp8=True) == 222
    assert bench._traffic("w", "down_scatter") is None          # no counters for that kernel
    assert bench._traffic("other", "gateup_swiglu") is None     # no record for the workload
    (src / "k.cu").write_text("kernel v2\n")                    # the kernel changed since the capture
    assert bench._traffic("w", "gateup_swiglu") is None
    assert bench._traffic("w", "gateup_swiglu", fp8=True) is None


def test_tile_width_rule_and_tensor_peak_per_workload():
    # wide tiles from an average of 24 routed rows per expert on (the library's tile_tokens)
    assert not bench.wide_tiles(24 * 384 // 8 - 1, 8, 384)
    assert bench.wide_tiles(24 * 384 // 8, 8, 384)
    widths = {name: bench.wide_tiles(wl.n_tokens, wl.top_k, wl.num_experts) for name, wl in syn.WORKLOADS.items()}
    assert widths["k2_decode"] is False
    assert widths["k2_prefill"] and widths["k2_skewed"] and widths["k2_block"]
    # at the f16 rate the full block's GEMMs stay tensor-bound, prefill's HBM-bound
    BF16 = 1720.0
    _, a = _alg("k2_block", 384)
    r = bench.kernel_roofline("gateup_swiglu", a["gateup_bytes"], a["gateup_flops"], 1.0, HBM, "m", BF16, "m", None)
    assert r["bound"] == "tensor" and r["peak"] == BF16
    _, a = _alg("k2_prefill", 384)
    r = bench.kernel_roofline("gateup_swiglu", a["gateup_bytes"], a["gateup_flops"], 1.0, HBM, "m", BF16, "m", None)
    assert r["bound"] == "hbm"
