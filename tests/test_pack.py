"""moe_pack_weights: the tiled streaming layout is a pure rearrangement of the
e4m3 codes (checked byte for byte against a torch statement of the layout),
and results computed from a tiled bank equal those from the row-major bank."""

import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu


def _expected_tiles(q: torch.Tensor) -> torch.Tensor:
    """[E, R, C] codes -> tiles [E, R/128, C/128, 128 rows, 8 chunks, 16 B] with chunk j of row r at j ^ (r % 8)."""
    E, R, C = q.shape
    t = q.reshape(E, R // 128, 128, C // 128, 8, 16).permute(0, 1, 3, 2, 4, 5).contiguous()
    out = torch.empty_like(t)
    r = torch.arange(128)
    for j in range(8):
        out[:, :, :, r, (j ^ (r % 8)), :] = t[:, :, :, r, j, :]
    return out.reshape(-1)


def test_pack_layout_bytes():
    bank = syn.expert_bank(3, 384, 256, seed=5)
    dev = cases.bank_to(bank, "cuda")
    tiled = mx.pack_bank(dev)
    torch.cuda.synchronize()
    for name in ("w_gate", "w_up", "w_down"):
        got = getattr(tiled, name).reshape(-1).cpu()
        assert torch.equal(got, _expected_tiles(getattr(bank, name))), name


def test_pack_rejects_overlap_and_tiled_source():
    bank = cases.bank_to(syn.expert_bank(1, 128, 128, seed=1), "cuda")
    w = mx.weights(bank)
    with pytest.raises(mx.MoeError):
        mx.moe_pack_weights(1, 128, 128, w, w)
    t = mx.pack_bank(bank)
    with pytest.raises(mx.MoeError):
        mx.moe_pack_weights(1, 128, 128, mx.weights(t), w)


@pytest.mark.parametrize("name", ["tiny", "k2_decode"])
def test_tiled_bank_gives_identical_results(name):
    c = cases.workload(name)
    y_rm = mx.infer(c.x, c.ids, c.w, c.bank)
    tiled = mx.pack_bank(c.bank)
    y_t = mx.infer(c.x, c.ids, c.w, tiled)
    assert torch.equal(y_rm, y_t)
    del tiled


def test_tiled_layer_with_shared_expert():
    wl = syn.Workload("blk", 40, 256, 256, 6, 3, full_block=True, d_ff_shared=128, seed=3)
    c = cases.workload(wl)
    a = mx.layer_forward(c.x, c.gain, c.inp.eps, c.ids, c.w, c.bank, c.shared)
    b = mx.layer_forward(c.x, c.gain, c.inp.eps, c.ids, c.w, mx.pack_bank(c.bank), mx.pack_bank(c.shared))
    assert torch.equal(a, b)
