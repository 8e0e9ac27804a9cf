"""moe_pack_weights: the tiled streaming layout is a pure rearrangement of the
e4m3 codes (checked byte for byte against a torch statement of the layout),
and results computed from a tiled bank equal those from the row-major bank."""

import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu


def _swizzled_tiles(q: torch.Tensor) -> torch.Tensor:
    """[E, R, C] codes -> [E, R/128, C/128, 128 rows, 8 chunks, 16 B] with chunk j of row r at j ^ (r % 8)."""
    E, R, C = q.shape
    t = q.reshape(E, R // 128, 128, C // 128, 8, 16).permute(0, 1, 3, 2, 4, 5).contiguous()
    out = torch.empty_like(t)
    r = torch.arange(128)
    for j in range(8):
        out[:, :, :, r, (j ^ (r % 8)), :] = t[:, :, :, r, j, :]
    return out


def _expected_gate_up(gate, up):
    """Tile (e, b, c, m): gate (m = 0) and up (m = 1) of row block b, column block c."""
    return torch.stack([_swizzled_tiles(gate), _swizzled_tiles(up)], dim=3).reshape(-1)


def _expected_down(down):
    """Tile (e, p, c, m): down row block 2p + m (zeros past the last block), column block c."""
    t = _swizzled_tiles(down)                      # [E, nrb, nc, ...]
    E, nrb = t.shape[:2]
    if nrb % 2:
        t = torch.cat([t, torch.zeros_like(t[:, :1])], dim=1)
    t = t.reshape(E, t.shape[1] // 2, 2, *t.shape[2:]).transpose(2, 3)
    return t.reshape(-1)


def test_pack_layout_bytes():
    # d / 128 = 3 row blocks of down: the last pair has one block and a zero tile
    bank = syn.expert_bank(3, 384, 256, seed=5)
    dev = cases.bank_to(bank, "cuda")
    tiled = mx.pack_bank(dev)
    torch.cuda.synchronize()
    assert tiled.w_gate.numel() == mx.moe_tiled_bytes(0, 3, 384, 256) == 2 * bank.w_gate.numel()
    assert tiled.w_down.numel() == mx.moe_tiled_bytes(2, 3, 384, 256) == 3 * 4 * 128 * 256
    assert torch.equal(tiled.w_gate.cpu(), _expected_gate_up(bank.w_gate, bank.w_up))
    assert torch.equal(tiled.w_down.cpu(), _expected_down(bank.w_down))


def test_pack_rejects_overlap_and_tiled_source():
    bank = cases.bank_to(syn.expert_bank(1, 128, 128, seed=1), "cuda")
    w = mx.weights(bank)
    with pytest.raises(mx.MoeError):
        mx.moe_pack_weights(1, 128, 128, w, w)
    t = mx.pack_bank(bank)
    with pytest.raises(mx.MoeError):
        mx.moe_pack_weights(1, 128, 128, mx.weights(t), w)


@pytest.mark.parametrize("name", ["tiny", "k2_decode",
                                  syn.Workload("odd16", 37, 384, 384, 5, 3, seed=1),    # 16-token tiles, 3 down blocks
                                  syn.Workload("oddw", 150, 1152, 256, 4, 2, seed=8)])  # wide tiles, 9 down blocks
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
