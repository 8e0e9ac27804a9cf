"""Expert-parallel kernels on one GPU, the ranks simulated in one process.

Every device step of mixture_experts_ffn_infer_gb300/ep.py (moe_ep_dispatch_plan,
moe_ep_gather, moe_ep_regroup, moe_ep_experts_forward, moe_ep_combine) runs
through the C ABI for each simulated rank; the three exchanges are done by
slicing the ranks' buffers, as an all-to-all would deliver them.  Checked:

* the plans bit for bit against the oracle's restatement of the pages'
  multi-rank branch (oracle/ep.py): send splits, the count exchange, the
  position of every entry in the sorted order, the regroup order;
* every rank's output against the single-rank oracle on the whole bank, under
  the parity tolerance, with exact and fixed-capacity split sizes.
"""

import numpy as np
import pytest
import torch

import mixture_experts_ffn_infer_gb300 as mx
import oracle
from mixture_experts_ffn_infer_gb300 import ep as mep
from mixture_experts_ffn_infer_gb300 import synthetic as syn
from oracle import ep as oep
from tests import gpu_cases as cases

pytestmark = pytest.mark.gpu


def _simulate(xs, ids, ws, bank, ep, capacity):
    """The multi-rank forward of ep ranks on this GPU.  Returns (outputs, per-rank plan tensors)."""
    E = bank.w_gate.shape[0]
    epr = E // ep
    d, dff = xs[0].shape[1], bank.w_gate.shape[1]
    k = ids[0].shape[1]
    ops = [mep.DeviceOps(d, dff, E, k) for _ in range(ep)]
    disp = [mep.dispatch(ops[r], xs[r], ids[r], ep, capacity) for r in range(ep)]
    sc = [dp.send_counts.cpu().tolist() for dp in disp]

    def send_piece(s, r):  # rows source s sends to rank r, in its slot order
        if capacity:
            return disp[s].send_rows[r * capacity:(r + 1) * capacity]
        start = sum(sc[s][:r])
        return disp[s].send_rows[start:start + sc[s][r]]

    recv_counts = [torch.cat([disp[s].counts[r * epr:(r + 1) * epr] for s in range(ep)]) for r in range(ep)]
    recv_rows = [torch.cat([send_piece(s, r) for s in range(ep)]) for r in range(ep)]
    outs, regroups = [], []
    for r in range(ep):
        local = mep.shard_bank(bank, r, ep)
        lo, rp, pr = ops[r].regroup(recv_counts[r], epr, ep, capacity, recv_rows[r].shape[0])
        regroups.append((lo, rp, pr))
        outs.append(ops[r].experts(recv_rows[r], lo, rp, pr, local, epr, recv_rows[r].shape[0]))
    ys = []
    for s in range(ep):
        back = torch.zeros(disp[s].n_slots, d, dtype=torch.float16, device="cuda")
        for r in range(ep):
            # the piece of rank r's outputs that came from source s, back to s's slots
            if capacity:
                back[r * capacity:(r + 1) * capacity] = outs[r][s * capacity:(s + 1) * capacity]
            else:
                rstart = sum(sc[q][r] for q in range(s))
                start = sum(sc[s][:r])
                back[start:start + sc[s][r]] = outs[r][rstart:rstart + sc[s][r]]
        ys.append(mep.combine(ops[s], disp[s], back, ws[s]))
    torch.cuda.synchronize()
    for o in ops:
        assert o.errors() == mx.MOE_OK
    return ys, disp, recv_counts, regroups


def _inputs(ep, n, d, dff, E, k, routing="uniform", seed=0, bank=None):
    xs, ids, ws = [], [], []
    for r in range(ep):
        wl = syn.Workload("ep", n, d, dff, E, k, routing=routing, seed=seed + 17 * r)
        x, i, w, _ = syn.make_host_inputs(wl)
        xs.append(x.cuda())
        ids.append(i.cuda())
        ws.append(w.cuda())
    if bank is None:
        bank = syn.ExpertBank(*(t.cuda() for t in dataclass_astuple(syn.expert_bank(E, d, dff, seed + 3, "cpu"))))
    return xs, ids, ws, bank


def dataclass_astuple(b):
    return (b.w_gate, b.w_up, b.w_down, b.s_gate, b.s_up, b.s_down)


@pytest.mark.parametrize("ep,capacity,routing", [(2, 0, "uniform"), (2, 1, "zipf"), (4, 0, "zipf"),
                                                 (4, 1, "uniform")])
def test_ep_plans_bit_exact_and_outputs_small(ep, capacity, routing):
    d, dff, E, k, n = 256, 256, 16, 4, 60
    xs, ids, ws, bank = _inputs(ep, n, d, dff, E, k, routing, seed=ep * 10 + capacity)
    cap = n * k if capacity else 0
    ys, disp, recv_counts, regroups = _simulate(xs, ids, ws, bank, ep, cap)
    plans = oep.ep_plan([i.cpu() for i in ids], E, ep)
    for r in range(ep):
        p = plans[r]
        assert disp[r].counts.cpu().tolist() == p["tokens_per_expert"].tolist()
        assert disp[r].send_counts.cpu().tolist() == p["input_split_sizes"].tolist()
        slot = disp[r].tok_slot.cpu().numpy()
        if cap == 0:
            assert np.array_equal(slot[p["idxs"]], np.arange(slot.size))   # entry idxs[i] travels in slot i
        assert recv_counts[r].cpu().tolist() == p["tokens_per_expert_group"].tolist()
        lo, rp, pr = (t.cpu().numpy() for t in regroups[r])
        assert lo[-1] == p["gatherd_idxs"].size
        assert np.array_equal(np.diff(lo), p["tokens_per_expert_post_gather"])
        if cap == 0:
            # gatherd_idxs[q] is the received row at expert-order position q
            assert np.array_equal(rp[p["gatherd_idxs"]], np.arange(p["gatherd_idxs"].size))
            assert np.array_equal(pr[:lo[-1]], p["gatherd_idxs"])
        ref = oracle.moe_infer(xs[r].cpu(), ids[r].cpu(), ws[r].cpu(), syn.ExpertBank(*(t.cpu() for t in dataclass_astuple(bank))))
        rep = oracle.parity_report(ys[r], ref, bf16_output=True)
        assert rep["ok"], (r, rep)


@pytest.mark.parametrize("ep,n", [(4, 320), (2, 16)])
def test_ep_k2_shards(ep, n):
    # the K2 bank split over simulated ranks: 4 ranks of 96 experts with 320 tokens each give each local
    # expert about 27 received rows (wide tiles); 2 ranks with 16 tokens each, decode-sized (16-token
    # tiles).  The oracle checks a sample of every rank's tokens.
    bank = cases.k2_bank(1)
    xs, ids, ws, _ = _inputs(ep, n, 7168, 2048, 384, 8, seed=5, bank=bank)
    ys, disp, recv_counts, regroups = _simulate(xs, ids, ws, bank, ep, 0)
    tot = sum(int(rc.sum()) for rc in recv_counts)
    assert tot == ep * n * 8
    g = torch.Generator().manual_seed(0)
    for r in range(ep):
        tok = sorted(torch.randperm(n, generator=g)[:min(n, 12)].tolist())
        ref = oracle.moe_infer(xs[r].cpu(), ids[r].cpu(), ws[r].cpu(), bank, tokens=tok)
        rep = oracle.parity_report(ys[r][tok], ref, bf16_output=True)
        assert rep["ok"], (r, rep)
