"""The local steps of the expert-parallel forward on the CPU, from the oracle.

For tests of the exchanges on gloo ranks (CPU processes): the orchestrator in
mixture_experts_ffn_infer_gb300/ep.py runs unchanged, with this object in place
of its device steps, so the all-to-alls, split sizes, slot layouts and the
reverse path are exercised across real ranks.  The arithmetic is the oracle's
(fp64 expert rows, slots summed in ascending order), so each rank's result
must equal the single-rank oracle bit for bit.  Rows travel as fp64.
"""

import numpy as np
import torch

import oracle


def _bf16_to_f64(x: torch.Tensor) -> torch.Tensor:
    bits = x.view(torch.int16).numpy().astype(np.uint16)
    return torch.from_numpy((bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64))


class OracleOps:
    def __init__(self, d, num_experts, top_k):
        self.d, self.E, self.k = d, num_experts, top_k

    def plan(self, topk_ids, ep, capacity):
        flat = topk_ids.reshape(-1).long()
        epr = self.E // ep
        counts = torch.bincount(flat, minlength=self.E).to(torch.int32)
        idxs = torch.argsort(flat, stable=True)
        inv = torch.empty_like(idxs)
        inv[idxs] = torch.arange(idxs.numel())
        send_counts = counts.view(ep, epr).sum(dim=1).to(torch.int32)
        if capacity == 0:
            slot = inv
        else:
            starts = torch.cumsum(send_counts, 0) - send_counts   # first sorted position of each rank's rows
            d = flat // epr
            slot = d * capacity + (inv - starts[d])
            assert int((inv - starts[d]).max()) < capacity
        return counts, send_counts, slot.to(torch.int32)

    def gather(self, x, tok_slot, n_slots):
        rows = torch.zeros(n_slots, self.d, dtype=torch.float64)
        xv = _bf16_to_f64(x)
        for f, s in enumerate(tok_slot.tolist()):
            if s >= 0:
                rows[s] = xv[f // self.k]
        return rows

    def regroup(self, recv_counts, epr, ep, capacity, n_slots):
        cnt = recv_counts.view(ep, epr).long()
        labels = torch.full((n_slots,), -1, dtype=torch.long)
        s = 0
        for r in range(ep):
            if capacity:
                s = r * capacity
            for e in range(epr):
                labels[s:s + cnt[r, e]] = e
                s += int(cnt[r, e])
        used = (labels >= 0).nonzero().flatten()
        order = used[torch.argsort(labels[used], stable=True)]   # received slots in expert order
        row_pos = torch.full((n_slots,), -1, dtype=torch.int32)
        row_pos[order] = torch.arange(order.numel(), dtype=torch.int32)
        pos_row = order.to(torch.int32)
        local_offsets = torch.zeros(epr + 1, dtype=torch.int32)
        local_offsets[1:] = torch.cumsum(cnt.sum(dim=0), 0)
        return local_offsets, row_pos, pos_row

    def experts(self, recv_rows, local_offsets, row_pos, pos_row, local_bank, epr, n_slots):
        out = torch.zeros(n_slots, self.d, dtype=torch.float64)
        for e in range(epr):
            lo, hi = int(local_offsets[e]), int(local_offsets[e + 1])
            if hi == lo:
                continue
            slots = pos_row[lo:hi].long()
            W = [getattr(local_bank, nm)[e] for nm in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")]
            out[slots] = torch.from_numpy(oracle.expert_forward(recv_rows[slots].numpy(), *W))
        return out

    def combine(self, back_rows, tok_slot, n_slots, topk_weight, out_is_fp32=False):
        n, k = topk_weight.shape
        w = topk_weight.double()
        acc = torch.zeros(n, self.d, dtype=torch.float64)
        slot = tok_slot.view(n, k).long()
        for j in range(k):  # ascending slot order
            acc += w[:, j:j + 1] * back_rows[slot[:, j]]
        return acc
