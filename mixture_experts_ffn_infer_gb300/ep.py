"""Expert-parallel routed-expert forward over a torch.distributed group.

"Input features" page, expert construction: with ep_size ranks, rank r holds
experts [r * E/ep, (r + 1) * E/ep).  "Mixture of experts" page, moe_infer,
ep_size > 1 branch: each rank sends the rows it routes to rank r's experts to
rank r, runs its experts on what it receives (grouped by local expert), sends
the outputs back, and each token sums its k rows weighted by topk_weight.

This module only sequences the steps and performs the three exchanges
(torch.distributed all-to-all: NCCL between GPUs); every step on either side
of them runs in the library's kernels (``moe_ep_*`` in include/moe_ffn.h),
through ``DeviceOps``.

Split sizes of the row exchanges:
  capacity = 0  the pages' exact splits: after the count exchange the rank
                reads its send and receive counts back to the host (one
                synchronisation per call, as the pages' ``.cpu()`` calls);
  capacity = C  fixed splits of C rows per peer, no synchronisation: the send
                buffer holds ep * C slots, a rank routing more than C entries
                to one peer drops the rest and raises MOE_ERR_ROUTING
                (C = n * k never drops).
"""

from __future__ import annotations

import dataclasses
from typing import Any, Optional

import mixture_experts_ffn_infer_gb300 as mx


@dataclasses.dataclass
class Dispatch:
    """What a rank keeps between sending its rows and combining what comes back."""
    n_tokens: int
    top_k: int
    counts: Any           # [E] int32: entries per (global) expert, exchanged in step 3
    send_counts: Any      # [ep] int32: entries for each rank
    tok_slot: Any         # [n k] int32: send slot of each (token, slot) entry, -1 for none
    n_slots: int          # rows of the send buffer
    send_rows: Any        # [n_slots, d]


class DeviceOps:
    """The local steps on this process's CUDA device, through the C ABI."""

    def __init__(self, d: int, d_ff: int, num_experts: int, top_k: int, act_scheme: int = mx.MOE_ACT_EXACT):
        self.d, self.d_ff, self.E, self.k, self.act = d, d_ff, num_experts, top_k, act_scheme

    def dims(self):
        return mx.dims(self.d, self.d_ff, self.E, self.k, self.act)

    def plan(self, topk_ids, ep: int, capacity: int):
        import torch
        n = topk_ids.shape[0]
        dev = topk_ids.device
        dm = self.dims()
        ws = torch.zeros(max(mx.moe_ep_plan_workspace_size(dm, n), 256), dtype=torch.uint8, device=dev)
        counts = torch.empty(self.E, dtype=torch.int32, device=dev)
        send_counts = torch.empty(ep, dtype=torch.int32, device=dev)
        tok_slot = torch.empty(max(n * self.k, 1), dtype=torch.int32, device=dev)
        mx.moe_ep_dispatch_plan(dm, ep, n, topk_ids, counts, send_counts, tok_slot, capacity, ws)
        self.plan_ws = ws
        return counts, send_counts, tok_slot

    def gather(self, x, tok_slot, n_slots: int):
        import torch
        rows = torch.empty(max(n_slots, 1), self.d, dtype=x.dtype, device=x.device)
        mx.moe_ep_gather(self.dims(), x.shape[0], x, tok_slot, n_slots, rows)
        return rows[:n_slots]

    def regroup(self, recv_counts, epr: int, ep: int, capacity: int, n_slots: int):
        import torch
        dev = recv_counts.device
        ws = torch.zeros(mx.moe_ep_regroup_workspace_size(epr, ep), dtype=torch.uint8, device=dev)
        local_counts = torch.empty(epr, dtype=torch.int32, device=dev)
        local_offsets = torch.empty(epr + 1, dtype=torch.int32, device=dev)
        row_pos = torch.empty(max(n_slots, 1), dtype=torch.int32, device=dev)
        pos_row = torch.empty(max(n_slots, 1), dtype=torch.int32, device=dev)
        mx.moe_ep_regroup(epr, ep, recv_counts, capacity, n_slots, local_counts, local_offsets, row_pos, pos_row, ws)
        self.regroup_ws = ws
        return local_offsets, row_pos, pos_row

    def experts(self, recv_rows, local_offsets, row_pos, pos_row, local_bank, epr: int, n_slots: int):
        import torch
        dm = mx.dims(self.d, self.d_ff, epr, 1, self.act)
        out = torch.empty(max(n_slots, 1), self.d, dtype=torch.float16, device=recv_rows.device)
        if n_slots > 0:
            ws = mx.workspace(dm, n_slots, 0, recv_rows.device)
            mx.moe_ep_experts_forward(dm, n_slots, recv_rows, local_offsets, row_pos, pos_row, mx.weights(local_bank),
                                      out, ws)
            self.experts_ws = ws
        return out[:n_slots]

    def combine(self, back_rows, tok_slot, n_slots: int, topk_weight, out_is_fp32: bool = False):
        import torch
        n = topk_weight.shape[0]
        out = torch.empty(n, self.d, dtype=torch.float32 if out_is_fp32 else torch.bfloat16,
                          device=topk_weight.device)
        if n_slots == 0:
            back_rows = torch.zeros(1, self.d, dtype=torch.float16, device=topk_weight.device)
        mx.moe_ep_combine(self.dims(), n, back_rows, tok_slot, max(n_slots, 1), topk_weight, out, out_is_fp32)
        return out

    def errors(self) -> int:
        """First device-detected error of the last plan / regroup / expert pass (MOE_OK if none)."""
        for ws in (getattr(self, "plan_ws", None), getattr(self, "regroup_ws", None),
                   getattr(self, "experts_ws", None)):
            if ws is not None:
                st = mx.moe_get_error(ws)
                if st != mx.MOE_OK:
                    return st
        return mx.MOE_OK


# ------------------------------------------------------------------ the steps

def dispatch(ops, x, topk_ids, ep: int, capacity: int) -> Dispatch:
    """Steps 1-2: the rank's plan and its send rows (slot order)."""
    n, k = topk_ids.shape
    counts, send_counts, tok_slot = ops.plan(topk_ids, ep, capacity)
    n_slots = ep * capacity if capacity else n * k
    rows = ops.gather(x, tok_slot, n_slots)
    return Dispatch(n, k, counts, send_counts, tok_slot, n_slots, rows)


def expert_pass(ops, recv_counts, recv_rows, local_bank, epr: int, ep: int, capacity: int):
    """Steps 4-5 on the receiving rank: regroup by local expert, run the experts,
    outputs in received slot order."""
    n_slots = recv_rows.shape[0]
    local_offsets, row_pos, pos_row = ops.regroup(recv_counts, epr, ep, capacity, n_slots)
    return ops.experts(recv_rows, local_offsets, row_pos, pos_row, local_bank, epr, n_slots)


def combine(ops, disp: Dispatch, back_rows, topk_weight, out_is_fp32: bool = False):
    """Step 7: each token's k returned rows, weighted and summed in slot order."""
    return ops.combine(back_rows, disp.tok_slot, disp.n_slots, topk_weight, out_is_fp32)


# ------------------------------------------------------------------ the exchanges

def moe_infer_ep(x, topk_ids, topk_weight, local_bank, num_experts: int, group=None, capacity: int = 0,
                 ops: Optional[Any] = None, out_is_fp32: bool = False):
    """This rank's routed sum for its tokens x [n, d], with the experts spread over the
    ranks of `group` (local_bank: this rank's E / ep experts, in global order).
    Every rank of the group calls it (collectively)."""
    import torch
    import torch.distributed as dist

    ep = dist.get_world_size(group)
    if num_experts % ep:
        raise ValueError("the expert count must be a multiple of the group size")
    epr = num_experts // ep
    if ops is None:
        ops = DeviceOps(x.shape[1], mx.bank_sizes(local_bank)[1], num_experts, topk_ids.shape[1])
    disp = dispatch(ops, x, topk_ids, ep, capacity)
    # step 3: the counts (equal splits of E / ep), then the rows
    recv_counts = torch.empty_like(disp.counts)
    dist.all_to_all_single(recv_counts, disp.counts, group=group)
    if capacity:
        in_splits = out_splits = [capacity] * ep
    else:
        in_splits = [int(v) for v in disp.send_counts.cpu().tolist()]
        out_splits = [int(v) for v in recv_counts.view(ep, epr).sum(dim=1).cpu().tolist()]
    n_send, n_recv = sum(in_splits), sum(out_splits)
    recv_rows = disp.send_rows.new_empty((n_recv,) + tuple(disp.send_rows.shape[1:]))
    dist.all_to_all_single(recv_rows, disp.send_rows[:n_send].contiguous(), out_splits, in_splits, group=group)
    out_rows = expert_pass(ops, recv_counts, recv_rows, local_bank, epr, ep, capacity)
    # step 6: the outputs back to their send slots
    back = out_rows.new_empty((disp.n_slots,) + tuple(out_rows.shape[1:]))
    dist.all_to_all_single(back[:n_send], out_rows.contiguous(), in_splits, out_splits, group=group)
    return combine(ops, disp, back, topk_weight, out_is_fp32)


def shard_bank(bank, rank: int, ep: int):
    """Experts [rank * E/ep, (rank + 1) * E/ep) of a row-major bank (views, no copy)."""
    E = bank.w_gate.shape[0]
    epr = E // ep
    sl = slice(rank * epr, (rank + 1) * epr)
    return type(bank)(*(getattr(bank, nm)[sl] for nm in ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")))
