"""Expert-parallel routed-expert forward, restated from the pages (test infrastructure only).

Only the tests and the benchmark's CPU-baseline leg may use this module; the
product path never imports it.

"Input features" page, expert construction: with ep_size ranks, rank r holds
the experts [r * E / ep, (r + 1) * E / ep) (experts_per_rank = E / ep).
"Mixture of experts" page, moe_infer, ep_size > 1 branch, in its order:

  1. every rank counts its (token, slot) entries per expert (tokens_per_expert)
     and sorts the flattened ids (idxs); sorted_tokens = x[idxs // k];
  2. tokens_per_ep_rank = tokens_per_expert summed per owning rank (the rows
     it sends to each rank, input_split_sizes);
  3. an all-to-all of tokens_per_expert gives each rank, per source rank, the
     counts of its own experts (tokens_per_expert_group, source-major);
     output_splits = those counts summed per source;
  4. an all-to-all of sorted_tokens gives each rank the rows routed to its
     experts, source after source (gathered_tokens);
  5. each received row is labelled with its local expert (runs of
     tokens_per_expert_group, label = run index % experts_per_rank) and the
     rows are put in label order (gatherd_idxs = argsort of the labels);
  6. each local expert runs on its contiguous slice;
  7. the outputs go back to received order (new_x[gatherd_idxs] = outs), a
     reverse all-to-all returns them to their source ranks, they go back to
     flat (token, slot) order (new_x[idxs] = outs) and each token sums its k
     rows weighted by topk_weight.

The all-to-alls are written out as indexing over all ranks' arrays.  Readings
where the pages are silent: both argsorts are taken stable (ties by position;
the output does not depend on it), ids are valid (0 <= id < E, distinct per
token) and E is a multiple of ep.  Arithmetic of each expert and of the final
weighted sum is the oracle's own (`oracle.expert_forward`, fp64, slots in
ascending order), so the result equals `oracle.moe_infer` bit for bit.
"""

from __future__ import annotations

import numpy as np

from . import _np, expert_forward


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> their exact fp64 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ep_plan(topk_ids_per_rank, num_experts: int, ep_size: int):
    """Bookkeeping of steps 1-5 for every rank.  Returns one dict per rank with
    tokens_per_expert [E], idxs [n k], input_split_sizes [ep], tokens_per_expert_group [ep * E/ep]
    (source-major), output_splits [ep], gatherd_idxs [received rows] and
    tokens_per_expert_post_gather [E/ep], all int64 numpy arrays."""
    assert num_experts % ep_size == 0
    epr = num_experts // ep_size
    ids = [_np(t, np.int32).astype(np.int64) for t in topk_ids_per_rank]
    plans = []
    for r in range(ep_size):
        flat = ids[r].reshape(-1)
        tpe = np.bincount(flat, minlength=num_experts)[:num_experts]
        plans.append({
            "tokens_per_expert": tpe,
            "idxs": np.argsort(flat, kind="stable"),
            "input_split_sizes": tpe.reshape(ep_size, epr).sum(axis=1),
        })
    for r in range(ep_size):
        # all-to-all of the counts: piece r of every source's tokens_per_expert
        group = np.concatenate([plans[s]["tokens_per_expert"][r * epr:(r + 1) * epr] for s in range(ep_size)])
        labels = np.repeat(np.arange(group.size) % epr, group)
        plans[r]["tokens_per_expert_group"] = group
        plans[r]["output_splits"] = group.reshape(ep_size, epr).sum(axis=1)
        plans[r]["gatherd_idxs"] = np.argsort(labels, kind="stable")
        plans[r]["tokens_per_expert_post_gather"] = group.reshape(ep_size, epr).sum(axis=0)
    return plans


def _split(a: np.ndarray, sizes):
    out, s = [], 0
    for n in sizes:
        out.append(a[s:s + int(n)])
        s += int(n)
    return out


def moe_infer_ep(x_per_rank, topk_ids_per_rank, topk_weight_per_rank, bank, ep_size: int, fp8_act=False):
    """The whole multi-rank forward (steps 1-7) simulated in one process: rank r's routed
    sum for its tokens, fp64 [n_r, d] per rank.  bank holds all E experts (rank r uses
    experts r * E/ep ..)."""
    E = bank.w_gate.shape[0]
    epr = E // ep_size
    plans = ep_plan(topk_ids_per_rank, E, ep_size)
    xs = [_bf16_to_f64(_np(x, np.uint16)) for x in x_per_rank]
    ks = [_np(t, np.int32).shape[1] for t in topk_ids_per_rank]
    sorted_tokens = [xs[r][plans[r]["idxs"] // ks[r]] for r in range(ep_size)]
    # step 4: rank r receives, from each source s, piece r of s's sorted rows
    pieces = [_split(sorted_tokens[s], plans[s]["input_split_sizes"]) for s in range(ep_size)]
    back = [None] * ep_size
    for r in range(ep_size):
        d = xs[r].shape[1]
        gathered = np.concatenate([pieces[s][r] for s in range(ep_size)]) if ep_size else np.zeros((0, d))
        gi = plans[r]["gatherd_idxs"]
        local_sorted = gathered[gi]
        outs = []
        start = 0
        for i, cnt in enumerate(plans[r]["tokens_per_expert_post_gather"]):
            if cnt == 0:
                continue
            e = i + r * epr
            W = [getattr(bank, nm)[e] for nm in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down")]
            outs.append(expert_forward(local_sorted[start:start + cnt], *W, fp8_act=fp8_act))
            start += cnt
        outs = np.concatenate(outs) if outs else np.zeros((0, d))
        new_x = np.empty_like(outs)
        new_x[gi] = outs
        back[r] = _split(new_x, plans[r]["output_splits"])
    y = []
    for s in range(ep_size):
        # reverse all-to-all: source s gets back its piece from every rank, in rank order
        returned = np.concatenate([back[r][s] for r in range(ep_size)])
        new_x = np.empty_like(returned)
        new_x[plans[s]["idxs"]] = returned
        w = _np(topk_weight_per_rank[s], np.float32).astype(np.float64)
        n, k = w.shape
        rows = new_x.reshape(n, k, -1)
        acc = np.zeros((n, rows.shape[2]))
        for j in range(k):  # ascending slot order, as the single-rank oracle sums
            acc += w[:, j:j + 1] * rows[:, j]
        y.append(acc)
    return y
