"""Workload construction shared by the GPU tests (seeded, synthetic).

Small workloads are drawn on the CPU and copied to the GPU, so the oracle and
the library read the same bytes.  The K2-sized routed bank (16.9 GB) is drawn
once per process on the GPU; the oracle copies the experts it needs back."""

import dataclasses

import torch

from mixture_experts_ffn_infer_gb300 import synthetic as syn

_K2_BANK = {}


def k2_bank(seed: int = 1):
    if seed not in _K2_BANK:
        _K2_BANK.clear()
        torch.cuda.empty_cache()
        _K2_BANK[seed] = syn.expert_bank(384, 7168, 2048, seed, "cuda")
    return _K2_BANK[seed]


def bank_to(bank, device):
    return syn.ExpertBank(*(t.to(device) for t in dataclasses.astuple(bank)))


@dataclasses.dataclass
class Case:
    inp: syn.Inputs          # host tensors (bank may live on the GPU)
    x: torch.Tensor
    ids: torch.Tensor
    w: torch.Tensor
    bank: syn.ExpertBank     # on the GPU
    gain: torch.Tensor = None
    shared: syn.ExpertBank = None


def workload(name_or_wl, n_tokens=None, ids=None) -> Case:
    wl = syn.WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    big = wl.d == 7168 and wl.num_experts == 384 and wl.d_ff == 2048
    if big:
        inp = syn.make_inputs(wl, n_tokens=n_tokens, bank=k2_bank(syn.bank_seed_of(wl)), weight_device="cuda")
    else:
        inp = syn.make_inputs(wl, n_tokens=n_tokens)
    if ids is not None:
        inp.topk_ids = ids
    bank = inp.bank if big else bank_to(inp.bank, "cuda")
    shared = bank_to(inp.shared, "cuda") if inp.shared is not None else None
    return Case(inp, inp.x.cuda(), inp.topk_ids.cuda(), inp.topk_weight.cuda(), bank,
                inp.gain.cuda() if inp.gain is not None else None, shared)


def parity_tokens(ids: torch.Tensor, n_min: int = 512, top: int = 3, tile: int = 128, seed: int = 0):
    """Token subset of a K2-sized batch that the oracle computes one by one (at least n_min tokens):

    * one token of every expert that the batch selects (a greedy cover: a token covers its k experts),
      so every expert's slice of both grouped GEMMs is compared;
    * the tokens at the first and the last row of every `tile`-row tile of the `top` most-loaded experts,
      in the sorted order (stable by expert, then flat index t * k + j), so every tile boundary of the
      experts that span several tiles is compared;
    * the first and the last token of the batch;
    * seeded uniform tokens until n_min are picked."""
    ids = ids.cpu().long()
    n, k = ids.shape
    g = torch.Generator().manual_seed(seed)
    pick = {0, n - 1}
    flat = ids.reshape(-1)
    E = int(flat.max()) + 1
    counts = torch.bincount(flat, minlength=E)
    # every touched expert, in a seeded order; a token already picked may cover it
    covered = torch.zeros(E, dtype=torch.bool)
    for t in pick:
        covered[ids[t]] = True
    for e in torch.randperm(E, generator=g).tolist():
        if counts[e] == 0 or covered[e]:
            continue
        toks = (ids == e).any(dim=1).nonzero().flatten()
        t = int(toks[int(torch.randint(toks.numel(), (1,), generator=g))])
        pick.add(t)
        covered[ids[t]] = True
    # first and last row of every tile of the most-loaded experts
    for e in torch.argsort(counts, descending=True, stable=True)[:top].tolist():
        rows = (flat == e).nonzero().flatten()       # ascending flat index = the stable sorted order
        c = rows.numel()
        for r0 in range(0, c, tile):
            for r in (r0, min(r0 + tile - 1, c - 1)):
                pick.add(int(rows[r]) // k)
    rest = [t for t in torch.randperm(n, generator=g).tolist() if t not in pick]
    pick.update(rest[:max(0, n_min - len(pick))])
    return sorted(pick)
