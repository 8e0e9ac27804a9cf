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


def sample_tokens(ids: torch.Tensor, n_random: int, n_hot: int, seed: int = 0):
    """Token subset for the oracle: n_random uniform tokens, n_hot tokens of the most loaded expert,
    the first and the last token."""
    n = ids.shape[0]
    g = torch.Generator().manual_seed(seed)
    pick = set(torch.randperm(n, generator=g)[:n_random].tolist())
    counts = torch.bincount(ids.reshape(-1).long().cpu(), minlength=int(ids.max()) + 1)
    hot = int(counts.argmax())
    hot_tokens = (ids.cpu() == hot).any(dim=1).nonzero().flatten()
    pick |= set(hot_tokens[torch.randperm(hot_tokens.numel(), generator=g)[:n_hot]].tolist())
    pick |= {0, n - 1}
    return sorted(pick)
