"""Seeded synthetic inputs shaped like a Kimi K2 MoE block.

This module only draws inputs. It holds none of the arithmetic of the
routed-expert forward: no dequantisation, no SwiGLU, no sorting, no combine.
Both the CPU oracle and the CUDA library consume the exact bytes produced
here, so a parity test compares the two on identical inputs.

Shapes follow the Kimi K2 pages ("Mixture of experts" page, parameter table:
gate/up projections ``[2048, 7168]``, down ``[7168, 2048]``; 384 routed
experts, 8 selected per position; "Input features" page: ``x`` is
``[B, T, 7168]``).  Weights are stored the way the model's quantisation
config says ("Input features" page, FP8 quantisation config): e4m3 codes
with one fp32 scale per 128 x 128 block.

Recipe (seeded, reproducible):

* ``x`` ~ N(0, 1), rounded to bf16.
* each projection ~ N(0, 0.02) in fp32, then per 128 x 128 block
  ``s = amax / 448`` (``s = 1`` for an all-zero block) and
  ``q = e4m3(clamp(w / s, -448, 448))`` with round-to-nearest-even
  (``torch.float8_e4m3fn``).
* uniform routing: per token the ``k`` largest of ``E`` U(0,1) keys, so the
  ``k`` experts are distinct and uniform; order within a token = key order.
* skewed routing: popularity ``p_e ~ rank(e)^-s`` over a seeded random
  permutation of the experts, ``k`` drawn without replacement by
  Gumbel-top-k (keys ``log p_e + Gumbel``).
* ``topk_weight`` = softmax of N(0, 1) logits over the ``k`` picks (fp32).
* full block: residual ``h`` ~ N(0, 1) bf16, RMSNorm gain ``1 + N(0, 0.1)``
  in bf16, eps = 1e-6, one shared SwiGLU expert from the same weight recipe.

Host-side draws (x, routing, residual, gain) use a CPU ``torch.Generator``
seeded with ``seed``; the expert bank uses a generator on the device it is
built on, seeded with ``seed + 7919``.  The same seed therefore gives the
same weights only on the same kind of device; every consumer of a given
workload reads the same tensors, wherever they were drawn.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import torch

E4M3_MAX = 448.0
BLOCK = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_tokens: int
    d: int
    d_ff: int
    num_experts: int
    top_k: int
    routing: str = "uniform"      # "uniform" | "zipf"
    zipf_s: float = 1.2
    full_block: bool = False      # RMSNorm + shared expert + residual
    d_ff_shared: int = 0
    seed: int = 0
    bank_seed: Optional[int] = None   # seed of the expert bank (default: seed)


# The five workloads of the routed-expert forward, named by what they are.
WORKLOADS = {
    "tiny": Workload("tiny", 128, 1024, 256, 16, 4, seed=0),
    "k2_decode": Workload("k2_decode", 16, 7168, 2048, 384, 8, seed=1, bank_seed=1),
    "k2_prefill": Workload("k2_prefill", 4096, 7168, 2048, 384, 8, seed=2, bank_seed=1),
    "k2_skewed": Workload("k2_skewed", 8192, 7168, 2048, 384, 8,
                          routing="zipf", zipf_s=1.2, seed=3, bank_seed=1),
    "k2_block": Workload("k2_block", 32768, 7168, 2048, 384, 8,
                         full_block=True, d_ff_shared=2048, seed=4, bank_seed=1),
}
# The four K2-sized workloads share one routed bank (bank_seed 1, 16.9 GB of
# e4m3 codes) so that a process can keep a single copy resident.


def quantize_blockwise(w: torch.Tensor):
    """fp32 ``[R, C]`` -> (e4m3 codes as uint8 ``[R, C]``, fp32 scales ``[R/128, C/128]``)."""
    R, C = w.shape
    assert R % BLOCK == 0 and C % BLOCK == 0
    wb = w.reshape(R // BLOCK, BLOCK, C // BLOCK, BLOCK)
    amax = wb.abs().amax(dim=(1, 3))
    s = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (wb / s[:, None, :, None]).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.reshape(R, C).view(torch.uint8), s.contiguous()


@dataclasses.dataclass
class ExpertBank:
    """Stacked FP8 expert weights: gate/up ``[E, d_ff, d]``, down ``[E, d, d_ff]`` (uint8 e4m3 codes),
    scales gate/up ``[E, d_ff/128, d/128]``, down ``[E, d/128, d_ff/128]`` (fp32)."""
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor
    s_gate: torch.Tensor
    s_up: torch.Tensor
    s_down: torch.Tensor

    @property
    def num_experts(self) -> int:
        return self.w_gate.shape[0]

    def to(self, device) -> "ExpertBank":
        return ExpertBank(*(t.to(device) for t in dataclasses.astuple(self)))

    def subset(self, experts) -> "ExpertBank":
        idx = torch.as_tensor(list(experts), dtype=torch.long, device=self.w_gate.device)
        return ExpertBank(*(t.index_select(0, idx) for t in dataclasses.astuple(self)))


def expert_bank(num_experts: int, d: int, d_ff: int, seed: int, device="cpu",
                std: float = 0.02) -> ExpertBank:
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(seed + 7919)
    u8 = dict(dtype=torch.uint8, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    bank = ExpertBank(
        torch.empty(num_experts, d_ff, d, **u8), torch.empty(num_experts, d_ff, d, **u8),
        torch.empty(num_experts, d, d_ff, **u8),
        torch.empty(num_experts, d_ff // BLOCK, d // BLOCK, **f32),
        torch.empty(num_experts, d_ff // BLOCK, d // BLOCK, **f32),
        torch.empty(num_experts, d // BLOCK, d_ff // BLOCK, **f32))
    for e in range(num_experts):
        for q, s, shape in ((bank.w_gate, bank.s_gate, (d_ff, d)),
                            (bank.w_up, bank.s_up, (d_ff, d)),
                            (bank.w_down, bank.s_down, (d, d_ff))):
            w = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
            q[e], s[e] = quantize_blockwise(w)
    return bank


def routing_uniform(n: int, num_experts: int, k: int, g: torch.Generator):
    keys = torch.rand(n, num_experts, generator=g)
    return keys.topk(k, dim=1).indices.to(torch.int32).contiguous()


def routing_zipf(n: int, num_experts: int, k: int, s: float, g: torch.Generator):
    perm = torch.randperm(num_experts, generator=g)
    rank = torch.empty(num_experts)
    rank[perm] = torch.arange(1, num_experts + 1, dtype=torch.float32)
    logp = -s * torch.log(rank)
    u = torch.rand(n, num_experts, generator=g).clamp_min(1e-20)
    gumbel = -torch.log(-torch.log(u))
    return (logp[None, :] + gumbel).topk(k, dim=1).indices.to(torch.int32).contiguous()


def routing_subset(n: int, experts, k: int, g: torch.Generator):
    """Uniform distinct routing restricted to the listed experts (the rest stay empty)."""
    experts = torch.as_tensor(list(experts), dtype=torch.int32)
    keys = torch.rand(n, experts.numel(), generator=g)
    return experts[keys.topk(k, dim=1).indices].contiguous()


def router_weights(n: int, k: int, g: torch.Generator):
    return torch.softmax(torch.randn(n, k, generator=g), dim=1).to(torch.float32).contiguous()


@dataclasses.dataclass
class Inputs:
    wl: Workload
    x: torch.Tensor                  # [N, d] bf16 (normalised features, or the residual for a full block)
    topk_ids: torch.Tensor           # [N, k] int32
    topk_weight: torch.Tensor        # [N, k] fp32
    bank: ExpertBank
    gain: Optional[torch.Tensor] = None      # [d] bf16 (full block)
    eps: float = 1e-6
    shared: Optional[ExpertBank] = None      # E = 1 (full block)


def make_host_inputs(wl: Workload, n_tokens: Optional[int] = None):
    """The host-side draws of a workload: (x bf16 [N, d], topk_ids int32 [N, k], topk_weight fp32 [N, k],
    gain bf16 [d] or None)."""
    n = wl.n_tokens if n_tokens is None else n_tokens
    g = torch.Generator().manual_seed(wl.seed)
    x = torch.randn(n, wl.d, generator=g).to(torch.bfloat16)
    if wl.routing == "uniform":
        ids = routing_uniform(n, wl.num_experts, wl.top_k, g)
    elif wl.routing == "zipf":
        ids = routing_zipf(n, wl.num_experts, wl.top_k, wl.zipf_s, g)
    else:
        raise ValueError(wl.routing)
    w = router_weights(n, wl.top_k, g)
    gain = None
    if wl.full_block:
        gain = (1.0 + 0.1 * torch.randn(wl.d, generator=g)).to(torch.bfloat16)
    return x, ids, w, gain


def make_inputs(wl: Workload, weight_device="cpu", n_tokens: Optional[int] = None,
                bank: Optional[ExpertBank] = None) -> Inputs:
    """Draw one workload.  ``n_tokens`` overrides N (keeps every other draw's recipe); ``bank``
    reuses an expert bank already drawn for the same ``bank_seed``."""
    x, ids, w, gain = make_host_inputs(wl, n_tokens)
    bank = bank if bank is not None else expert_bank(wl.num_experts, wl.d, wl.d_ff, bank_seed_of(wl),
                                                     weight_device)
    shared = None
    if wl.full_block and wl.d_ff_shared:
        shared = expert_bank(1, wl.d, wl.d_ff_shared, wl.seed + 1_000_003, weight_device)
    return Inputs(wl, x, ids, w, bank, gain, 1e-6, shared)


def bank_seed_of(wl: Workload) -> int:
    return wl.seed if wl.bank_seed is None else wl.bank_seed


def bank_bytes(d: int, d_ff: int) -> int:
    """Bytes of one expert's FP8 weights plus fp32 block scales."""
    return 3 * d * d_ff + 3 * (d // BLOCK) * (d_ff // BLOCK) * 4


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def touched_experts(topk_ids: torch.Tensor) -> int:
    return int(torch.unique(topk_ids).numel())


__all__ = ["Workload", "WORKLOADS", "ExpertBank", "Inputs", "make_inputs", "make_host_inputs", "expert_bank",
           "bank_seed_of",
           "quantize_blockwise", "routing_uniform", "routing_zipf", "routing_subset",
           "router_weights", "bank_bytes", "touched_experts", "ceil_div"]
