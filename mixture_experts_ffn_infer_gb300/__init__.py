"""GB300 routed-expert forward of a Kimi K2 MoE block.

A thin ctypes binding over ``libmoe_ffn.so`` (declared in ``include/moe_ffn.h``).
The functions carry the C names and only marshal arguments: torch tensors are
passed by device pointer together with the current CUDA stream; every step of
the computation runs in the library's sm_103a kernels.  There is no fallback:
if the library is missing or cannot load, every call raises.

PyTorch supplies device memory and streams.  Convenience helpers
(``workspace``, ``infer``, ``layer_forward``, ``permute``) allocate outputs with
torch and then call the same entry points.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_ffn.so")

MOE_TRACE_MAX = 16

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_ROUTING", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_RANGE", 7: "MOE_ERR_CUDA"}
MOE_OK = 0


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


class moe_dims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("act_scheme", ctypes.c_int32)]


MOE_ACT_EXACT = 0          # activations carried exactly as e4m3 split terms
MOE_ACT_FP8_DYNAMIC = 1    # per-128-feature e4m3 activations, scale amax / 448


MOE_LAYOUT_ROW_MAJOR = 0
MOE_LAYOUT_TILED = 1


class moe_weights(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
                ("layout", ctypes.c_int32)]


class moe_trace(ctypes.Structure):
    _fields_ = [("events", ctypes.c_void_p * MOE_TRACE_MAX), ("n_events", ctypes.c_int32),
                ("n_recorded", ctypes.c_int32), ("labels", ctypes.c_char_p * MOE_TRACE_MAX),
                ("gemms_only", ctypes.c_int32), ("n_launched", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()

_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(moe_dims), ctypes.c_int64, ctypes.c_int32]),
    "moe_tiled_bytes": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "moe_permute_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(moe_dims), ctypes.c_int64]),
    "moe_pack_weights": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(moe_weights),
                                         ctypes.POINTER(moe_weights), ctypes.c_void_p]),
    "moe_permute": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64] + [ctypes.c_void_p] * 5
                    + [ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_experts_forward": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64] + [ctypes.c_void_p] * 4
                            + [ctypes.POINTER(moe_weights), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                               ctypes.c_void_p]),
    "moe_combine": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64] + [ctypes.c_void_p] * 4
                    + [ctypes.c_int32, ctypes.c_void_p]),
    "moe_infer": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64] + [ctypes.c_void_p] * 3
                  + [ctypes.POINTER(moe_weights), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                     ctypes.c_size_t, ctypes.c_void_p, ctypes.POINTER(moe_trace)]),
    "moe_layer_forward": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.POINTER(moe_weights), ctypes.POINTER(moe_weights), ctypes.c_int32,
                                         ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_void_p, ctypes.POINTER(moe_trace)]),
    "moe_mlp_forward": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64, ctypes.c_void_p,
                                       ctypes.POINTER(moe_weights), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                       ctypes.c_size_t, ctypes.c_void_p]),
    "moe_infer_static": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64] + [ctypes.c_void_p] * 3
                         + [ctypes.POINTER(moe_weights), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "moe_ep_plan_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(moe_dims), ctypes.c_int64]),
    "moe_ep_dispatch_plan": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int32, ctypes.c_int64]
                             + [ctypes.c_void_p] * 4 + [ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                                                        ctypes.c_void_p]),
    "moe_ep_gather": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_ep_regroup_workspace_size": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32]),
    "moe_ep_regroup": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_int64] + [ctypes.c_void_p] * 5 + [ctypes.c_size_t, ctypes.c_void_p]),
    "moe_ep_experts_forward": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64] + [ctypes.c_void_p] * 4
                               + [ctypes.POINTER(moe_weights), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                  ctypes.c_void_p]),
    "moe_ep_combine": (ctypes.c_int, [ctypes.POINTER(moe_dims), ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                      ctypes.c_void_p]),
    "moe_check_bounded_wait": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "moe_get_error": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
}

MOE_STATIC_SCRATCH_BYTES = 8 << 20


def load_library(path: Optional[str] = None):
    """Load the CUDA library (raises if it is absent: there is no other implementation)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing; build it with `python -m mixture_experts_ffn_infer_gb300.build`")
            L = ctypes.CDLL(p)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


# ---------------------------------------------------------------- marshalling helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def dims(d: int, d_ff: int, num_experts: int, top_k: int, act_scheme: int = MOE_ACT_EXACT) -> moe_dims:
    return moe_dims(d, d_ff, num_experts, top_k, act_scheme)


def weights(bank) -> moe_weights:
    """moe_weights from an object with w_gate/w_up/w_down/s_gate/s_up/s_down device tensors
    (and an optional ``layout`` attribute, default row-major)."""
    return moe_weights(*((t.data_ptr() if t is not None else None) for t in (bank.w_gate, bank.w_up, bank.w_down,
                                                                              bank.s_gate, bank.s_up, bank.s_down)),
                       int(getattr(bank, "layout", MOE_LAYOUT_ROW_MAJOR)))


# ---------------------------------------------------------------- C entry points (same names)

def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


def moe_workspace_size(dm: moe_dims, n_tokens: int, d_ff_shared: int = 0) -> int:
    return load_library().moe_workspace_size(ctypes.byref(dm), n_tokens, d_ff_shared)


def moe_permute_workspace_size(dm: moe_dims, n_tokens: int) -> int:
    return load_library().moe_permute_workspace_size(ctypes.byref(dm), n_tokens)


def moe_tiled_bytes(which: int, num_experts: int, d: int, d_ff: int) -> int:
    return load_library().moe_tiled_bytes(which, num_experts, d, d_ff)


def moe_pack_weights(num_experts, d, d_ff, src: moe_weights, dst: moe_weights, stream=None):
    st = load_library().moe_pack_weights(num_experts, d, d_ff, ctypes.byref(src), ctypes.byref(dst),
                                         _stream(stream))
    _check(st, "moe_pack_weights")


def moe_permute(dm, n_tokens, topk_ids, tokens_per_expert, expert_offsets, sorted_pos, inv_pos, ws,
                validate=False, stream=None):
    st = load_library().moe_permute(ctypes.byref(dm), n_tokens, _ptr(topk_ids), _ptr(tokens_per_expert),
                                    _ptr(expert_offsets), _ptr(sorted_pos), _ptr(inv_pos), int(bool(validate)),
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "moe_permute")


def moe_experts_forward(dm, n_tokens, x, topk_weight, expert_offsets, sorted_pos, w: moe_weights, rows, ws,
                        stream=None):
    st = load_library().moe_experts_forward(ctypes.byref(dm), n_tokens, _ptr(x), _ptr(topk_weight),
                                            _ptr(expert_offsets), _ptr(sorted_pos), ctypes.byref(w), _ptr(rows),
                                            _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "moe_experts_forward")


def moe_combine(dm, n_tokens, rows, shared, residual, out, out_is_fp32=False, stream=None):
    st = load_library().moe_combine(ctypes.byref(dm), n_tokens, _ptr(rows), _ptr(shared), _ptr(residual), _ptr(out),
                                    int(bool(out_is_fp32)), _stream(stream))
    _check(st, "moe_combine")


def moe_infer(dm, n_tokens, x, topk_ids, topk_weight, w: moe_weights, out, ws, out_is_fp32=False, stream=None,
              trace: Optional[moe_trace] = None):
    st = load_library().moe_infer(ctypes.byref(dm), n_tokens, _ptr(x), _ptr(topk_ids), _ptr(topk_weight),
                                  ctypes.byref(w), _ptr(out), int(bool(out_is_fp32)), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream),
                                  ctypes.byref(trace) if trace is not None else None)
    _check(st, "moe_infer")


def moe_mlp_forward(dm, n_tokens, x, w: moe_weights, out, ws, out_is_fp32=False, stream=None):
    st = load_library().moe_mlp_forward(ctypes.byref(dm), n_tokens, _ptr(x), ctypes.byref(w), _ptr(out),
                                        int(bool(out_is_fp32)), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream))
    _check(st, "moe_mlp_forward")


def moe_layer_forward(dm, n_tokens, hidden, gain, eps, topk_ids, topk_weight, routed: moe_weights,
                      shared: Optional[moe_weights], d_ff_shared, out, ws, out_is_fp32=False, stream=None,
                      trace: Optional[moe_trace] = None):
    st = load_library().moe_layer_forward(ctypes.byref(dm), n_tokens, _ptr(hidden), _ptr(gain), float(eps),
                                          _ptr(topk_ids), _ptr(topk_weight), ctypes.byref(routed),
                                          ctypes.byref(shared) if shared is not None else None, int(d_ff_shared),
                                          _ptr(out), int(bool(out_is_fp32)), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(stream),
                                          ctypes.byref(trace) if trace is not None else None)
    _check(st, "moe_layer_forward")


def moe_infer_static(dm, n_tokens, x, topk_ids, topk_weight, w: moe_weights, out, out_is_fp32=False, stream=None):
    """moe_infer on the library's built-in scratch (no workspace argument)."""
    st = load_library().moe_infer_static(ctypes.byref(dm), n_tokens, _ptr(x), _ptr(topk_ids), _ptr(topk_weight),
                                         ctypes.byref(w), _ptr(out), int(bool(out_is_fp32)), _stream(stream))
    _check(st, "moe_infer_static")


def moe_ep_plan_workspace_size(dm: moe_dims, n_tokens: int) -> int:
    return load_library().moe_ep_plan_workspace_size(ctypes.byref(dm), n_tokens)


def moe_ep_dispatch_plan(dm, ep_size, n_tokens, topk_ids, tokens_per_expert, send_counts, tok_slot, capacity, ws,
                         stream=None):
    st = load_library().moe_ep_dispatch_plan(ctypes.byref(dm), ep_size, n_tokens, _ptr(topk_ids),
                                             _ptr(tokens_per_expert), _ptr(send_counts), _ptr(tok_slot), capacity,
                                             _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "moe_ep_dispatch_plan")


def moe_ep_gather(dm, n_tokens, x, tok_slot, n_slots, send_rows, stream=None):
    st = load_library().moe_ep_gather(ctypes.byref(dm), n_tokens, _ptr(x), _ptr(tok_slot), n_slots, _ptr(send_rows),
                                      _stream(stream))
    _check(st, "moe_ep_gather")


def moe_ep_regroup_workspace_size(experts_per_rank: int, ep_size: int) -> int:
    return load_library().moe_ep_regroup_workspace_size(experts_per_rank, ep_size)


def moe_ep_regroup(experts_per_rank, ep_size, recv_counts, capacity, n_slots, local_counts, local_offsets, row_pos,
                   pos_row, ws, stream=None):
    st = load_library().moe_ep_regroup(experts_per_rank, ep_size, _ptr(recv_counts), capacity, n_slots,
                                       _ptr(local_counts), _ptr(local_offsets), _ptr(row_pos), _ptr(pos_row),
                                       _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "moe_ep_regroup")


def moe_ep_experts_forward(dm, n_slots, recv_rows, local_offsets, row_pos, pos_row, w: moe_weights, out_rows, ws,
                           stream=None):
    st = load_library().moe_ep_experts_forward(ctypes.byref(dm), n_slots, _ptr(recv_rows), _ptr(local_offsets),
                                               _ptr(row_pos), _ptr(pos_row), ctypes.byref(w), _ptr(out_rows),
                                               _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "moe_ep_experts_forward")


def moe_ep_combine(dm, n_tokens, back_rows, tok_slot, n_slots, topk_weight, out, out_is_fp32=False, stream=None):
    st = load_library().moe_ep_combine(ctypes.byref(dm), n_tokens, _ptr(back_rows), _ptr(tok_slot), n_slots,
                                       _ptr(topk_weight), _ptr(out), int(bool(out_is_fp32)), _stream(stream))
    _check(st, "moe_ep_combine")


def moe_check_bounded_wait(ws, stream=None):
    st = load_library().moe_check_bounded_wait(_ptr(ws), _stream(stream))
    _check(st, "moe_check_bounded_wait")


def moe_get_error(ws, stream=None) -> int:
    return load_library().moe_get_error(_ptr(ws), _stream(stream))


# ---------------------------------------------------------------- allocating conveniences

class TiledBank:
    """A bank whose e4m3 codes are in the tiled streaming layout: w_gate holds gate and up
    interleaved, w_up is None, w_down holds down row blocks in pairs (flat uint8 tensors)."""

    layout = MOE_LAYOUT_TILED

    def __init__(self, w_gate, w_down, s_gate, s_up, s_down, num_experts, d_ff, d):
        self.w_gate, self.w_up, self.w_down = w_gate, None, w_down
        self.s_gate, self.s_up, self.s_down = s_gate, s_up, s_down
        self.num_experts, self.d_ff, self.d = num_experts, d_ff, d


def bank_sizes(bank):
    """(num_experts, d_ff, d) of a row-major or tiled bank."""
    if isinstance(bank, TiledBank):
        return bank.num_experts, bank.d_ff, bank.d
    return tuple(bank.w_gate.shape)


def pack_bank(bank, stream=None) -> TiledBank:
    """Tiled copy of a row-major bank's codes (scales shared with the source)."""
    import torch
    E, d_ff, d = bank.w_gate.shape
    dev = bank.w_gate.device
    gu = torch.empty(moe_tiled_bytes(0, E, d, d_ff), dtype=torch.uint8, device=dev)
    dn = torch.empty(moe_tiled_bytes(2, E, d, d_ff), dtype=torch.uint8, device=dev)
    out = TiledBank(gu, dn, bank.s_gate, bank.s_up, bank.s_down, E, d_ff, d)
    moe_pack_weights(E, d, d_ff, weights(bank), weights(out), stream)
    return out


def workspace(dm: moe_dims, n_tokens: int, d_ff_shared: int = 0, device="cuda"):
    import torch
    nbytes = moe_workspace_size(dm, n_tokens, d_ff_shared)
    if nbytes == 0:
        raise MoeError(2, "moe_workspace_size")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def permute(topk_ids, num_experts: int, ws=None, validate=False, stream=None):
    """-> (tokens_per_expert, expert_offsets, sorted_pos, inv_pos) int32 device tensors."""
    import torch
    n, k = topk_ids.shape
    dm = moe_dims(128, 128, num_experts, k)
    if ws is None:
        nbytes = load_library().moe_permute_workspace_size(ctypes.byref(dm), n)
        if nbytes == 0:
            raise MoeError(2, "moe_permute_workspace_size")
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=topk_ids.device)
    dev = topk_ids.device
    counts = torch.empty(num_experts, dtype=torch.int32, device=dev)
    offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(max(n * k, 1), dtype=torch.int32, device=dev)
    ip = torch.empty(max(n * k, 1), dtype=torch.int32, device=dev)
    moe_permute(dm, n, topk_ids, counts, offsets, sp, ip, ws, validate=validate, stream=stream)
    return counts, offsets, sp[: n * k], ip[: n * k]


def infer(x, topk_ids, topk_weight, bank, ws=None, out_is_fp32=False, stream=None, act_scheme=MOE_ACT_EXACT):
    import torch
    n, d = x.shape
    E, d_ff, _ = bank_sizes(bank)
    dm = moe_dims(d, d_ff, E, topk_ids.shape[1], act_scheme)
    if ws is None:
        ws = workspace(dm, n, 0, x.device)
    out = torch.empty(n, d, dtype=torch.float32 if out_is_fp32 else torch.bfloat16, device=x.device)
    moe_infer(dm, n, x, topk_ids, topk_weight, weights(bank), out, ws, out_is_fp32, stream)
    return out


def mlp_forward(x, bank, ws=None, out_is_fp32=False, stream=None, act_scheme=MOE_ACT_EXACT):
    """One SwiGLU MLP (a bank with E = 1) on every row of x."""
    import torch
    n, d = x.shape
    E, d_ff, _ = bank_sizes(bank)
    dm = moe_dims(d, d_ff, E, 1, act_scheme)
    if ws is None:
        ws = workspace(dm, n, 0, x.device)
    out = torch.empty(n, d, dtype=torch.float32 if out_is_fp32 else torch.bfloat16, device=x.device)
    moe_mlp_forward(dm, n, x, weights(bank), out, ws, out_is_fp32, stream)
    return out


def layer_forward(hidden, gain, eps, topk_ids, topk_weight, bank, shared=None, ws=None, out_is_fp32=False,
                  stream=None, act_scheme=MOE_ACT_EXACT):
    import torch
    n, d = hidden.shape
    E, d_ff, _ = bank_sizes(bank)
    dm = moe_dims(d, d_ff, E, topk_ids.shape[1], act_scheme)
    dff_sh = bank_sizes(shared)[1] if shared is not None else 0
    if ws is None:
        ws = workspace(dm, n, dff_sh, hidden.device)
    out = torch.empty(n, d, dtype=torch.float32 if out_is_fp32 else torch.bfloat16, device=hidden.device)
    moe_layer_forward(dm, n, hidden, gain, eps, topk_ids, topk_weight, weights(bank),
                      weights(shared) if shared is not None else None, dff_sh, out, ws, out_is_fp32, stream)
    return out
