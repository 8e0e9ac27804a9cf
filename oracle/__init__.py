"""CPU oracle of the routed-expert forward (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The product path never does: it runs entirely in
the CUDA library and fails loudly when that library is missing.

``oracle/moe_oracle.c`` holds the arithmetic (fp64, plain loops, one thread per
token); this module only marshals numpy/torch buffers into it with ctypes and
builds it with gcc on first use.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C, no target-specific flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(L):
    """Declare the C signatures on a loaded oracle library."""
    i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    L.oracle_e4m3_value.restype = dbl
    L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    L.oracle_bf16_value.restype = dbl
    L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    L.oracle_silu.restype = dbl
    L.oracle_silu.argtypes = [dbl]
    L.oracle_dequant.restype = dbl
    L.oracle_dequant.argtypes = [vp, vp, i64, i64, i64, i64]
    L.oracle_expert_forward.restype = None
    L.oracle_expert_forward.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, i32]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_fp8_dynamic.restype = None
    L.oracle_fp8_dynamic.argtypes = [i64, vp, vp, vp, vp]
    L.oracle_rmsnorm.restype = None
    L.oracle_rmsnorm.argtypes = [i64, i64, vp, vp, dbl, vp]
    L.oracle_permute.restype = i64
    L.oracle_permute.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp]
    L.oracle_moe_infer.restype = None
    L.oracle_moe_infer.argtypes = [i64, i64, i64, i64, vp, vp, vp] + [vp] * 6 + [vp, i64, vp, i32, i32]
    L.oracle_layer_forward.restype = None
    L.oracle_layer_forward.argtypes = ([i64, i64, i64, i64, vp, vp, dbl, vp, vp] + [vp] * 6
                                       + [vp] * 6 + [i64, vp, i64, vp, i32, i32])
    L.oracle_moe_infer_sorted.restype = None
    L.oracle_moe_infer_sorted.argtypes = [i64, i64, i64, i64, i64, vp, vp, vp] + [vp] * 6 + [vp, i32]
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


# --------------------------------------------------------------------------- helpers

def _np(t, dtype):
    """Host numpy view of a tensor/array with the given numpy dtype (contiguous)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().to("cpu").contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            t = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


class _Bank:
    """Per-expert pointer tables for the C oracle; keeps the host arrays alive."""

    def __init__(self, bank, experts=None):
        E = bank.w_gate.shape[0]
        need = range(E) if experts is None else sorted(set(int(e) for e in experts))
        self.keep = []
        self.tables = []
        for name, dt in (("w_gate", np.uint8), ("s_gate", np.float32), ("w_up", np.uint8),
                         ("s_up", np.float32), ("w_down", np.uint8), ("s_down", np.float32)):
            arr_t = (ctypes.c_void_p * E)()
            full = getattr(bank, name)
            for e in need:
                a = _np(full[e], dt)
                self.keep.append(a)
                arr_t[e] = a.ctypes.data
            self.keep.append(arr_t)
            self.tables.append(arr_t)

    def args(self):
        return [ctypes.cast(t, ctypes.c_void_p) for t in self.tables]


# --------------------------------------------------------------------------- API

def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(code)


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(bits)


def silu(a: float) -> float:
    return lib().oracle_silu(a)


def dequant(q, s):
    """Full dequantised matrix (fp64) of one e4m3 [R, C] matrix with [R/128, C/128] scales."""
    q = _np(q, np.uint8)
    s = _np(s, np.float32)
    R, C = q.shape
    out = np.empty((R, C), np.float64)
    L = lib()
    for r in range(R):
        for c in range(C):
            out[r, c] = L.oracle_dequant(_ptr(q), _ptr(s), R, C, r, c)
    return out


def e4m3_encode(v: float) -> int:
    """Nearest e4m3 code of a float32 value (ties to even, saturating at 448)."""
    return int(lib().oracle_e4m3_encode(float(v)))


def fp8_dynamic(v):
    """Dynamic FP8 quantisation of rows v [..., n] (n a multiple of 128), per group of 128 features.
    Returns (dequantised fp64 values, e4m3 codes uint8, group scales float32 [..., n/128])."""
    v = np.ascontiguousarray(np.asarray(v, np.float64))
    n = v.shape[-1]
    rows = v.reshape(-1, n)
    out = np.empty_like(rows)
    codes = np.empty(rows.shape, np.uint8)
    scales = np.empty((rows.shape[0], n // 128), np.float32)
    L = lib()
    for i in range(rows.shape[0]):
        L.oracle_fp8_dynamic(n, _ptr(rows[i]), _ptr(out[i]), _ptr(codes[i]), _ptr(scales[i]))
    return (out.reshape(v.shape), codes.reshape(v.shape), scales.reshape(v.shape[:-1] + (n // 128,)))


def expert_forward(x, wg, sg, wu, su, wd, sd, fp8_act=False):
    """One SwiGLU expert on fp64 rows x [n, d] -> [n, d] (fp8_act: dynamic FP8 activations)."""
    x = np.ascontiguousarray(np.asarray(x, np.float64))
    n, d = x.shape
    wg, wu, wd = (_np(a, np.uint8) for a in (wg, wu, wd))
    sg, su, sd = (_np(a, np.float32) for a in (sg, su, sd))
    dff = wg.shape[0]
    out = np.empty((n, d), np.float64)
    lib().oracle_expert_forward(n, d, dff, _ptr(x), _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su), _ptr(wd),
                                _ptr(sd), _ptr(out), int(bool(fp8_act)))
    return out


def rmsnorm(h, gain, eps):
    h = _np(h, np.uint16)
    gain = _np(gain, np.uint16)
    n, d = h.shape
    out = np.empty((n, d), np.float64)
    lib().oracle_rmsnorm(n, d, _ptr(h), _ptr(gain), float(eps), _ptr(out))
    return out


def permute(topk_ids, num_experts: int):
    """-> (counts[E], offsets[E+1], sorted_pos[R], inv_pos[R], n_bad) as int32 numpy arrays."""
    ids = _np(topk_ids, np.int32)
    n, k = ids.shape
    R = n * k
    counts = np.empty(num_experts, np.int32)
    offsets = np.empty(num_experts + 1, np.int32)
    sp = np.empty(max(R, 1), np.int32)
    ip = np.empty(max(R, 1), np.int32)
    bad = lib().oracle_permute(n, k, num_experts, _ptr(ids), _ptr(counts), _ptr(offsets), _ptr(sp), _ptr(ip))
    return counts, offsets, sp[:R], ip[:R], int(bad)


def moe_infer(x, topk_ids, topk_weight, bank, tokens=None, threads=None, fp8_act=False):
    """Routed sum for the selected tokens (default: all).  Returns fp64 [len(tokens), d].
    fp8_act: dynamic FP8 activations (per-128-feature e4m3 with scale amax/448)."""
    xb = _np(x, np.uint16)
    ids = _np(topk_ids, np.int32)
    w = _np(topk_weight, np.float32)
    n, d = xb.shape
    k = ids.shape[1]
    E = bank.w_gate.shape[0]
    dff = bank.w_gate.shape[1]
    tok = np.arange(n, dtype=np.int64) if tokens is None else np.ascontiguousarray(np.asarray(tokens, np.int64))
    used = np.unique(ids[tok].reshape(-1))
    used = used[(used >= 0) & (used < E)]
    b = _Bank(bank, used)
    y = np.empty((tok.size, d), np.float64)
    lib().oracle_moe_infer(d, dff, k, E, _ptr(xb), _ptr(ids), _ptr(w), *b.args(), _ptr(tok), tok.size, _ptr(y),
                           threads or default_threads(), int(bool(fp8_act)))
    return y


def layer_forward(hidden, gain, eps, topk_ids, topk_weight, bank, shared=None, tokens=None, threads=None,
                  fp8_act=False):
    """Full block for the selected tokens: h + routed(RMSNorm(h)) + shared(RMSNorm(h)).  fp64."""
    hb = _np(hidden, np.uint16)
    gb = _np(gain, np.uint16)
    ids = _np(topk_ids, np.int32)
    w = _np(topk_weight, np.float32)
    n, d = hb.shape
    k = ids.shape[1]
    E = bank.w_gate.shape[0]
    dff = bank.w_gate.shape[1]
    tok = np.arange(n, dtype=np.int64) if tokens is None else np.ascontiguousarray(np.asarray(tokens, np.int64))
    used = np.unique(ids[tok].reshape(-1))
    used = used[(used >= 0) & (used < E)]
    b = _Bank(bank, used)
    if shared is not None:
        sh = [_np(getattr(shared, nm)[0], dt) for nm, dt in
              (("w_gate", np.uint8), ("s_gate", np.float32), ("w_up", np.uint8), ("s_up", np.float32),
               ("w_down", np.uint8), ("s_down", np.float32))]
        sh_args = [_ptr(a) for a in sh]
        dff_sh = sh[0].shape[0]
    else:
        sh_args = [None] * 6
        dff_sh = 0
    y = np.empty((tok.size, d), np.float64)
    lib().oracle_layer_forward(d, dff, k, E, _ptr(hb), _ptr(gb), float(eps), _ptr(ids), _ptr(w), *b.args(),
                               *sh_args, dff_sh, _ptr(tok), tok.size, _ptr(y), threads or default_threads(),
                               int(bool(fp8_act)))
    return y


def moe_infer_sorted(x, topk_ids, topk_weight, bank, fp8_act=False):
    """The sorted-slice form (small inputs only).  fp64 [n, d]."""
    xb = _np(x, np.uint16)
    ids = _np(topk_ids, np.int32)
    w = _np(topk_weight, np.float32)
    n, d = xb.shape
    k = ids.shape[1]
    E = bank.w_gate.shape[0]
    dff = bank.w_gate.shape[1]
    b = _Bank(bank)
    y = np.empty((n, d), np.float64)
    lib().oracle_moe_infer_sorted(n, d, dff, k, E, _ptr(xb), _ptr(ids), _ptr(w), *b.args(), _ptr(y),
                                  int(bool(fp8_act)))
    return y


# --------------------------------------------------------------------------- acceptance criterion

MAX_REL_RMS = 1e-2       # max |y - y_ref| <= 1e-2 * rms(y_ref) (+ half a bf16 ulp when the output is bf16)
MEAN_REL = 2e-3          # mean |y - y_ref| / mean |y_ref| <= 2e-3
BF16_HALF_ULP_REL = 2.0 ** -8


def parity_report(y, y_ref, bf16_output: bool = True) -> dict:
    """Compare a library output with the oracle (fp64) under the stated tolerance.

    Per element: |y - y_ref| <= 1e-2 * rms(y_ref) + (2^-8 * |y_ref| if the output is bf16),
    the second term being the largest rounding error of a bf16 result (half an ulp).
    Overall: mean |y - y_ref| / mean |y_ref| <= 2e-3."""
    import torch
    y = y.detach().to("cpu", torch.float64).numpy() if isinstance(y, torch.Tensor) else np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    err = np.abs(y - y_ref)
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    bound = MAX_REL_RMS * rms + (BF16_HALF_ULP_REL * np.abs(y_ref) if bf16_output else 0.0)
    excess = float(np.max(err - bound)) if err.size else 0.0
    mean_rel = float(err.mean() / max(np.abs(y_ref).mean(), 1e-300)) if err.size else 0.0
    finite = bool(np.isfinite(y).all())
    return {
        "ok": finite and excess <= 0.0 and mean_rel <= MEAN_REL,
        "finite": finite,
        "max_err_over_rms": float(err.max() / rms) if err.size and rms > 0 else 0.0,
        "max_excess_over_bound": excess,
        "mean_rel": mean_rel,
        "rms_ref": rms,
        "n": int(err.size),
    }
