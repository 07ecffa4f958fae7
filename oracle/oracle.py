"""ctypes binding of ``oracle.c``, the fp64 CPU reference (test infrastructure).

Parity unpinned: none.  Every function here is pinned by ``tests/test_oracle.py``
(closed forms, invariants, finite differences with the pages' epsilon and
threshold, textbook special cases).

Definitions followed ("NanoEuler: Hand-writing GPT-2 in Pure C/CUDA"):
section "Tiled FlashAttention" (exact softmax attention, computed row by row
here), "Architecture Deep Dive" (decoder, hence causal), "Build and Run"
(the config's 12 query / 4 KV heads, hence grouped-query attention) and
"Hand-written Backpropagation" (the hand-derived backward); the FAQ that
compares the project with llm.c names RoPE among its techniques, taken here as
the original rotary embedding on pairs (2i, 2i+1) (see ``rope``); the FAQ on
production inference says inference works (see ``attn_decode`` for the
cache reading taken).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def lib_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc + OpenMP (plain C, no target-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_attn_fwd_f64.argtypes = [_dp, _dp, _dp, _dp, _dp] + [ctypes.c_int] * 5 + [
                ctypes.c_double, ctypes.c_int]
            lib.oracle_attn_fwd_f64.restype = ctypes.c_int
            lib.oracle_attn_bwd_f64.argtypes = [_dp] * 9 + [ctypes.c_int] * 5 + [
                ctypes.c_double, ctypes.c_int]
            lib.oracle_attn_bwd_f64.restype = ctypes.c_int
            lib.oracle_rowdot_f64.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_int]
            lib.oracle_rowdot_f64.restype = ctypes.c_int
            lib.oracle_rope_f64.argtypes = [_dp, _dp, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int]
            lib.oracle_rope_f64.restype = ctypes.c_int
            lib.oracle_attn_decode_f64.argtypes = [_dp, _dp, _dp, ctypes.POINTER(ctypes.c_int),
                                                   _dp, _dp] + [ctypes.c_int] * 6 + [
                                                       ctypes.c_double]
            lib.oracle_attn_decode_f64.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _f64(a) -> np.ndarray:
    """Widen to a contiguous fp64 array.  Accepts numpy or (CPU) torch tensors;
    bf16 torch tensors are widened exactly through fp32."""
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        if str(a.dtype) == "torch.bfloat16":
            a = a.float()
        a = a.double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def attn_fwd(q, k, v, scale: float, causal: bool = True):
    """Softmax attention forward.  q [B,H,N,d], k/v [B,Hkv,N,d].

    Returns (O [B,H,N,d], LSE [B,H,N]) as fp64 numpy arrays; LSE in natural-log
    units of the scaled logits.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    assert k.shape == (B, Hkv, N, d) and v.shape == k.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attn_fwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                     B, H, Hkv, N, d, float(scale), int(bool(causal)))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_f64 rejected its arguments")
    return o, lse


def attn_bwd(q, k, v, do, scale: float, causal: bool = True, return_delta: bool = False):
    """Softmax attention backward for an upstream gradient ``do``.

    Returns (dQ, dK, dV) and, with ``return_delta``, also (D, Dalt): the two
    forms of the per-row term, sum_k dO*O and sum_j P*dP.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    assert k.shape == (B, Hkv, N, d) and v.shape == k.shape and do.shape == q.shape
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    D = np.empty((B, H, N), dtype=np.float64)
    Dalt = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attn_bwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk),
                                     _ptr(dv), _ptr(D), _ptr(Dalt), B, H, Hkv, N, d,
                                     float(scale), int(bool(causal)))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_f64 rejected its arguments")
    if return_delta:
        return dq, dk, dv, D, Dalt
    return dq, dk, dv


def rowdot(o, do):
    """D = sum over the last axis of O * dO, in fp64 (shape o.shape[:-1])."""
    o, do = _f64(o), _f64(do)
    assert o.shape == do.shape
    d = o.shape[-1]
    rows = int(np.prod(o.shape[:-1])) if o.ndim > 1 else 1
    out = np.empty(o.shape[:-1], dtype=np.float64)
    rc = _load().oracle_rowdot_f64(_ptr(o), _ptr(do), _ptr(out), rows, d)
    if rc != 0:
        raise ValueError("oracle_rowdot_f64 rejected its arguments")
    return out


def rope(x, base: float = 10000.0, inverse: bool = False):
    """Rotary position embedding of x [..., N, d] in fp64 (d even).

    Pair (x_2i, x_2i+1) of the row at position n is turned by n * theta_i,
    theta_i = base^(-2i/d); ``inverse`` turns by the opposite angle (the
    transpose, which maps gradients of the rotated rows back).
    """
    x = _f64(x)
    N, d = x.shape[-2], x.shape[-1]
    rows = x.size // d
    y = np.empty_like(x)
    rc = _load().oracle_rope_f64(_ptr(x), _ptr(y), rows, N, d, float(base), int(bool(inverse)))
    if rc != 0:
        raise ValueError("oracle_rope_f64 rejected its arguments")
    return y


def attn_decode(q, k_cache, v_cache, lens, scale: float):
    """Decode attention: q [B,H,nq,d] (the nq newest tokens), caches
    [B,Hkv,Lmax,d] holding lens[b] valid rows that include the new tokens.
    New token t of batch b sits at position lens[b] - nq + t and sees cache
    rows up to it.  Returns (O [B,H,nq,d], LSE [B,H,nq]) in fp64."""
    q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
    B, H, nq, d = q.shape
    Hkv, Lmax = kc.shape[1], kc.shape[2]
    assert kc.shape == (B, Hkv, Lmax, d) and vc.shape == kc.shape
    ln = np.ascontiguousarray(np.asarray(lens, dtype=np.int32).reshape(B))
    o = np.empty_like(q)
    lse = np.empty((B, H, nq), dtype=np.float64)
    rc = _load().oracle_attn_decode_f64(_ptr(q), _ptr(kc), _ptr(vc),
                                        ln.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), _ptr(o),
                                        _ptr(lse), B, H, Hkv, nq, Lmax, d, float(scale))
    if rc != 0:
        raise ValueError("oracle_attn_decode_f64 rejected its arguments")
    return o, lse
