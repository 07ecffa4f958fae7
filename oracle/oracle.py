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


def attn_bwd_dq_rows(q, k, v, do, rows, scale: float, causal: bool = True):
    """dQ for selected query rows only, fp64, from the definitions (for
    sequences too long for the full backward): for row i of head h
    (group g = h / (H / Hkv)),
        P_ij  = softmax_j(scale q_i . k_j) over j <= i (all j if not causal)
        O_i   = sum_j P_ij v_j,   D_i = dO_i . O_i,   dP_ij = dO_i . v_j
        dQ_i  = scale sum_j P_ij (dP_ij - D_i) k_j.
    ``rows`` is a list of (b, h, i); returns an array [len(rows), d]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    H, Hkv = q.shape[1], k.shape[1]
    N = q.shape[2]
    out = np.empty((len(rows), q.shape[3]))
    for n, (b, h, i) in enumerate(rows):
        g = h // (H // Hkv)
        end = i + 1 if causal else N
        K, V = k[b, g, :end], v[b, g, :end]
        s = scale * (K @ q[b, h, i])
        p = np.exp(s - s.max())
        p /= p.sum()
        o = p @ V
        dp = V @ do[b, h, i]
        ds = p * (dp - do[b, h, i] @ o)
        out[n] = scale * (ds @ K)
    return out


def attn_bwd_dkdv_rows(q, k, v, do, rows, scale: float, causal: bool = True):
    """dK and dV for selected key rows, fp64, from the definitions: for key
    row j of KV head g, summed over the group's query heads h and the query
    rows i that see it (i >= j under the causal mask),
        dK_j = scale sum_{h, i} P_ij (dP_ij - D_i) q_i,   dV_j = sum_{h, i} P_ij dO_i,
    each P_ij, D_i from row i's full softmax.  Cheap for the last key rows of
    a causal sequence.  ``rows`` is a list of (b, g, j); returns (dK, dV),
    each [len(rows), d]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    H, Hkv, N, d = q.shape[1], k.shape[1], q.shape[2], q.shape[3]
    G = H // Hkv
    dk = np.zeros((len(rows), d))
    dv = np.zeros((len(rows), d))
    for n, (b, g, j) in enumerate(rows):
        for h in range(g * G, (g + 1) * G):
            for i in range(j if causal else 0, N):
                end = i + 1 if causal else N
                K, V = k[b, g, :end], v[b, g, :end]
                s = scale * (K @ q[b, h, i])
                p = np.exp(s - s.max())
                p /= p.sum()
                o = p @ V
                dij = p[j] * (V[j] @ do[b, h, i] - do[b, h, i] @ o)
                dk[n] += scale * dij * q[b, h, i]
                dv[n] += p[j] * do[b, h, i]
    return dk, dv
