"""ctypes binding of ``libnea_attn.so`` (the C ABI of include/nea_attn.h).

Argument marshalling only: every step of the attention runs in the library's
CUDA kernels.  PyTorch provides device memory (output tensors are allocated
with ``torch.empty`` when the caller passes none) and the current stream.
There is no fallback: if the library is missing or a call fails, this module
raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnea_attn.so")

NEA_OK = 0
NEA_ERR_INVALID = -1
NEA_ERR_UNSUPPORTED = -2
NEA_ERR_CUDA = -3
NEA_ERR_TIMEOUT = -4
NEA_ERR_WORKSPACE = -5
NEA_BF16 = 0
NEA_F32 = 1

_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float


class NeaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def lib():
    """Load the library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            _lib = load_library(LIB_PATH)
    return _lib


def load_library(path):
    """Load a build of the library from ``path`` and declare its C ABI."""
    L = ctypes.CDLL(path)
    L.nea_attn_fwd.argtypes = [_vp] * 5 + [_i] * 5 + [_f, _i, _i, _vp]
    L.nea_attn_fwd.restype = _i
    L.nea_attn_bwd_workspace_bytes.argtypes = [_i] * 6
    L.nea_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.nea_attn_bwd.argtypes = [_vp] * 10 + [ctypes.c_size_t] + [_i] * 5 + [_f, _i, _i, _vp]
    L.nea_attn_bwd.restype = _i
    L.nea_attn_bwd_preprocess.argtypes = [_vp] * 5 + [ctypes.c_size_t] + [_i] * 5 + [
        _f, _i, _vp]
    L.nea_attn_bwd_preprocess.restype = _i
    L.nea_attn_bwd_main.argtypes = [_vp] * 8 + [ctypes.c_size_t] + [_i] * 5 + [
        _f, _i, _i, _vp]
    L.nea_attn_bwd_main.restype = _i
    L.nea_attn_bwd_finalize.argtypes = [_vp] * 2 + [ctypes.c_size_t] + [_i] * 6 + [_vp]
    L.nea_attn_bwd_finalize.restype = _i
    L.nea_rope_table.argtypes = [_vp, _i, _i, ctypes.c_double, _vp]
    L.nea_rope_table.restype = _i
    L.nea_attn_fwd_rope_q.argtypes = [_vp] * 6 + [_i] * 5 + [ctypes.c_float] + [_i] * 2 + [_vp]
    L.nea_attn_fwd_rope_q.restype = _i
    L.nea_rope_qk.argtypes = [_vp] * 5 + [_i] * 6 + [_vp]
    L.nea_rope_qk.restype = _i
    L.nea_attn_bwd_rope.argtypes = [_vp] * 11 + [ctypes.c_size_t] + [_i] * 5 + [
        _f, _i, _i, _vp]
    L.nea_attn_bwd_rope.restype = _i
    L.nea_attn_bwd_ex.argtypes = [_vp] * 7 + [_i] + [_vp] * 4 + [ctypes.c_size_t] + [
        _i] * 5 + [_f, _i, _i, _vp]
    L.nea_attn_bwd_ex.restype = _i
    L.nea_attn_decode_workspace_bytes.argtypes = [_i] * 6
    L.nea_attn_decode_workspace_bytes.restype = ctypes.c_size_t
    L.nea_attn_decode.argtypes = [_vp] * 7 + [ctypes.c_size_t] + [_i] * 6 + [_f, _i, _vp]
    L.nea_attn_decode.restype = _i
    L.nea_attn_check_status.argtypes = [_vp]
    L.nea_attn_check_status.restype = _i
    L.nea_status_string.argtypes = [_i]
    L.nea_status_string.restype = ctypes.c_char_p
    L.nea_version.restype = _i
    return L


def use_library(L):
    """Make the calls of this module go to the loaded library ``L`` (from
    load_library, e.g. a test build); returns the one they used before."""
    global _lib
    prev = lib()
    with _lock:
        _lib = L
    return prev


def status_string(status: int) -> str:
    return lib().nea_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return NEA_BF16
    if t.dtype == torch.float32:
        return NEA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check(q, k, v):
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape:
        raise ValueError("k / v must be [B, Hkv, N, d]")
    return B, H, Hkv, N, d


def attn_fwd(q, k, v, *, causal=True, scale=None, out=None, lse=None, stream=None,
             rope_q_cs=None):
    """O, LSE = attention(q, k, v).  q [B,H,N,d], k/v [B,Hkv,N,d] (bf16).

    With ``rope_q_cs`` (a RoPE table), ``q`` is the unrotated Q, ``k`` the
    rotated K, and the kernel rotates Q itself (nea_attn_fwd_rope_q)."""
    B, H, Hkv, N, d = _check(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    s = ctypes.c_void_p(_stream_handle(stream))
    if rope_q_cs is None:
        st = lib().nea_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse_t), B, H, Hkv, N, d,
                                scale, int(bool(causal)), _dtype_code(q), s)
        what = "nea_attn_fwd"
    else:
        st = lib().nea_attn_fwd_rope_q(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse_t),
                                       _ptr(rope_q_cs), B, H, Hkv, N, d, scale,
                                       int(bool(causal)), _dtype_code(q), s)
        what = "nea_attn_fwd_rope_q"
    if st != NEA_OK:
        raise NeaError(st, what)
    return o, lse_t


def bwd_workspace_bytes(B, H, Hkv, N, d, dtype=NEA_BF16) -> int:
    return int(lib().nea_attn_bwd_workspace_bytes(B, H, Hkv, N, d, dtype))


def rope_table(N, d, *, base=10000.0, device=None, out=None, stream=None):
    """RoPE (cos, sin) table [N, d/2, 2] fp32 for positions 0..N-1, computed on the GPU."""
    cs = out if out is not None else torch.empty((N, d // 2, 2), dtype=torch.float32,
                                                 device=device or "cuda")
    st = lib().nea_rope_table(_ptr(cs), int(N), int(d), float(base),
                              ctypes.c_void_p(_stream_handle(stream)))
    if st != NEA_OK:
        raise NeaError(st, "nea_rope_table")
    return cs


def rope_qk(q, k, cos_sin, *, qr=None, kr=None, stream=None):
    """Qr, Kr = R(q), R(k): the rotary embedding of q [B,H,N,d] and k [B,Hkv,N,d]."""
    B, H, Hkv, N, d = _check(q, k, k)
    qr = torch.empty_like(q) if qr is None else qr
    kr = torch.empty_like(k) if kr is None else kr
    st = lib().nea_rope_qk(_ptr(q), _ptr(k), _ptr(qr), _ptr(kr), _ptr(cos_sin), B, H, Hkv, N, d,
                           _dtype_code(q), ctypes.c_void_p(_stream_handle(stream)))
    if st != NEA_OK:
        raise NeaError(st, "nea_rope_qk")
    return qr, kr


NEA_BWD_DETERMINISTIC = 1


def attn_bwd(q, k, v, o, do, lse, *, causal=True, scale=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None, rope_cs=None, deterministic=False):
    """dQ, dK, dV for upstream gradient ``do``, using the forward's O and LSE.

    With ``rope_cs`` (the table ``q`` and ``k`` were rotated with), ``q`` and
    ``k`` are the rotated inputs and dQ, dK are returned with respect to the
    unrotated ones.  ``deterministic`` selects the bit-reproducible dQ path."""
    B, H, Hkv, N, d = _check(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    code = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_bytes(B, H, Hkv, N, d, code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if deterministic:
        st = lib().nea_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                   _ptr(rope_cs), NEA_BWD_DETERMINISTIC, _ptr(dq), _ptr(dk),
                                   _ptr(dv), _ptr(workspace), workspace.numel(), B, H, Hkv, N, d,
                                   scale, int(bool(causal)), code,
                                   ctypes.c_void_p(_stream_handle(stream)))
        what = "nea_attn_bwd_ex"
    elif rope_cs is None:
        st = lib().nea_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, H,
                                Hkv, N, d, scale, int(bool(causal)), code,
                                ctypes.c_void_p(_stream_handle(stream)))
        what = "nea_attn_bwd"
    else:
        st = lib().nea_attn_bwd_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                     _ptr(rope_cs), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                     workspace.numel(), B, H, Hkv, N, d, scale,
                                     int(bool(causal)), code,
                                     ctypes.c_void_p(_stream_handle(stream)))
        what = "nea_attn_bwd_rope"
    if st != NEA_OK:
        raise NeaError(st, what)
    return dq, dk, dv


def attn_bwd_stages(q, k, v, o, do, lse, dq, dk, dv, workspace, *, causal=True, scale=None,
                    stream=None, between=None, only=None):
    """The backward as its three ABI stages (same work as ``attn_bwd``).
    ``between(i)`` is called before stage i (0, 1, 2) and after the last
    (i = 3), e.g. to record CUDA events between the kernels.  ``only``: a set
    of stage indices to run (default all), e.g. to time one stage alone on a
    workspace that earlier calls have filled."""
    B, H, Hkv, N, d = _check(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    code = _dtype_code(q)
    s = ctypes.c_void_p(_stream_handle(stream))
    L = lib()
    nb = workspace.numel()
    run = (lambda i: True) if only is None else (lambda i: i in only)
    if between:
        between(0)
    if run(0):
        st = L.nea_attn_bwd_preprocess(_ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(workspace),
                                       nb, B, H, Hkv, N, d, scale, code, s)
        if st != NEA_OK:
            raise NeaError(st, "nea_attn_bwd_preprocess")
    if between:
        between(1)
    if run(1):
        st = L.nea_attn_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(workspace), nb, B, H, Hkv, N, d, scale,
                                 int(bool(causal)), code, s)
        if st != NEA_OK:
            raise NeaError(st, "nea_attn_bwd_main")
    if between:
        between(2)
    if run(2):
        st = L.nea_attn_bwd_finalize(_ptr(dq), _ptr(workspace), nb, B, H, Hkv, N, d, code, s)
        if st != NEA_OK:
            raise NeaError(st, "nea_attn_bwd_finalize")
    if between:
        between(3)
    return dq, dk, dv


def decode_workspace_bytes(B, H, Hkv, nq, Lmax, d) -> int:
    return int(lib().nea_attn_decode_workspace_bytes(B, H, Hkv, nq, Lmax, d))


def attn_decode(q, k_cache, v_cache, lens, *, scale=None, out=None, lse=None, workspace=None,
                stream=None):
    """Decode attention of q [B,H,nq,d] (the newest nq tokens) against caches
    [B,Hkv,Lmax,d] with ``lens`` [B] int32 (device) valid rows each, the new
    tokens included.  Returns (O [B,H,nq,d], LSE [B,H,nq])."""
    for t in (q, k_cache, v_cache, lens):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    if lens.dtype != torch.int32:
        raise TypeError("lens must be int32")
    B, H, nq, d = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Hkv, Lmax, d) or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [B, Hkv, Lmax, d]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty((B, H, nq), dtype=torch.float32, device=q.device) if lse is None else lse
    need = decode_workspace_bytes(B, H, Hkv, nq, Lmax, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = lib().nea_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), _ptr(o),
                               _ptr(lse_t), _ptr(workspace), workspace.numel(), B, H, Hkv, nq,
                               Lmax, d, scale, _dtype_code(q),
                               ctypes.c_void_p(_stream_handle(stream)))
    if st != NEA_OK:
        raise NeaError(st, "nea_attn_decode")
    return o, lse_t


def check_status(stream=None) -> int:
    return int(lib().nea_attn_check_status(ctypes.c_void_p(_stream_handle(stream))))
