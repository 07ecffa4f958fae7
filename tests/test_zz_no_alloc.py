"""The workspace-free backward entry point, nea_attn_bwd_noalloc().

It exists for callers that cannot allocate device memory themselves (a host
framework that hands over only input / output pointers, or a path where
cudaMalloc's implicit device synchronisation is not acceptable); its scratch
is a fixed array inside the library.  This test calls it through the C ABI
twice in a row and checks both results against nea_attn_bwd() with a
caller-owned workspace and against the fp64 oracle, within the parity
tolerances of the other GPU tests (relative L2 1e-2 on dQ, dK, dV for bf16,
5e-3 for fp32 inputs on TF32 tensor cores).  The file name makes pytest
collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

from causal_gqa_flashattention_gb300.workloads import custom, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(cuda_device):
    from causal_gqa_flashattention_gb300 import build, nea
    build.build()
    L = nea.lib()
    L.nea_attn_bwd_noalloc.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    L.nea_attn_bwd_noalloc.restype = ctypes.c_int
    L.nea_attn_bwd_noalloc_max_bytes.restype = ctypes.c_size_t
    return nea, L


def rel_l2(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


def rel_l2_oracle(a, ref):
    a = a.detach().float().cpu().numpy().astype(np.float64)
    return float(np.linalg.norm(a - ref) / np.linalg.norm(ref))


def call_noalloc(L, w, code, q, k, v, o, do, lse, dq, dk, dv):
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.nea_attn_bwd_noalloc(p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv),
                                  w.B, w.H, w.Hkv, w.N, w.d, w.scale, 1, code, stream)


@pytest.mark.parametrize("w", [custom(2, 6, 2, 512, 64), custom(1, 4, 2, 256, 128),
                               custom(1, 2, 1, 128, 64, dtype="f32")],
                         ids=lambda w: w.name)
def test_noalloc_matches_workspace_entry_point(lib, w):
    nea, L = lib
    dev = torch.device("cuda:0")
    code = nea.NEA_BF16 if w.dtype == "bf16" else nea.NEA_F32
    tol = 1e-2 if w.dtype == "bf16" else 5e-3
    q, k, v, do = make_inputs(w, seed=3, device=dev)
    o, lse = nea.attn_fwd(q, k, v, causal=True, scale=w.scale)
    ref = nea.attn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    exact = oracle.attn_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), w.scale, True)
    for _ in range(2):  # two calls in a row: the shared scratch is reused
        dq = torch.full_like(q, float("nan"))
        dk = torch.full_like(k, float("nan"))
        dv = torch.full_like(v, float("nan"))
        st = call_noalloc(L, w, code, q, k, v, o, do, lse, dq, dk, dv)
        assert st == nea.NEA_OK, nea.status_string(st)
        torch.cuda.synchronize()
        assert nea.check_status() == nea.NEA_OK
        for got, want, r in zip((dq, dk, dv), ref, exact):
            assert bool(torch.isfinite(got.float()).all())
            assert rel_l2(got, want) <= tol
            assert rel_l2_oracle(got, r) <= tol


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    nea, L = lib
    w = custom(4, 16, 4, 2048, 128)  # needs ~68 MB of scratch
    assert nea.bwd_workspace_bytes(w.B, w.H, w.Hkv, w.N, w.d, 0) > L.nea_attn_bwd_noalloc_max_bytes()
    t = torch.empty(16, device="cuda:0")
    p = ctypes.c_void_p(t.data_ptr())
    st = L.nea_attn_bwd_noalloc(*([p] * 9), w.B, w.H, w.Hkv, w.N, w.d, w.scale, 1, 0,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == nea.NEA_ERR_WORKSPACE
