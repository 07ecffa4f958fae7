"""GPU: the backward's three public stages on one reused workspace.

The bf16 backward adds every dQ partial into an fp32 accumulator in the
workspace, which the preprocess clears and the cast reads back.  These tests
run the stages in sequence on a workspace full of 0xFF bytes (NaN as fp32),
and then again on the same workspace with other inputs, so that anything the
preprocess failed to clear, or left from the previous call, would show up.
Each result is checked against the fp64 oracle at the parity tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_flashattention_gb300.workloads import custom, make_inputs

pytestmark = pytest.mark.gpu

GRAD_REL = 1e-2


@pytest.fixture(scope="module")
def nea(cuda_device):
    from causal_gqa_flashattention_gb300 import build, nea as binding
    build.build()
    binding.lib()
    return binding


def rel_l2(a, ref):
    a = a.detach().float().cpu().numpy().astype(np.float64)
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), 1e-3 * np.sqrt(ref.size)))


CASES = [
    custom(1, 2, 1, 1, 64),                    # one row
    custom(2, 6, 2, 640, 64),                  # 1 to 5 partials per query tile
    custom(1, 4, 2, 333, 64, causal=False),    # every tile gets T partials; ragged
    custom(1, 4, 1, 520, 128),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_staged_calls_reuse_one_workspace(nea, w):
    dev = torch.device("cuda:0")
    ws = torch.full((nea.bwd_workspace_bytes(w.B, w.H, w.Hkv, w.N, w.d, 0),), 0xFF,
                    dtype=torch.uint8, device=dev)
    for seed in (0, 1):
        q, k, v, do = make_inputs(w, seed=seed, device=dev)
        o, lse = nea.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
        dq = torch.full_like(q, float("nan"))
        dk = torch.full_like(k, float("nan"))
        dv = torch.full_like(v, float("nan"))
        nea.attn_bwd_stages(q, k, v, o, do, lse, dq, dk, dv, ws, causal=w.causal, scale=w.scale)
        torch.cuda.synchronize()
        assert nea.check_status() == 0
        rdq, rdk, rdv = oracle.attn_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), w.scale, w.causal)
        errs = dict(dq=rel_l2(dq, rdq), dk=rel_l2(dk, rdk), dv=rel_l2(dv, rdv))
        assert max(errs.values()) <= GRAD_REL, (seed, errs)


def test_back_to_back_calls_without_sync(nea):
    """Several backward calls queued on one stream with one workspace: each
    call's preprocess clears what the previous call left there."""
    w = custom(2, 6, 2, 384, 64)
    dev = torch.device("cuda:0")
    ws = torch.empty(nea.bwd_workspace_bytes(w.B, w.H, w.Hkv, w.N, w.d, 0), dtype=torch.uint8,
                     device=dev)
    runs = []
    for seed in (3, 4, 5):
        q, k, v, do = make_inputs(w, seed=seed, device=dev)
        o, lse = nea.attn_fwd(q, k, v, causal=True, scale=w.scale)
        dq, dk, dv = nea.attn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale, workspace=ws)
        runs.append((q, k, v, do, dq, dk, dv))
    torch.cuda.synchronize()
    assert nea.check_status() == 0
    for q, k, v, do, dq, dk, dv in runs:
        rdq, rdk, rdv = oracle.attn_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), w.scale, True)
        errs = dict(dq=rel_l2(dq, rdq), dk=rel_l2(dk, rdk), dv=rel_l2(dv, rdv))
        assert max(errs.values()) <= GRAD_REL, errs
