"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulate): O max-abs <= 2e-2, LSE max-abs
<= 1e-3, dQ / dK / dV relative L2 <= 1e-2; no NaN / Inf anywhere.  Shapes
span several 128-row tiles, GQA groups of 1..4 heads, causal and full masks,
head_dim 64 and 128, and the full-size workloads.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_flashattention_gb300.workloads import WORKLOADS, custom, make_inputs

pytestmark = pytest.mark.gpu

O_MAXABS = 2e-2
LSE_MAXABS = 1e-3
GRAD_REL = 1e-2
F32_REL = 5e-3


@pytest.fixture(scope="module")
def nea(cuda_device):
    from causal_gqa_flashattention_gb300 import build, nea as binding
    build.build()
    binding.lib()
    return binding


def rel_l2(a, ref):
    """Relative L2 error; a reference that is zero (N = 1 gives dQ = dK = 0
    exactly) is measured against an RMS floor of 1e-3, bf16's resolution at
    unit scale, instead of dividing by ~0."""
    a = a.detach().float().cpu().numpy().astype(np.float64)
    floor = 1e-3 * np.sqrt(ref.size)
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), floor))


def maxabs(a, ref):
    a = a.detach().float().cpu().numpy().astype(np.float64)
    return float(np.abs(a - ref).max())


def finite(*ts):
    return all(bool(torch.isfinite(t.float()).all()) for t in ts)


def run_case(nea, w, seed=0, check_bwd=True):
    dev = torch.device("cuda:0")
    q, k, v, do = make_inputs(w, seed=seed, device=dev)
    # poison outputs: every element must be overwritten
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.N), float("nan"), device=dev)
    nea.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert nea.check_status() == 0
    qc, kc, vc, doc = q.cpu(), k.cpu(), v.cpu(), do.cpu()
    ro, rlse = oracle.attn_fwd(qc, kc, vc, w.scale, w.causal)
    assert finite(o, lse)
    e_o, e_lse = maxabs(o, ro), maxabs(lse, rlse)
    if w.dtype == "bf16":
        assert e_o <= O_MAXABS, e_o
    else:  # fp32 inputs, TF32 tensor-core operands
        assert rel_l2(o, ro) <= F32_REL, rel_l2(o, ro)
    assert e_lse <= LSE_MAXABS, e_lse
    if not check_bwd:
        return
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    code = 0 if w.dtype == "bf16" else 1
    ws = torch.full((nea.bwd_workspace_bytes(w.B, w.H, w.Hkv, w.N, w.d, code),), 0xFF,
                    dtype=torch.uint8, device=dev)
    nea.attn_bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, dq=dq, dk=dk, dv=dv,
                 workspace=ws)
    torch.cuda.synchronize()
    assert nea.check_status() == 0
    assert finite(dq, dk, dv)
    rdq, rdk, rdv = oracle.attn_bwd(qc, kc, vc, doc, w.scale, w.causal)
    errs = dict(dq=rel_l2(dq, rdq), dk=rel_l2(dk, rdk), dv=rel_l2(dv, rdv))
    assert max(errs.values()) <= (GRAD_REL if w.dtype == "bf16" else F32_REL), errs
    # the preprocess row term, against the oracle's D on the same (GPU) O;
    # the workspace holds it per head padded to whole 128-row tiles
    npad = -(-w.N // 128) * 128
    prows = w.B * w.H * npad
    ds = ws[: prows * 4].view(torch.float32).cpu().numpy().reshape(w.B, w.H, npad)[..., : w.N]
    rD = oracle.rowdot(o.cpu(), doc) * w.scale
    assert float(np.abs(ds - rD).max()) <= 1e-4 * max(1.0, float(np.abs(rD).max()))
    return errs


SMALL = [
    custom(1, 2, 1, 128, 64),
    custom(1, 1, 1, 256, 64),
    custom(2, 6, 2, 384, 64),
    custom(1, 4, 1, 512, 64, qk_std=2.0),
    custom(1, 8, 2, 256, 64, causal=False),
    custom(1, 2, 1, 128, 128),
    custom(2, 4, 2, 384, 128, qk_std=2.0),
    custom(1, 4, 4, 256, 128, causal=False),
]


# N not a multiple of the 128-row tile: the last query and key tiles are
# partial (one row, a tile plus one, mid-tile), causal and full masks.
RAGGED = [
    custom(1, 2, 1, 1, 64),
    custom(1, 3, 1, 100, 64),
    custom(2, 6, 2, 129, 64),
    custom(1, 4, 2, 200, 64, causal=False),
    custom(1, 12, 4, 1000, 64),
    custom(1, 2, 1, 77, 128),
    custom(1, 4, 2, 300, 128, causal=False),
    custom(1, 4, 1, 250, 128, qk_std=2.0),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_shapes(nea, w):
    run_case(nea, w)


@pytest.mark.parametrize("w", RAGGED, ids=lambda w: w.name)
def test_ragged_lengths(nea, w):
    run_case(nea, w)


# The forward runs one wave of persistent CTAs (two per SM at d = 64, one at
# d = 128 on a 152-SM GB300), each walking several (head, query tile) items:
# more items than CTAs, with a partial last tile, causal and full masks.
MULTI_ITEM = [
    custom(4, 12, 4, 1000, 64),                 # 384 items, ragged, causal
    custom(2, 12, 4, 1700, 64, causal=False),   # 336 items, ragged, full mask
    custom(2, 8, 2, 1300, 128),                 # 176 items at d = 128
]


@pytest.mark.parametrize("w", MULTI_ITEM, ids=lambda w: w.name)
def test_forward_items_per_cta(nea, w):
    run_case(nea, w)


def test_second_seed_and_repeat(nea):
    w = custom(1, 6, 2, 512, 64)
    run_case(nea, w, seed=1)
    run_case(nea, w, seed=1)


@pytest.mark.parametrize("name", ["gpt2s_bf16", "long_bf16", "wide_bf16"])
def test_full_size_workloads(nea, name):
    run_case(nea, WORKLOADS[name])


@pytest.mark.parametrize("w", [WORKLOADS["tiny_f32"], custom(2, 6, 2, 384, 64, "f32"),
                               custom(1, 4, 2, 256, 64, "f32", causal=False),
                               custom(1, 3, 1, 100, 64, "f32"),
                               custom(1, 4, 2, 200, 64, "f32", causal=False),
                               custom(2, 2, 2, 321, 64, "f32"),
                               WORKLOADS["gpt2s_f32"]], ids=lambda w: w.name)
def test_f32_forward_backward(nea, w):
    run_case(nea, w)


# Maximum sizes: sequences too long for the full fp64 oracle are checked on
# sampled outputs the oracle computes one by one (an O row is the decode
# oracle with one new token at that position; a dQ row needs only its own
# softmax; dK / dV rows of the last key rows need only the few queries that
# see them) and on identities that hold at any size:
# sum_j dV_j = sum over the group's heads and rows of dO, and sum_j dK_j = 0.
LONG = [custom(1, 4, 1, 16384, 64), custom(1, 2, 1, 8192, 128, causal=False)]


@pytest.mark.parametrize("w", LONG, ids=lambda w: w.name)
def test_long_sequence_sampled(nea, w):
    dev = torch.device("cuda:0")
    q, k, v, do = make_inputs(w, seed=11, device=dev)
    o, lse = nea.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = nea.attn_bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert nea.check_status() == 0
    assert finite(o, lse, dq, dk, dv)
    qc, kc, vc, doc = q.cpu(), k.cpu(), v.cpu(), do.cpu()
    G = w.H // w.Hkv
    N = w.N
    rng = np.random.default_rng(5)
    picks = sorted({0, 1, 127, 128, 129, N // 2, N - 129, N - 2, N - 1} |
                   set(int(x) for x in rng.integers(0, N, 12)))
    rows = [(0, h, i) for i in picks for h in (0, w.H - 1)]
    # forward rows
    for (b, h, i) in rows:
        g = h // G
        L = i + 1 if w.causal else N
        ro, rl = oracle.attn_decode(qc[b:b + 1, h:h + 1, i:i + 1], kc[b:b + 1, g:g + 1],
                                    vc[b:b + 1, g:g + 1], [L], w.scale)
        got = o[b, h, i].float().cpu().numpy().astype(np.float64)
        assert np.abs(got - ro[0, 0, 0]).max() <= O_MAXABS, (h, i)
        assert abs(float(lse[b, h, i]) - rl[0, 0, 0]) <= LSE_MAXABS, (h, i)
    # dQ rows
    rdq = oracle.attn_bwd_dq_rows(qc, kc, vc, doc, rows, w.scale, w.causal)
    gdq = np.stack([dq[b, h, i].float().cpu().numpy() for (b, h, i) in rows]).astype(np.float64)
    assert np.linalg.norm(gdq - rdq) / np.linalg.norm(rdq) <= GRAD_REL
    # dK, dV rows (the last key rows: only the queries after them contribute)
    if w.causal:
        krows = [(0, g, j) for g in range(w.Hkv) for j in (N - 1, N - 2, N - 129)]
        rdk, rdv = oracle.attn_bwd_dkdv_rows(qc, kc, vc, doc, krows, w.scale, True)
        gdk = np.stack([dk[b, g, j].float().cpu().numpy() for (b, g, j) in krows]).astype(np.float64)
        gdv = np.stack([dv[b, g, j].float().cpu().numpy() for (b, g, j) in krows]).astype(np.float64)
        assert np.linalg.norm(gdk - rdk) / np.linalg.norm(rdk) <= GRAD_REL
        assert np.linalg.norm(gdv - rdv) / np.linalg.norm(rdv) <= GRAD_REL
    # identities over every key row
    dv64 = dv.double().cpu().numpy()
    dk64 = dk.double().cpu().numpy()
    do64 = doc.double().numpy()
    for g in range(w.Hkv):
        want = do64[0, g * G:(g + 1) * G].sum(axis=(0, 1))
        got = dv64[0, g].sum(axis=0)
        assert np.linalg.norm(got - want) <= 1e-2 * np.linalg.norm(want)
        scale_k = np.abs(dk64[0, g]).sum(axis=0)
        assert np.all(np.abs(dk64[0, g].sum(axis=0)) <= 1e-2 * scale_k + 1e-6)
