"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test targets a mistake the oracle could plausibly make (a dropped term,
a wrong sign, a transposed operand, an off-by-one mask, a wrong GQA index):
- a hand-derived worked example (tests/golden/worked_n2_gqa.json);
- closed forms: Q = 0 gives the causal prefix mean of V and LSE = ln(i+1);
  row 0 gives O = V_0 and LSE = scale * q_0 . k_0;
- softmax rows are a probability distribution with causal support;
- central finite differences of L = sum(O * dO) with the pages' epsilon 1e-5
  and relative-error threshold 1e-4 ("NanoEuler: Hand-writing GPT-2 in Pure
  C/CUDA", section "Hand-written Backpropagation" and the FAQ answer on
  gradient checking);
- special cases: constant V, N = 1, the dV / dK sum identities;
- reductions to library routines: scipy's softmax for textbook attention,
  torch fp64 autograd for the gradients, and MHA with K/V repeated per group.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rand(*shape, std=1.0):
    return rng.standard_normal(shape) * std


def test_worked_example_by_hand():
    ex = json.load(open(os.path.join(GOLD, "worked_n2_gqa.json")))
    s = ex["shape"]
    inp = {k: np.array(v, dtype=np.float64) for k, v in ex["inputs"].items()}
    exp = {k: np.array(v, dtype=np.float64) for k, v in ex["expected"].items()}
    o, lse = oracle.attn_fwd(inp["q"], inp["k"], inp["v"], s["scale"], s["causal"])
    np.testing.assert_allclose(o, exp["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, exp["lse"], rtol=0, atol=1e-12)
    dq, dk, dv, D, Dalt = oracle.attn_bwd(inp["q"], inp["k"], inp["v"], inp["do"], s["scale"],
                                          s["causal"], return_delta=True)
    np.testing.assert_allclose(dq, exp["dq"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, exp["dk"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, exp["dv"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(D, exp["D"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(Dalt, exp["D"], rtol=0, atol=1e-12)


def test_page_config_shapes():
    """The GPT-2-small workload carries the page's config-file attention shape."""
    from causal_gqa_flashattention_gb300.workloads import WORKLOADS
    cfg = json.load(open(os.path.join(GOLD, "gpt2_small_config.json")))
    w = WORKLOADS["gpt2s_bf16"]
    m = cfg["model"]
    assert w.H == m["num_heads"] and w.Hkv == m["num_kv_heads"]
    assert w.N == m["max_seq_len"] and w.B == cfg["training"]["batch_size"]
    assert w.d == m["hidden_dim"] // m["num_heads"] == cfg["derived"]["head_dim"]
    assert w.H // w.Hkv == cfg["derived"]["group_size"]


@pytest.mark.parametrize("causal", [True, False])
def test_q_zero_closed_form(causal):
    B, H, Hkv, N, d = 2, 4, 2, 37, 8
    q = np.zeros((B, H, N, d))
    k, v = rand(B, Hkv, N, d), rand(B, Hkv, N, d)
    o, lse = oracle.attn_fwd(q, k, v, 0.3, causal)
    G = H // Hkv
    for h in range(H):
        vg = v[:, h // G]
        if causal:
            want = np.cumsum(vg, axis=1) / np.arange(1, N + 1)[None, :, None]
            want_lse = np.log(np.arange(1, N + 1))[None, :].repeat(B, 0)
        else:
            want = np.repeat(vg.mean(axis=1, keepdims=True), N, axis=1)
            want_lse = np.full((B, N), math.log(N))
        np.testing.assert_allclose(o[:, h], want, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[:, h], want_lse, rtol=1e-12, atol=1e-12)


def test_row0_closed_form():
    B, H, Hkv, N, d, s = 1, 6, 2, 20, 16, 0.25
    q, k, v = rand(B, H, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d)
    o, lse = oracle.attn_fwd(q, k, v, s, True)
    for h in range(H):
        g = h // 3
        np.testing.assert_allclose(o[0, h, 0], v[0, g, 0], rtol=0, atol=1e-14)
        assert abs(lse[0, h, 0] - s * q[0, h, 0] @ k[0, g, 0]) < 1e-13


def test_softmax_rows_are_distributions():
    """With V the identity (N = d), O_i is the softmax row P_i itself."""
    N = d = 24
    q, k = rand(1, 1, N, d, std=2.0), rand(1, 1, N, d, std=2.0)
    v = np.eye(N)[None, None]
    for causal in (True, False):
        P, _ = oracle.attn_fwd(q, k, v, 1 / math.sqrt(d), causal)
        P = P[0, 0]
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-13)
        assert (P >= 0).all()
        if causal:
            assert np.all(np.triu(P, 1) == 0.0)
            assert np.all(np.diag(P) > 0)


def _textbook(q, k, v, s, causal):
    from scipy.special import logsumexp, softmax
    S = s * np.einsum("bhid,bhjd->bhij", q, k)
    if causal:
        N = S.shape[-1]
        S = np.where(np.tril(np.ones((N, N), bool)), S, -np.inf)
    return softmax(S, axis=-1) @ v, logsumexp(S, axis=-1)


@pytest.mark.parametrize("causal", [True, False])
def test_mha_matches_scipy_softmax(causal):
    B, H, N, d, s = 2, 3, 33, 16, 0.2
    q, k, v = rand(B, H, N, d, std=2.0), rand(B, H, N, d, std=2.0), rand(B, H, N, d)
    o, lse = oracle.attn_fwd(q, k, v, s, causal)
    want_o, want_lse = _textbook(q, k, v, s, causal)
    np.testing.assert_allclose(o, want_o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_gqa_equals_mha_with_repeated_kv(causal):
    B, H, Hkv, N, d, s = 2, 6, 2, 19, 8, 0.35
    G = H // Hkv
    q, k, v, do = rand(B, H, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, H, N, d)
    o, lse = oracle.attn_fwd(q, k, v, s, causal)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)   # head h -> KV head h // G
    o2, lse2 = oracle.attn_fwd(q, kr, vr, s, causal)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-13)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, s, causal)
    dq2, dk2, dv2 = oracle.attn_bwd(q, kr, vr, do, s, causal)
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, G, N, d).sum(2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, G, N, d).sum(2), rtol=0, atol=1e-12)


def test_gqa_group_index_is_contiguous():
    """Head h must read KV head h // G: moving KV head 1 only changes heads 3..5."""
    B, H, Hkv, N, d = 1, 6, 2, 10, 8
    q, k, v = rand(B, H, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d)
    o1, _ = oracle.attn_fwd(q, k, v, 0.3, True)
    v2 = v.copy()
    v2[:, 1] += 1.0
    o2, _ = oracle.attn_fwd(q, k, v2, 0.3, True)
    np.testing.assert_array_equal(o1[:, :3], o2[:, :3])
    np.testing.assert_allclose(o2[:, 3:], o1[:, 3:] + 1.0, rtol=0, atol=1e-12)


def _loss(q, k, v, do, s, causal):
    o, _ = oracle.attn_fwd(q, k, v, s, causal)
    return float((o * do).sum())


def _fd_check(q, k, v, do, s, causal, coords=None, eps=1e-5, tol=1e-4):
    """Central finite differences vs the oracle's backward, the pages' method:
    perturb by eps = 1e-5, relative error under 1e-4."""
    grads = dict(zip("qkv", oracle.attn_bwd(q, k, v, do, s, causal)))
    arrs = {"q": q, "k": k, "v": v}
    worst = 0.0
    for name, a in arrs.items():
        idxs = list(np.ndindex(a.shape)) if coords is None else coords[name]
        for idx in idxs:
            orig = a[idx]
            a[idx] = orig + eps
            lp = _loss(q, k, v, do, s, causal)
            a[idx] = orig - eps
            lm = _loss(q, k, v, do, s, causal)
            a[idx] = orig
            fd = (lp - lm) / (2 * eps)
            an = grads[name][idx]
            denom = max(abs(fd), abs(an), 1e-6)
            rel = abs(fd - an) / denom
            worst = max(worst, rel)
            assert rel < tol, (name, idx, fd, an)
    return worst


@pytest.mark.parametrize("causal", [True, False])
def test_finite_difference_every_coordinate(causal):
    B, H, Hkv, N, d = 1, 2, 1, 16, 8
    q, k, v, do = rand(B, H, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, H, N, d)
    _fd_check(q, k, v, do, 1 / math.sqrt(d), causal)


def test_finite_difference_sampled_gqa_large_logits():
    B, H, Hkv, N, d = 1, 6, 2, 40, 16
    q, k = rand(B, H, N, d, std=2.0), rand(B, Hkv, N, d, std=2.0)
    v, do = rand(B, Hkv, N, d), rand(B, H, N, d)
    coords = {}
    for name, shp in (("q", q.shape), ("k", k.shape), ("v", v.shape)):
        coords[name] = [tuple(int(rng.integers(0, n)) for n in shp) for _ in range(40)]
    _fd_check(q, k, v, do, 1 / math.sqrt(d), True, coords)


def test_backward_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    B, H, Hkv, N, d, s = 2, 6, 2, 29, 16, 0.125
    G = H // Hkv
    q, k, v, do = rand(B, H, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, H, N, d)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    kr, vr = tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1)
    S = s * tq @ kr.transpose(-1, -2)
    S = S.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    o = torch.softmax(S, -1) @ vr
    (o * torch.tensor(do)).sum().backward()
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, s, True)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_constant_v():
    B, H, Hkv, N, d = 1, 3, 1, 25, 8
    q, k, do = rand(B, H, N, d), rand(B, Hkv, N, d), rand(B, H, N, d)
    c = rand(d)
    v = np.broadcast_to(c, (B, Hkv, N, d)).copy()
    o, _ = oracle.attn_fwd(q, k, v, 0.4, True)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-13)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.4, True)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def test_n_equals_one():
    B, H, Hkv, d = 2, 4, 2, 8
    q, k, v, do = rand(B, H, 1, d), rand(B, Hkv, 1, d), rand(B, Hkv, 1, d), rand(B, H, 1, d)
    o, lse = oracle.attn_fwd(q, k, v, 0.5, True)
    np.testing.assert_allclose(o, np.repeat(v, 2, axis=1), rtol=0, atol=0)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0.5, True)
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0
    np.testing.assert_allclose(dv, do.reshape(B, Hkv, 2, 1, d).sum(2), rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal", [True, False])
def test_sum_identities(causal):
    """sum_j dV_j = sum over the group's heads and rows of dO; sum_j dK_j = 0
    (every dS row sums to zero); the two D forms agree."""
    B, H, Hkv, N, d = 2, 6, 2, 31, 8
    G = H // Hkv
    q, k, v, do = rand(B, H, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, H, N, d)
    dq, dk, dv, D, Dalt = oracle.attn_bwd(q, k, v, do, 0.3, causal, return_delta=True)
    np.testing.assert_allclose(dv.sum(2), do.reshape(B, Hkv, G, N, d).sum((2, 3)), atol=1e-11)
    np.testing.assert_allclose(dk.sum(2), 0.0, atol=1e-11)
    np.testing.assert_allclose(D, Dalt, rtol=1e-11, atol=1e-12)
    o, _ = oracle.attn_fwd(q, k, v, 0.3, causal)
    np.testing.assert_allclose(oracle.rowdot(o, do), D, rtol=1e-12, atol=1e-12)


def test_rowdot_matches_einsum():
    o, do = rand(3, 5, 7, 64), rand(3, 5, 7, 64)
    np.testing.assert_allclose(oracle.rowdot(o, do), np.einsum("abcd,abcd->abc", o, do),
                               rtol=1e-13, atol=1e-13)


def test_rejects_bad_group():
    with pytest.raises(ValueError):
        oracle.attn_fwd(rand(1, 3, 4, 8), rand(1, 2, 4, 8), rand(1, 2, 4, 8), 1.0, True)


@pytest.mark.parametrize("causal", [True, False])
def test_dq_rows_match_full_backward(causal):
    """The per-row dQ (used for long sequences) equals the full backward."""
    B, H, Hkv, N, d = 2, 6, 2, 37, 8
    q, k, v, do = rand(B, H, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, H, N, d)
    s = 1 / math.sqrt(d)
    dq, _, _ = oracle.attn_bwd(q, k, v, do, s, causal)
    rows = [(0, 0, 0), (0, 5, 36), (1, 3, 17), (1, 1, 1), (0, 2, 30)]
    got = oracle.attn_bwd_dq_rows(q, k, v, do, rows, s, causal)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(got[n], dq[b, h, i], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_dkdv_rows_match_full_backward(causal):
    """The per-key-row dK, dV (used for long sequences) equal the full backward."""
    B, H, Hkv, N, d = 1, 6, 2, 29, 8
    q, k, v, do = rand(B, H, N, d), rand(B, Hkv, N, d), rand(B, Hkv, N, d), rand(B, H, N, d)
    s = 1 / math.sqrt(d)
    _, dk, dv = oracle.attn_bwd(q, k, v, do, s, causal)
    rows = [(0, 0, 28), (0, 1, 27), (0, 1, 0), (0, 0, 13)]
    gk, gv = oracle.attn_bwd_dkdv_rows(q, k, v, do, rows, s, causal)
    for n, (b, g, j) in enumerate(rows):
        np.testing.assert_allclose(gk[n], dk[b, g, j], rtol=0, atol=1e-12)
        np.testing.assert_allclose(gv[n], dv[b, g, j], rtol=0, atol=1e-12)
