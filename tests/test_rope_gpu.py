"""GPU parity of the rotary embedding path against the fp64 oracle.

- nea_rope_table + nea_rope_qk against oracle.rope: the GPU result is the
  fp32 rotation rounded once to the dtype, so each element must lie within
  one unit in the last place of the dtype (bf16: 2^-8 relative) of the fp64
  value, plus the fp32 table's rounding (absolute 2e-6 * |row|);
- nea_attn_bwd_rope against the oracle composition: the backward on the
  GPU's own rotated Qr, Kr, then the inverse rotation of dQ and dK, within
  the backward tolerances (bf16: relative L2 1e-2; fp32: 5e-3).
"""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_flashattention_gb300.workloads import custom, make_inputs

pytestmark = pytest.mark.gpu


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


def check_rotation(got, x, base, dtype):
    ref = oracle.rope(x.cpu(), base=base)
    g = got.detach().float().cpu().numpy().astype(np.float64)
    ulp = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -23
    rown = np.sqrt((ref ** 2).sum(-1, keepdims=True))
    bound = ulp * np.abs(ref) + 2e-6 * rown + 1e-30
    excess = np.abs(g - ref) - bound
    assert excess.max() <= 0, float(excess.max())


@pytest.mark.parametrize("w,base", [
    (custom(2, 6, 2, 384, 64), 10000.0),
    (custom(1, 4, 2, 300, 128, causal=False), 10000.0),
    (custom(1, 3, 1, 4096, 64), 500000.0),
    (custom(1, 4, 2, 200, 64, "f32"), 10000.0),
], ids=lambda x: getattr(x, "name", str(x)))
def test_rotation_matches_oracle(nea, w, base):
    dev = torch.device("cuda:0")
    q, k, _, _ = make_inputs(w, seed=3, device=dev)
    cs = nea.rope_table(w.N, w.d, base=base, device=dev)
    qr, kr = nea.rope_qk(q, k, cs)
    torch.cuda.synchronize()
    check_rotation(qr, q, base, w.dtype)
    check_rotation(kr, k, base, w.dtype)
    # in place gives the same bits
    q2, k2 = q.clone(), k.clone()
    nea.rope_qk(q2, k2, cs, qr=q2, kr=k2)
    torch.cuda.synchronize()
    assert torch.equal(q2, qr) and torch.equal(k2, kr)


@pytest.mark.parametrize("w", [
    custom(1, 6, 2, 384, 64),
    custom(1, 4, 2, 300, 128, causal=False),
    custom(2, 4, 4, 129, 64),
    custom(1, 4, 2, 256, 64, "f32"),
    custom(8, 12, 4, 1024, 64),
], ids=lambda w: w.name)
def test_backward_through_rotation(nea, w):
    dev = torch.device("cuda:0")
    q, k, v, do = make_inputs(w, seed=5, device=dev)
    cs = nea.rope_table(w.N, w.d, device=dev)
    qr, kr = nea.rope_qk(q, k, cs)
    o, lse = nea.attn_fwd(qr, kr, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = nea.attn_bwd(qr, kr, v, o, do, lse, causal=w.causal, scale=w.scale, rope_cs=cs)
    torch.cuda.synchronize()
    assert nea.check_status() == 0
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    dqr, dkr, rdv = oracle.attn_bwd(qr.cpu(), kr.cpu(), v.cpu(), do.cpu(), w.scale, w.causal)
    rdq = oracle.rope(dqr, inverse=True)
    rdk = oracle.rope(dkr, inverse=True)
    tol = 1e-2 if w.dtype == "bf16" else 5e-3
    errs = dict(dq=rel_l2(dq, rdq), dk=rel_l2(dk, rdk), dv=rel_l2(dv, rdv))
    assert max(errs.values()) <= tol, errs
    # the unrotated gradients differ from the rotated ones (the mapping ran)
    assert rel_l2(dq, dqr) > 0.05 and rel_l2(dk, dkr) > 0.05


@pytest.mark.parametrize("w", [custom(2, 6, 2, 384, 64), custom(1, 4, 2, 300, 128, causal=False),
                               custom(1, 3, 1, 77, 64), custom(4, 12, 4, 1000, 64)],
                         ids=lambda w: w.name)
def test_forward_rotating_q_in_kernel(nea, w):
    """nea_attn_fwd_rope_q (Q rotated in shared memory, K by the pass): bit-
    identical to the forward on the pass's rotated Q (the same fp32
    arithmetic and one rounding to bf16 feed the same MMAs), and, like every
    forward, within the forward tolerances (O max-abs 2e-2, LSE max-abs 1e-3)
    of the oracle on the same bf16 inputs: the pass's Qr and Kr, which
    test_rotation_matches_oracle pins to oracle.rope within one bf16 ulp."""
    dev = torch.device("cuda:0")
    q, k, v, _ = make_inputs(w, seed=5, device=dev)
    cs = nea.rope_table(w.N, w.d, device=dev)
    qr, kr = nea.rope_qk(q, k, cs)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.N), float("nan"), device=dev)
    nea.attn_fwd(q, kr, v, causal=w.causal, scale=w.scale, out=o, lse=lse, rope_q_cs=cs)
    o2, lse2 = nea.attn_fwd(qr, kr, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert nea.check_status() == 0
    ro, rlse = oracle.attn_fwd(qr.cpu(), kr.cpu(), v.cpu(), w.scale, w.causal)
    og = o.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(og).all()
    assert np.abs(og - ro).max() <= 2e-2
    assert np.abs(lse.cpu().numpy().astype(np.float64) - rlse).max() <= 1e-3
    # the in-kernel rotation rounds exactly like the pass: same inputs to the MMAs
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
