"""Pins of the oracle's decode attention (``oracle.attn_decode``).

Reading taken (the pages say only that inference works): each batch element
has a contiguous cache of lens[b] rows that already holds the nq new tokens;
new token t sits at position lens[b] - nq + t and sees cache rows up to it.
Pinned by facts that do not come from the decode code itself:
- it equals the last nq rows of the (separately pinned) causal forward run on
  the first lens[b] rows of the sequence;
- closed forms: q = 0 gives the mean of the visible V rows and LSE = ln(count);
  one visible row gives O = V_0, LSE = scale * q . k_0;
- cache rows past lens[b], and rows after a token's own position, do not
  take part (NaN there changes nothing; perturbing them changes only later
  tokens);
- grouped heads read KV head h / (H / Hkv): equal to MHA on repeated K/V.
"""
import math

import numpy as np
import pytest

import oracle

rng = np.random.default_rng(99)


def make(B, H, Hkv, nq, Lmax, d):
    return (rng.standard_normal((B, H, nq, d)), rng.standard_normal((B, Hkv, Lmax, d)),
            rng.standard_normal((B, Hkv, Lmax, d)))


def test_equals_last_rows_of_causal_forward():
    B, H, Hkv, nq, Lmax, d = 3, 6, 2, 3, 50, 8
    q, kc, vc = make(B, H, Hkv, nq, Lmax, d)
    lens = [50, 17, 3]
    s = 1 / math.sqrt(d)
    o, lse = oracle.attn_decode(q, kc, vc, lens, s)
    for b, L in enumerate(lens):
        qf = rng.standard_normal((1, H, L, d))
        qf[0, :, L - nq:] = q[b]
        of, lf = oracle.attn_fwd(qf, kc[b:b + 1, :, :L], vc[b:b + 1, :, :L], s, True)
        np.testing.assert_allclose(o[b], of[0, :, L - nq:], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], lf[0, :, L - nq:], rtol=0, atol=1e-12)


def test_zero_query_closed_form():
    B, H, Hkv, nq, Lmax, d = 2, 4, 2, 2, 20, 4
    _, kc, vc = make(B, H, Hkv, nq, Lmax, d)
    q = np.zeros((B, H, nq, d))
    lens = [20, 9]
    o, lse = oracle.attn_decode(q, kc, vc, lens, 0.5)
    for b, L in enumerate(lens):
        for h in range(H):
            for t in range(nq):
                cnt = L - nq + t + 1
                np.testing.assert_allclose(o[b, h, t], vc[b, h // 2, :cnt].mean(0), atol=1e-13)
                assert abs(lse[b, h, t] - math.log(cnt)) < 1e-13


def test_single_visible_row():
    q, kc, vc = make(1, 2, 1, 1, 5, 4)
    o, lse = oracle.attn_decode(q, kc, vc, [1], 0.7)
    for h in range(2):
        np.testing.assert_allclose(o[0, h, 0], vc[0, 0, 0], atol=1e-15)
        assert abs(lse[0, h, 0] - 0.7 * q[0, h, 0] @ kc[0, 0, 0]) < 1e-13


def test_rows_past_length_and_position_do_not_take_part():
    B, H, Hkv, nq, Lmax, d = 1, 2, 1, 3, 12, 4
    q, kc, vc = make(B, H, Hkv, nq, Lmax, d)
    L = 9
    o1, l1 = oracle.attn_decode(q, kc, vc, [L], 0.5)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, :, L:] = np.nan
    vc2[:, :, L:] = np.nan
    o2, l2 = oracle.attn_decode(q, kc2, vc2, [L], 0.5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # row L-2 is the position of token 1: token 0 must not see it, token 1 must
    kc3 = kc.copy()
    kc3[0, 0, L - 2] += 3.0
    o3, _ = oracle.attn_decode(q, kc3, vc, [L], 0.5)
    np.testing.assert_array_equal(o3[:, :, 0], o1[:, :, 0])
    assert np.abs(o3[:, :, 1] - o1[:, :, 1]).max() > 1e-6


def test_gqa_equals_mha_with_repeated_cache():
    B, H, Hkv, nq, Lmax, d = 2, 6, 2, 2, 15, 8
    q, kc, vc = make(B, H, Hkv, nq, Lmax, d)
    lens = [15, 6]
    o, lse = oracle.attn_decode(q, kc, vc, lens, 0.3)
    om, lm = oracle.attn_decode(q, np.repeat(kc, 3, axis=1), np.repeat(vc, 3, axis=1), lens, 0.3)
    np.testing.assert_allclose(o, om, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lm, rtol=0, atol=1e-13)


def test_rejects_bad_lengths():
    q, kc, vc = make(1, 2, 1, 3, 8, 4)
    with pytest.raises(ValueError):
        oracle.attn_decode(q, kc, vc, [2], 0.5)     # fewer rows than new tokens
    with pytest.raises(ValueError):
        oracle.attn_decode(q, kc, vc, [9], 0.5)     # longer than the cache
