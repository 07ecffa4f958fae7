"""GPU parity of decode attention (nea_attn_decode) against the fp64 oracle.

Tolerances: bf16 (inputs exact in fp64, fp32 arithmetic, output rounded to
bf16 once): O max-abs <= 2e-2, LSE max-abs <= 1e-3.  fp32 (all fp32 CUDA-core
arithmetic, sums of at most Lmax terms): O relative L2 <= 1e-5, LSE max-abs
<= 1e-5.  Cases: ragged cache lengths from 1 row to the whole cache, several
new tokens per sequence, grouped and plain heads, d = 64 and 128, and the
GPT-2-small decode step; caches of at most 16 chunks of 128 rows (one
launch, one CTA per (batch, KV head)) and longer ones (split, then combine).
"""
import numpy as np
import pytest
import torch

import oracle
from causal_gqa_flashattention_gb300.workloads import (DECODE_WORKLOADS, DecodeWorkload,
                                                        make_decode_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nea(cuda_device):
    from causal_gqa_flashattention_gb300 import build, nea as binding
    build.build()
    binding.lib()
    return binding


CASES = [
    DecodeWorkload("ragged_nq1", 4, 12, 4, 1, 1024, 64, "bf16", (1, 77, 1000, 1024)),
    DecodeWorkload("nq4_d128", 2, 8, 2, 4, 300, 128, "bf16", (4, 300)),
    DecodeWorkload("mha_f32", 3, 6, 6, 2, 4096, 64, "f32", (4096, 129, 2)),
    DecodeWorkload("gqa8_f32_d128", 2, 16, 2, 2, 640, 128, "f32", (640, 257)),
    DECODE_WORKLOADS["decode_gpt2s_bf16"],
    # past 16 chunks of 128 rows: split over the cache, then the combine
    DecodeWorkload("split_bf16_nq2", 2, 12, 4, 2, 6144, 64, "bf16", (6144, 2050)),
    DecodeWorkload("split_bf16_d128", 1, 8, 2, 1, 2177, 128, "bf16", (2177,)),
    # 32 query rows per KV head (G = 8, nq = 4), short and long caches
    DecodeWorkload("rows32_cluster", 1, 16, 2, 4, 900, 64, "bf16", (900,)),
    DecodeWorkload("rows32_split", 2, 16, 2, 4, 4096, 64, "bf16", (4096, 1500)),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_decode_matches_oracle(nea, w):
    dev = torch.device("cuda:0")
    q, kc, vc, lens = make_decode_inputs(w, seed=2, device=dev)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.nq), float("nan"), device=dev)
    nea.attn_decode(q, kc, vc, lens, scale=w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert nea.check_status() == 0
    ro, rl = oracle.attn_decode(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu().numpy(), w.scale)
    got_o = o.float().cpu().numpy().astype(np.float64)
    got_l = lse.cpu().numpy().astype(np.float64)
    assert np.isfinite(got_o).all() and np.isfinite(got_l).all()
    if w.dtype == "bf16":
        assert np.abs(got_o - ro).max() <= 2e-2
        assert np.abs(got_l - rl).max() <= 1e-3
    else:
        assert np.linalg.norm(got_o - ro) / np.linalg.norm(ro) <= 1e-5
        assert np.abs(got_l - rl).max() <= 1e-5


def test_cache_rows_past_length_are_not_read(nea):
    w = DecodeWorkload("nan_tail", 2, 6, 2, 2, 512, 64, "bf16", (300, 130))
    dev = torch.device("cuda:0")
    q, kc, vc, lens = make_decode_inputs(w, seed=4, device=dev)
    o1, l1 = nea.attn_decode(q, kc, vc, lens)
    for b, L in enumerate(w.lens):
        kc[b, :, L:] = float("nan")
        vc[b, :, L:] = float("nan")
    o2, l2 = nea.attn_decode(q, kc, vc, lens)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_out_of_range_length_is_reported(nea):
    w = DecodeWorkload("bad_len", 2, 4, 2, 2, 256, 64, "bf16", (256, 200))
    dev = torch.device("cuda:0")
    q, kc, vc, lens = make_decode_inputs(w, seed=6, device=dev)
    nea.check_status()
    bad = torch.tensor([1, 300], dtype=torch.int32, device=dev)  # < nq and > Lmax
    nea.attn_decode(q, kc, vc, bad)
    assert nea.check_status() == nea.NEA_ERR_INVALID
    nea.attn_decode(q, kc, vc, lens)
    assert nea.check_status() == 0
