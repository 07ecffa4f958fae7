"""Seeded synthetic inputs for causal grouped-query attention.

This module holds no attention arithmetic: it only names the workload shapes
and draws random tensors.  Both the CUDA path and the fp64 oracle take their
inputs from here, so neither generates data for the other.

Shapes follow the GPT-2-small attention of "NanoEuler: Hand-writing GPT-2 in
Pure C/CUDA", section "Build and Run" (the config file: hidden 768, 12 query
heads, 4 KV heads, max_seq_len 1024, batch 8, hence head_dim 64), plus a
long-context and a wide-head variant.  The post trains on FineWeb-Edu /
OpenWebText; attention only sees Q/K/V/dO tensors of these shapes, so seeded
Gaussian / uniform tensors stand in for activations.

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` draws Q, K, V, dO in
that order, in fp32, each with the workload's distribution; the result is then
rounded to the workload dtype (bf16 or fp32).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    dtype: str          # "bf16" or "f32"
    qk_std: float = 1.0  # Q, K ~ N(0, qk_std^2)
    vdo: str = "normal"  # V, dO ~ N(0,1) ("normal") or U(-1,1) ("uniform")
    causal: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def causal_pairs(self) -> int:
        """(i, j) score pairs with j <= i, summed over batch and heads."""
        per_head = self.N * (self.N + 1) // 2 if self.causal else self.N * self.N
        return self.B * self.H * per_head

    def fwd_flops(self) -> float:
        """FlashAttention convention: 4*d flops per unmasked score pair, causal
        counted as half of the dense B*H*N^2 (the N(N+1)/2 exact-pair count
        differs by a factor 1 + 1/N)."""
        dense = 4.0 * self.B * self.H * self.N * self.N * self.d
        return dense / 2 if self.causal else dense

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 2, 1, 128, 64, "f32"),
    "gpt2s_bf16": Workload("gpt2s_bf16", 8, 12, 4, 1024, 64, "bf16"),
    "gpt2s_f32": Workload("gpt2s_f32", 8, 12, 4, 1024, 64, "f32"),
    "long_bf16": Workload("long_bf16", 2, 12, 4, 4096, 64, "bf16", vdo="uniform"),
    "wide_bf16": Workload("wide_bf16", 4, 16, 4, 2048, 128, "bf16", qk_std=2.0),
}


def make_inputs(w: Workload, seed: int = 0, device=None):
    """Return (q, k, v, do) on ``device`` (CPU if None), in ``w``'s dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    qshape = (w.B, w.H, w.N, w.d)
    kshape = (w.B, w.Hkv, w.N, w.d)

    def qk(shape):
        return torch.randn(shape, generator=g, dtype=torch.float32) * w.qk_std

    def vd(shape):
        if w.vdo == "uniform":
            return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
        return torch.randn(shape, generator=g, dtype=torch.float32)

    q = qk(qshape)
    k = qk(kshape)
    v = vd(kshape)
    do = vd(qshape)
    out = [t.to(w.torch_dtype).contiguous() for t in (q, k, v, do)]
    if device is not None:
        out = [t.to(device) for t in out]
    return tuple(out)


def custom(B, H, Hkv, N, d, dtype="bf16", causal=True, qk_std=1.0, vdo="normal") -> Workload:
    return Workload(f"B{B}_H{H}_Hkv{Hkv}_N{N}_d{d}_{dtype}{'' if causal else '_full'}",
                    B, H, Hkv, N, d, dtype, qk_std, vdo, causal)


@dataclass(frozen=True)
class DecodeWorkload:
    """One decode step: the newest nq tokens of B sequences against a cache of
    Lmax rows per sequence, lens[b] of them valid (new tokens included)."""
    name: str
    B: int
    H: int
    Hkv: int
    nq: int
    Lmax: int
    d: int
    dtype: str
    lens: tuple = ()     # empty: every sequence fills the cache (lens[b] = Lmax)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def lengths(self):
        return list(self.lens) if self.lens else [self.Lmax] * self.B

    def cache_bytes(self) -> int:
        """K and V rows the step must read (the valid ones), in bytes."""
        return 2 * self.Hkv * sum(self.lengths()) * self.d * self.esize


DECODE_WORKLOADS = {
    # one generated token per sequence at the training shape's full context
    "decode_gpt2s_bf16": DecodeWorkload("decode_gpt2s_bf16", 8, 12, 4, 1, 1024, 64, "bf16"),
    # a long cache, large enough to be bound by HBM bandwidth
    "decode_long_bf16": DecodeWorkload("decode_long_bf16", 32, 12, 4, 1, 16384, 64, "bf16"),
}


def make_decode_inputs(w: DecodeWorkload, seed: int = 0, device=None):
    """Return (q, k_cache, v_cache, lens): q [B,H,nq,d], caches [B,Hkv,Lmax,d]
    drawn N(0,1) in that order from a CPU generator seeded with ``seed``, then
    rounded to the dtype; lens [B] int32."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((w.B, w.H, w.nq, w.d), generator=g, dtype=torch.float32)
    kc = torch.randn((w.B, w.Hkv, w.Lmax, w.d), generator=g, dtype=torch.float32)
    vc = torch.randn((w.B, w.Hkv, w.Lmax, w.d), generator=g, dtype=torch.float32)
    lens = torch.tensor(w.lengths(), dtype=torch.int32)
    out = [t.to(w.torch_dtype).contiguous() for t in (q, kc, vc)] + [lens]
    if device is not None:
        out = [t.to(device) for t in out]
    return tuple(out)
