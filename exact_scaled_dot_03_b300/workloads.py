"""Seeded synthetic inputs for the attention workloads.

This module is shared by the tests, the benchmark and the smoke check. It only
draws random numbers and names shapes: it holds none of the attention
arithmetic, so the fp64 oracle and the CUDA path stay independent of each
other while reading bit-identical inputs.

Recipe (the same for every workload):
  * a CPU ``torch.Generator`` seeded with the workload's seed;
  * for decode, the per-sequence cache lengths are drawn first, uniform on the
    inclusive range [Lmin, Lmax];
  * then Q, K, V (or q, K cache, V cache) in that order, i.i.d. N(0, 1) in
    fp32, rounded to bf16 with round-to-nearest-even (``Tensor.to``).

Layouts are contiguous row-major: prefill Q/O ``[B, Hq, Nq, d]``, K/V
``[B, Hkv, Nk, d]``; decode q/o ``[B, Hq, d]``, caches ``[B, Hkv, Lmax, d]``.
Positions at or past ``seqlens[b]`` in the caches hold random data that a
correct decode never reads.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Prefill:
    """One prefill (or cross-attention) problem."""

    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        # 1/sqrt(d_k), rounded once to fp32: both sides use this same number.
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    def flops(self) -> float:
        """4*B*Hq*Nq*Nk*d (two contractions), halved when causal."""
        f = 4.0 * self.B * self.Hq * self.Nq * self.Nk * self.d
        return f / 2 if self.causal else f

    def io_bytes(self) -> int:
        """Q, K, V read once and O written once (bf16) plus the fp32 LSE."""
        qo = 2 * self.B * self.Hq * self.Nq * self.d * 2
        kv = 2 * self.B * self.Hkv * self.Nk * self.d * 2
        return qo + kv + 4 * self.B * self.Hq * self.Nq

    def with_(self, **kw) -> "Prefill":
        return replace(self, **kw)


@dataclass(frozen=True)
class Decode:
    """One KV-cache decode step: one new query token per sequence."""

    name: str
    B: int
    Hq: int
    Hkv: int
    Lmax: int
    Lmin: int
    d: int
    seed: int

    @property
    def scale(self) -> float:
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    def with_(self, **kw) -> "Decode":
        return replace(self, **kw)


# The five workloads; seeds 1001..1005 in this order.
SINGLE_HEAD = Prefill("single_head_n128_d64", B=1, Hq=1, Hkv=1, Nq=128, Nk=128, d=64,
                      causal=False, seed=1001)
MHA_2048 = Prefill("mha_b4_h12_n2048_d64", B=4, Hq=12, Hkv=12, Nq=2048, Nk=2048, d=64,
                   causal=False, seed=1002)
CAUSAL_MHA_4096 = Prefill("causal_mha_b2_h32_n4096_d128", B=2, Hq=32, Hkv=32, Nq=4096,
                          Nk=4096, d=128, causal=True, seed=1003)
CAUSAL_GQA_16384 = Prefill("causal_gqa_b1_hq64_hkv8_n16384_d128", B=1, Hq=64, Hkv=8,
                           Nq=16384, Nk=16384, d=128, causal=True, seed=1004)
DECODE_GQA = Decode("decode_b16_hq32_hkv8_d128_l1024to8192", B=16, Hq=32, Hkv=8, Lmax=8192,
                    Lmin=1024, d=128, seed=1005)

PREFILL_WORKLOADS = (SINGLE_HEAD, MHA_2048, CAUSAL_MHA_4096, CAUSAL_GQA_16384)


def _randn_bf16(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def prefill_inputs(w: Prefill):
    """(q, k, v) as contiguous CPU bf16 tensors, drawn in the order Q, K, V."""
    gen = torch.Generator().manual_seed(w.seed)
    q = _randn_bf16(gen, (w.B, w.Hq, w.Nq, w.d))
    k = _randn_bf16(gen, (w.B, w.Hkv, w.Nk, w.d))
    v = _randn_bf16(gen, (w.B, w.Hkv, w.Nk, w.d))
    return q, k, v


def backward_inputs(w: Prefill):
    """(q, k, v, dout) as contiguous CPU bf16 tensors: the prefill draw (Q, K, V),
    then dO = dL/dO from the same generator, all N(0, 1) rounded to bf16."""
    gen = torch.Generator().manual_seed(w.seed)
    q = _randn_bf16(gen, (w.B, w.Hq, w.Nq, w.d))
    k = _randn_bf16(gen, (w.B, w.Hkv, w.Nk, w.d))
    v = _randn_bf16(gen, (w.B, w.Hkv, w.Nk, w.d))
    dout = _randn_bf16(gen, (w.B, w.Hq, w.Nq, w.d))
    return q, k, v, dout


def decode_inputs(w: Decode):
    """(q, k_cache, v_cache, seqlens): lengths first, then q, K cache, V cache."""
    gen = torch.Generator().manual_seed(w.seed)
    seqlens = torch.randint(w.Lmin, w.Lmax + 1, (w.B,), generator=gen, dtype=torch.int64)
    seqlens = seqlens.to(torch.int32)
    q = _randn_bf16(gen, (w.B, w.Hq, w.d))
    kc = _randn_bf16(gen, (w.B, w.Hkv, w.Lmax, w.d))
    vc = _randn_bf16(gen, (w.B, w.Hkv, w.Lmax, w.d))
    return q, kc, vc, seqlens


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor as a numpy array (no rounding)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")


@dataclass(frozen=True)
class PagedDecode:
    """One decode step over a paged KV cache, optionally appending the new token."""

    name: str
    B: int
    Hq: int
    Hkv: int
    Lmin: int          # cached lengths uniform on [Lmin, Lmax] (before the append)
    Lmax: int
    d: int
    page_size: int
    append: bool
    seed: int

    @property
    def scale(self) -> float:
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    @property
    def max_pages(self) -> int:
        return (self.Lmax + 1 + self.page_size - 1) // self.page_size  # room for the appended token

    def with_(self, **kw) -> "PagedDecode":
        return replace(self, **kw)


def paged_decode_inputs(w: PagedDecode, lens=None):
    """(q, k_new, v_new, k_pages, v_pages, block_table, seqlens), CPU tensors.

    Draw order: cached lengths, q, k_new, v_new, the K page pool, the V page
    pool, then a random permutation that hands out physical pages. Each
    sequence gets the pages for its cached tokens plus the appended one; its
    remaining block-table entries point at page 0. The pool has a few spare
    pages so that not every page is in use.
    """
    gen = torch.Generator().manual_seed(w.seed)
    seqlens = torch.randint(w.Lmin, w.Lmax + 1, (w.B,), generator=gen, dtype=torch.int64).to(torch.int32)
    if lens is not None:
        seqlens = torch.tensor(lens, dtype=torch.int32)
    P = w.page_size
    need = [(int(L) + 1 + P - 1) // P for L in seqlens]
    num_pages = sum(need) + 3
    q = _randn_bf16(gen, (w.B, w.Hq, w.d))
    k_new = _randn_bf16(gen, (w.B, w.Hkv, w.d))
    v_new = _randn_bf16(gen, (w.B, w.Hkv, w.d))
    k_pages = _randn_bf16(gen, (num_pages, w.Hkv, P, w.d))
    v_pages = _randn_bf16(gen, (num_pages, w.Hkv, P, w.d))
    perm = torch.randperm(num_pages, generator=gen).to(torch.int32)
    block_table = torch.zeros(w.B, w.max_pages, dtype=torch.int32)
    nxt = 0
    for b in range(w.B):
        block_table[b, :need[b]] = perm[nxt:nxt + need[b]]
        nxt += need[b]
    if not w.append:
        k_new = v_new = None
    return q, k_new, v_new, k_pages, v_pages, block_table, seqlens


# Paged form of the decode workload: the same shapes and length mix, 64-token
# pages, the new token appended.
DECODE_GQA_PAGED = PagedDecode("decode_paged_b16_hq32_hkv8_d128_l1024to8192_p64", B=16, Hq=32, Hkv=8, Lmin=1024,
                               Lmax=8192, d=128, page_size=64, append=True, seed=1006)
