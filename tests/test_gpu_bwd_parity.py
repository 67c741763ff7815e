"""Attention backward (dQ, dK, dV): CUDA path vs the fp64 oracle.

The GPU forward supplies o and the LSE, as a training step would; the oracle
differentiates the forward definition directly from q, k, v and dO. Small
problems are compared over every gradient element (several tiles, ragged
tails, GQA/MQA, Nq != Nk, rows that see no key); the full-size workloads on
sampled query rows (dQ is row-wise) and sampled key rows (dK, dV need every
query that sees the key), plus invariants that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_03_b300 import binding
from exact_scaled_dot_03_b300.workloads import CAUSAL_GQA_16384, CAUSAL_MHA_4096, Prefill, backward_inputs
from tests.parity import BF16_U, compare_grad, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _fwd_bwd(q, k, v, do, causal, scale):
    q, k, v, do = (t.to(DEV) for t in (q, k, v, do))
    o, lse = binding.fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    st = binding.device_status()
    assert st[0] == 0, st
    return dq, dk, dv


SMALL = [
    Prefill("bwd_mha_d64_n384", B=2, Hq=4, Hkv=4, Nq=384, Nk=384, d=64, causal=False, seed=31),
    Prefill("bwd_causal_gqa_ragged_n333", B=1, Hq=8, Hkv=2, Nq=333, Nk=333, d=128, causal=True, seed=32),
    Prefill("bwd_causal_mqa_d64_n520", B=2, Hq=3, Hkv=1, Nq=520, Nk=520, d=64, causal=True, seed=33),
    Prefill("bwd_cross_nq200_nk520", B=1, Hq=4, Hkv=2, Nq=200, Nk=520, d=128, causal=False, seed=34),
    Prefill("bwd_cross_causal_nq200_nk520", B=1, Hq=4, Hkv=2, Nq=200, Nk=520, d=128, causal=True, seed=35),
    Prefill("bwd_cross_causal_nq300_nk130", B=1, Hq=2, Hkv=2, Nq=300, Nk=130, d=64, causal=True, seed=36),
    Prefill("bwd_n1", B=3, Hq=2, Hkv=1, Nq=1, Nk=1, d=128, causal=True, seed=37),
    Prefill("bwd_n129", B=1, Hq=2, Hkv=2, Nq=129, Nk=129, d=128, causal=True, seed=38),
    Prefill("bwd_mha_d128_n1024", B=1, Hq=2, Hkv=2, Nq=1024, Nk=1024, d=128, causal=False, seed=39),
    Prefill("bwd_causal_gqa8_n1000", B=1, Hq=16, Hkv=2, Nq=1000, Nk=1000, d=128, causal=True, seed=40),
    Prefill("bwd_gqa_hkv3_n300", B=2, Hq=6, Hkv=3, Nq=300, Nk=300, d=128, causal=True, seed=43),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_full_gradients(w):
    q, k, v, do = backward_inputs(w)
    dq, dk, dv = _fwd_bwd(q, k, v, do, w.causal, w.scale)
    *ref, m = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), w.scale, w.causal, magnitudes=True)
    for name, g, r, t, sd in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, (m["tq"], m["tk"], m["tv"]),
                                 (m["sq"], m["sk"], None)):
        res = compare_grad(g, r, t, sd, f"{w.name} {name}")
        print(w.name, name, res)
    if w.causal and w.Nq > w.Nk:  # rows that see no key get dq = 0
        assert (dq[:, :, : w.Nq - w.Nk] == 0).all()


def test_large_scores():
    """Scores of magnitude ~50 (a peaked softmax, P near 0 or 1)."""
    w = Prefill("bwd_big_scores", B=1, Hq=2, Hkv=1, Nq=300, Nk=700, d=128, causal=False, seed=41)
    q, k, v, do = backward_inputs(w)
    q = (q.float() * 4.0).to(torch.bfloat16)
    for causal in (False, True):
        dq, dk, dv = _fwd_bwd(q, k, v, do, causal, w.scale)
        *ref, m = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), w.scale, causal, magnitudes=True)
        for name, g, r, t, sd in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, (m["tq"], m["tk"], m["tv"]),
                                     (m["sq"], m["sk"], None)):
            print("big", causal, name, compare_grad(g, r, t, sd, f"big scores causal={causal} {name}"))


def test_deterministic():
    """No atomics: two calls give bit-identical gradients."""
    w = Prefill("bwd_repeat", B=1, Hq=8, Hkv=2, Nq=700, Nk=700, d=128, causal=True, seed=42)
    q, k, v, do = (t.to(DEV) for t in backward_inputs(w))
    o, lse = binding.fwd(q, k, v, causal=True, scale=w.scale)
    a = binding.bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    b = binding.bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_no_queries_or_no_keys():
    q = torch.randn(1, 2, 40, 64, device=DEV).to(torch.bfloat16)
    k0 = torch.empty(1, 1, 0, 64, device=DEV, dtype=torch.bfloat16)
    o, lse = binding.fwd(q, k0, k0, causal=False)
    dq, dk, dv = binding.bwd(q, k0, k0, o, lse, torch.randn_like(q), causal=False)
    q0 = torch.empty(1, 2, 0, 64, device=DEV, dtype=torch.bfloat16)
    k = torch.randn(1, 1, 50, 64, device=DEV).to(torch.bfloat16)
    lse0 = torch.empty(1, 2, 0, device=DEV)
    dq2, dk2, dv2 = binding.bwd(q0, k, k, q0, lse0, q0, causal=True)
    torch.cuda.synchronize()
    assert (dq == 0).all() and dk.numel() == 0
    assert dq2.numel() == 0 and (dk2 == 0).all() and (dv2 == 0).all()


def _full_size(w, q_samples, key_check):
    q, k, v, do = (t.to(DEV) for t in backward_inputs(w))
    o, lse = binding.fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert binding.device_status()[0] == 0
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    # dQ on sampled rows of sampled heads: row-wise, so the oracle is exact on them
    for (b, h, rows) in q_samples:
        g = h // (w.Hq // w.Hkv)
        ref, _, _, m = oracle.attention_backward(
            f64(q[b:b + 1, h:h + 1]), f64(k[b:b + 1, g:g + 1]), f64(v[b:b + 1, g:g + 1]), f64(do[b:b + 1, h:h + 1]),
            w.scale, w.causal, q_rows=rows, k_rows=np.array([], dtype=np.int64), magnitudes=True)
        print(w.name, "dq", b, h,
              compare_grad(dq[b:b + 1, h:h + 1, rows], ref, m["tq"], m["sq"], f"{w.name} dq b={b} h={h}"))
    key_check(q, k, v, do, dk, dv)
    # sum_j dK_j = 0 and sum_j dV_j = sum over the group's rows of dO, at any
    # size. Each row carries independent rounding errors of order u |row|, so
    # the sum's error grows like their root-sum-square: 4 u times it for the
    # bf16 rounding of P, dS and the outputs, and as much again for Dl, whose
    # error (from the bf16 forward output) enters sum_j dK_j as
    # scale sum_i dDl_i q_i, a random walk of the same order over the rows.
    G = w.Hq // w.Hkv
    for name, g, want in (("dk", dk, torch.zeros(w.B, w.Hkv, w.d, device=DEV, dtype=torch.float64)),
                          ("dv", dv, do.double().reshape(w.B, w.Hkv, G * w.Nq, w.d).sum(dim=2))):
        rss = g.double().pow(2).sum(dim=2).sqrt()
        dev = (g.double().sum(dim=2) - want).abs()
        print(w.name, name, "sum invariant: worst deviation / (8u rss)", (dev / (8 * BF16_U * rss)).max().item())
        assert (dev <= 8 * BF16_U * rss).all(), name


def test_causal_mha_4096_sampled():
    w = CAUSAL_MHA_4096
    rng = np.random.default_rng(50)

    def key_check(q, k, v, do, dk, dv):
        # every key row of one head needs all queries of that head: one head per batch
        for b, h in ((0, 5), (1, 30)):
            rows = np.sort(rng.choice(w.Nk, 96, replace=False))
            _, rk, rv, m = oracle.attention_backward(
                f64(q[b:b + 1, h:h + 1]), f64(k[b:b + 1, h:h + 1]), f64(v[b:b + 1, h:h + 1]),
                f64(do[b:b + 1, h:h + 1]), w.scale, True, q_rows=np.array([], dtype=np.int64), k_rows=rows,
                magnitudes=True)
            print(w.name, "dk", b, h,
                  compare_grad(dk[b:b + 1, h:h + 1, rows], rk, m["tk"], m["sk"], f"{w.name} dk b={b} h={h}"))
            print(w.name, "dv", b, h,
                  compare_grad(dv[b:b + 1, h:h + 1, rows], rv, m["tv"], None, f"{w.name} dv b={b} h={h}"))

    samples = [(0, 0, np.sort(rng.choice(w.Nq, 64, replace=False))),
               (1, 17, np.concatenate([np.arange(8), np.arange(w.Nq - 8, w.Nq)]))]
    _full_size(w, samples, key_check)


def test_causal_gqa_16384_sampled():
    w = CAUSAL_GQA_16384
    rng = np.random.default_rng(51)

    def key_check(q, k, v, do, dk, dv):
        # keys of the last tile are seen only by the last 128 query rows (of all
        # 8 heads of the group), so slicing the queries to those rows keeps every
        # contribution and the bottom-right alignment keeps their positions
        t0 = w.Nk - 128
        for g in (0, 7):
            hs = slice(g * 8, g * 8 + 8)
            _, rk, rv, m = oracle.attention_backward(
                f64(q[:, hs, t0:]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1]), f64(do[:, hs, t0:]), w.scale, True,
                q_rows=np.array([], dtype=np.int64), k_rows=np.arange(t0, w.Nk), magnitudes=True)
            print(w.name, "dk last tile", g,
                  compare_grad(dk[:, g:g + 1, t0:], rk, m["tk"], m["sk"], f"{w.name} dk last tile kv={g}"))
            print(w.name, "dv last tile", g,
                  compare_grad(dv[:, g:g + 1, t0:], rv, m["tv"], None, f"{w.name} dv last tile kv={g}"))
        # key tile 0 is the heaviest: every query row of the 8 heads of its group
        # (131 072 rows) adds to it, so it carries the most accumulated rounding;
        # the oracle takes every row in full (row-blocked), about a minute on the host
        g = 0
        hs = slice(0, 8)
        _, rk, rv, m = oracle.attention_backward(
            f64(q[:, hs]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1]), f64(do[:, hs]), w.scale, True,
            q_rows=np.array([], dtype=np.int64), k_rows=np.arange(128), row_block=2048, magnitudes=True)
        print(w.name, "dk first tile", g,
              compare_grad(dk[:, g:g + 1, :128], rk, m["tk"], m["sk"], f"{w.name} dk first tile kv={g}"))
        print(w.name, "dv first tile", g,
              compare_grad(dv[:, g:g + 1, :128], rv, m["tv"], None, f"{w.name} dv first tile kv={g}"))

    samples = [(0, 3, np.sort(rng.choice(w.Nq, 48, replace=False))),
               (0, 60, np.concatenate([np.arange(4), np.arange(w.Nq - 4, w.Nq)]))]
    _full_size(w, samples, key_check)


def test_calls_on_two_streams_back_to_back():
    """Two backward calls queued on two streams before any synchronisation share
    the library's dQ stream and events: each must return the bits it returns
    when run alone."""
    wa = Prefill("bwd_stream_a", B=1, Hq=4, Hkv=2, Nq=640, Nk=640, d=128, causal=True, seed=44)
    wb = Prefill("bwd_stream_b", B=2, Hq=2, Hkv=1, Nq=300, Nk=500, d=64, causal=True, seed=45)
    cases = []
    for w in (wa, wb):
        q, k, v, do = (t.to(DEV) for t in backward_inputs(w))
        o, lse = binding.fwd(q, k, v, causal=w.causal, scale=w.scale)
        alone = binding.bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
        torch.cuda.synchronize()
        cases.append((w, (q, k, v, o, lse, do), [t.clone() for t in alone]))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    results = []
    for (w, (q, k, v, o, lse, do), _), st in zip(cases, streams):
        with torch.cuda.stream(st):
            results.append(binding.bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale))
    torch.cuda.synchronize()
    assert binding.device_status()[0] == binding.OK
    for (w, _, alone), got in zip(cases, results):
        for name, a, g in zip(("dq", "dk", "dv"), alone, got):
            assert torch.equal(a, g), f"{w.name} {name}"
