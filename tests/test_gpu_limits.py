"""Sizes at and near the limits of the entry points: long sequences, the largest
batch the launch grid takes, thousands of heads or sequences. Each case is
compared with the fp64 oracle: on sampled rows where the full output would be
too slow on the host (the definitions are row-wise, so a row is exact), or on
a subset of whole batches and heads.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_03_b300 import binding
from exact_scaled_dot_03_b300.workloads import Decode, Prefill, backward_inputs, decode_inputs, prefill_inputs
from tests.parity import BF16_U, compare, compare_grad, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
LONG = Prefill("causal_n131072_d128", B=1, Hq=2, Hkv=1, Nq=131072, Nk=131072, d=128, causal=True, seed=81)
LONG_ROWS = np.array([0, 1, 127, 128, 4095, 4096, 65535, 65536, 100000, 131070, 131071])


def _sampled(q, k, v, o, lse, w, rows, what, window=0):
    for h in range(w.Hq):
        g = h // (w.Hq // w.Hkv)
        o_ref, lse_ref = oracle.attention_forward(f64(q[:, h:h + 1]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1]),
                                                  w.scale, w.causal, rows=rows, window=window)
        compare(o[:, h:h + 1, rows], lse[:, h:h + 1, rows], o_ref, lse_ref, f"{what} head {h}")


def test_prefill_128k_tokens():
    """A causal prefill over 131 072 tokens (1024 key tiles per late row) and the
    same with a 4096-key window, on rows at the tile edges and the ends."""
    q, k, v = prefill_inputs(LONG)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    for window in (0, 4096):
        o, lse = binding.fwd(qd, kd, vd, causal=True, scale=LONG.scale, window=window)
        torch.cuda.synchronize()
        assert binding.device_status()[0] == binding.OK
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        _sampled(q, k, v, o.cpu(), lse.cpu(), LONG, LONG_ROWS, f"N=131072 window={window}", window=window)


def test_rope_prefill_128k_positions():
    """Rotary embedding at positions up to 131 071 (angles up to ~1.3e5 rad),
    where the angle reduction must stay exact."""
    q, k, v = prefill_inputs(LONG)
    o, lse = binding.fwd_rope(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=LONG.scale, base=10000.0)
    torch.cuda.synchronize()
    assert binding.device_status()[0] == binding.OK
    rows = LONG_ROWS
    for h in range(LONG.Hq):
        o_ref, lse_ref = oracle.attention_forward_rope(f64(q[:, h:h + 1]), f64(k), f64(v), LONG.scale, True,
                                                       base=10000.0, rows=rows)
        compare(o.cpu()[:, h:h + 1, rows], lse.cpu()[:, h:h + 1, rows], o_ref, lse_ref, f"rope N=131072 head {h}")


def test_prefill_largest_batch():
    """B = 65535, the largest batch the launch grid takes; every batch is
    checked for finiteness, a spread of whole batches against the oracle."""
    w = Prefill("b65535_n20_d64", B=65535, Hq=1, Hkv=1, Nq=20, Nk=20, d=64, causal=True, seed=82)
    q, k, v = prefill_inputs(w)
    o, lse = binding.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert binding.device_status()[0] == binding.OK
    assert torch.isfinite(o.float()).all()
    o, lse = o.cpu(), lse.cpu()
    sel = np.array([0, 1, 2, 1000, 32767, 65533, 65534])
    o_ref, lse_ref = oracle.attention_forward(f64(q[sel]), f64(k[sel]), f64(v[sel]), w.scale, True)
    compare(o[sel], lse[sel], o_ref, lse_ref, w.name)
    with pytest.raises(binding.AttnError) as e:  # one more does not fit the grid
        binding.fwd(torch.empty(65536, 1, 1, 64, dtype=torch.bfloat16, device=DEV),
                    torch.empty(65536, 1, 1, 64, dtype=torch.bfloat16, device=DEV),
                    torch.empty(65536, 1, 1, 64, dtype=torch.bfloat16, device=DEV), causal=True)
    assert e.value.code == binding.ERR_UNSUPPORTED


def test_prefill_4096_heads():
    """4096 query heads sharing 64 KV heads (groups of 64), full output."""
    w = Prefill("hq4096_hkv64_n130_d64", B=1, Hq=4096, Hkv=64, Nq=130, Nk=130, d=64, causal=False, seed=83)
    q, k, v = prefill_inputs(w)
    o, lse = binding.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=False, scale=w.scale)
    torch.cuda.synchronize()
    assert binding.device_status()[0] == binding.OK
    o_ref, lse_ref = oracle.attention_forward(f64(q), f64(k), f64(v), w.scale, False)
    compare(o, lse, o_ref, lse_ref, w.name)


@pytest.mark.parametrize("Hq,Hkv,L,d", [(8, 1, 262144, 128), (16, 2, 199999, 64)], ids=["256k_mqa", "200k_d64"])
def test_decode_one_very_long_sequence(Hq, Hkv, L, d):
    """One sequence of up to 262 144 cached tokens: each unit is cut into
    pieces on every CTA and merged by the last piece to finish."""
    w = Decode(f"long{L}", B=1, Hq=Hq, Hkv=Hkv, Lmax=L, Lmin=L, d=d, seed=84)
    q, kc, vc, sl = decode_inputs(w)
    o, lse = binding.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), scale=w.scale)
    torch.cuda.synchronize()
    assert binding.device_status()[0] == binding.OK
    o_ref, lse_ref = oracle.attention_decode(f64(q), f64(kc), f64(vc), sl.numpy(), w.scale)
    compare(o, lse, o_ref, lse_ref, w.name)


def test_decode_4096_short_sequences():
    """4096 sequences of 0 to 128 cached tokens: each CTA's chunk spans dozens
    of whole units, and empty sequences are interleaved with the rest."""
    w = Decode("b4096_short", B=4096, Hq=4, Hkv=1, Lmax=128, Lmin=0, d=64, seed=85)
    q, kc, vc, sl = decode_inputs(w)
    assert (sl == 0).any()
    o, lse = binding.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), scale=w.scale)
    torch.cuda.synchronize()
    assert binding.device_status()[0] == binding.OK
    o_ref, lse_ref = oracle.attention_decode(f64(q), f64(kc), f64(vc), sl.numpy(), w.scale)
    compare(o, lse, o_ref, lse_ref, w.name)


def test_backward_32k_tokens():
    """The backward over 32 768 tokens: dQ on sampled rows, dK and dV on the
    last key tile (seen only by the last 128 query rows) and the sums over all
    key rows (the invariants of the full-size backward tests)."""
    w = Prefill("bwd_causal_n32768_d128", B=1, Hq=2, Hkv=1, Nq=32768, Nk=32768, d=128, causal=True, seed=86)
    q, k, v, do = (t.to(DEV) for t in backward_inputs(w))
    o, lse = binding.fwd(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert binding.device_status()[0] == binding.OK
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    rows = np.array([0, 1, 127, 128, 16383, 16384, 32766, 32767])
    for h in range(w.Hq):
        ref, _, _, m = oracle.attention_backward(f64(q[:, h:h + 1]), f64(k), f64(v), f64(do[:, h:h + 1]), w.scale,
                                                 True, q_rows=rows, k_rows=np.array([], dtype=np.int64),
                                                 magnitudes=True)
        compare_grad(dq[:, h:h + 1, rows], ref, m["tq"], m["sq"], f"{w.name} dq head {h}")
    t0 = w.Nk - 128
    _, rk, rv, m = oracle.attention_backward(f64(q[:, :, t0:]), f64(k), f64(v), f64(do[:, :, t0:]), w.scale, True,
                                             q_rows=np.array([], dtype=np.int64), k_rows=np.arange(t0, w.Nk),
                                             magnitudes=True)
    compare_grad(dk[:, :, t0:], rk, m["tk"], m["sk"], f"{w.name} dk last tile")
    compare_grad(dv[:, :, t0:], rv, m["tv"], None, f"{w.name} dv last tile")
    want_dv = do.double().reshape(w.B, w.Hkv, 2 * w.Nq, w.d).sum(dim=2)
    for name, g, want in (("dk", dk, torch.zeros_like(want_dv)), ("dv", dv, want_dv)):
        rss = g.double().pow(2).sum(dim=2).sqrt()
        assert ((g.double().sum(dim=2) - want).abs() <= 8 * BF16_U * rss).all(), name
