"""KV-cache decode: CUDA path vs the fp64 oracle, element by element."""
import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_03_b300 import binding
from exact_scaled_dot_03_b300.workloads import DECODE_GQA, Decode, decode_inputs
from tests.parity import compare, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(q, kc, vc, sl, scale, ws=None):
    o, lse = binding.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV), scale=scale, workspace=ws)
    torch.cuda.synchronize()
    return o, lse


def test_decode_full_workload():
    w = DECODE_GQA
    q, kc, vc, sl = decode_inputs(w)
    o, lse = _run(q, kc, vc, sl, w.scale)
    o_ref, lse_ref = oracle.attention_decode(f64(q), f64(kc), f64(vc), sl.numpy(), w.scale)
    compare(o, lse, o_ref, lse_ref, w.name)
    assert binding.device_status()[0] == binding.OK


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 8, 128), (32, 1, 128), (16, 8, 64), (16, 2, 128), (12, 4, 64)],
                         ids=["mha", "mqa_g32", "g2_d64", "g8", "g3_d64"])
def test_decode_edge_lengths(Hq, Hkv, d):
    """Lengths on and around the tile (64) and split (512) edges, 0, 1 and Lmax."""
    lens = [0, 1, 63, 64, 65, 511, 512, 513, 1000, 1100]
    w = Decode("edges", B=len(lens), Hq=Hq, Hkv=Hkv, Lmax=1100, Lmin=1, d=d, seed=31)
    q, kc, vc, _ = decode_inputs(w)
    sl = torch.tensor(lens, dtype=torch.int32)
    o, lse = _run(q, kc, vc, sl, w.scale)
    o_ref, lse_ref = oracle.attention_decode(f64(q), f64(kc), f64(vc), sl.numpy(), w.scale)
    compare(o, lse, o_ref, lse_ref, f"edges Hq={Hq} Hkv={Hkv} d={d}")


def test_decode_never_reads_past_length():
    """NaN in every cache row at or past seqlens must not reach the output."""
    w = Decode("poison", B=4, Hq=8, Hkv=2, Lmax=1500, Lmin=1, d=128, seed=32)
    q, kc, vc, _ = decode_inputs(w)
    sl = torch.tensor([1, 700, 1024, 1499], dtype=torch.int32)
    for b, L in enumerate(sl.tolist()):
        kc[b, :, L:] = float("nan")
        vc[b, :, L:] = float("nan")
    o, lse = _run(q, kc, vc, sl, w.scale)
    o_ref, lse_ref = oracle.attention_decode(f64(q), f64(kc), f64(vc), sl.numpy(), w.scale)
    compare(o, lse, o_ref, lse_ref, "poison")


def test_decode_workspace_reuse_and_status():
    w = Decode("reuse", B=3, Hq=8, Hkv=2, Lmax=3000, Lmin=600, d=128, seed=33)
    q, kc, vc, sl = decode_inputs(w)
    ws = binding.decode_workspace(w.B, w.Hq, w.Hkv, w.Lmax, w.d)
    o1, l1 = _run(q, kc, vc, sl, w.scale, ws)
    o2, l2 = _run(q, kc, vc, sl, w.scale, ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # the per-unit tickets (last 32 bytes here: 6 units x 4 bytes, rounded to 16) are back at zero
    assert int(ws[-32:].count_nonzero()) == 0
    o_ref, lse_ref = oracle.attention_decode(f64(q), f64(kc), f64(vc), sl.numpy(), w.scale)
    compare(o2, l2, o_ref, lse_ref, "reuse")
    # a length past Lmax is clamped and reported
    bad = sl.clone()
    bad[1] = w.Lmax + 5
    o3, l3 = _run(q, kc, vc, bad, w.scale, ws)
    code, detail = binding.device_status()
    assert code == binding.ERR_DEVICE_ARG, (code, detail)
    clamped = bad.clone()
    clamped[1] = w.Lmax
    o_ref3, lse_ref3 = oracle.attention_decode(f64(q), f64(kc), f64(vc), clamped.numpy(), w.scale)
    compare(o3, l3, o_ref3, lse_ref3, "clamped")
    assert binding.device_status()[0] == binding.OK   # cleared by the read


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,d,lens", [
    # one long sequence: its tiles are spread over many CTAs and merged by the last one
    (1, 8, 1, 20000, 128, [20000]),
    (2, 4, 2, 9000, 64, [9000, 8999]),
    # many short sequences: each CTA's chunk spans many whole units
    (300, 16, 4, 260, 128, None),
    (64, 32, 8, 1500, 128, None),
], ids=["long_mqa", "long_d64", "many_short", "gqa_b64"])
def test_decode_balanced_partition(B, Hq, Hkv, Lmax, d, lens):
    w = Decode("partition", B=B, Hq=Hq, Hkv=Hkv, Lmax=Lmax, Lmin=0, d=d, seed=34)
    q, kc, vc, sl = decode_inputs(w)
    if lens is not None:
        sl = torch.tensor(lens, dtype=torch.int32)
    o, lse = _run(q, kc, vc, sl, w.scale)
    o_ref, lse_ref = oracle.attention_decode(f64(q), f64(kc), f64(vc), sl.numpy(), w.scale)
    compare(o, lse, o_ref, lse_ref, f"partition B={B} Lmax={Lmax}")
    assert binding.device_status()[0] == binding.OK
