"""The give-up path of the kernels' bounded waits, exercised on the GPU
without a fault or a hang.

Every internal wait of the prefill, decode and backward kernels is bounded. The library's
test hook (attn_test_arm_stall) makes one role of the first CTA of the next
launch wait on a barrier that nothing arrives on, with a 1 ms limit. That wait
gives up, the kernel takes its normal abort path: the other roles of the CTA
stop waiting, copies and MMAs still in flight land, tensor memory is freed,
the kernel returns. The checks: the status word reports a timeout at the
stalled wait's site (and no other wait ran to its own 1 s limit, which would
overwrite the site and take a second), and the next normal call, on a fresh
workspace, matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_03_b300 import binding
from exact_scaled_dot_03_b300.workloads import Decode, Prefill, backward_inputs, decode_inputs, prefill_inputs
from tests.parity import compare, compare_grad, f64

pytestmark = pytest.mark.gpu

STALL_PREFILL, STALL_DECODE, STALL_BACKWARD = 1, 2, 3   # ATTN_TEST_STALL_* in include/attn.h
SITE_PREFILL_S_FULL = 8              # the prefill softmax warps' score wait
SITE_DECODE_FULL = 20                # the decode warps' K/V tile wait
SITE_BACKWARD_S_FULL = 38            # the dK/dV kernel's elementwise score wait


def _stalled(call, kind):
    """Run `call` with the hook armed; return (status, detail, seconds)."""
    assert binding.device_status()[0] == binding.OK
    torch.cuda.synchronize()
    assert binding.lib().attn_test_arm_stall(kind) == binding.OK
    t0 = time.perf_counter()
    call()
    code, detail = binding.device_status()
    return code, detail, time.perf_counter() - t0


@pytest.mark.parametrize("d", [128, 64])
def test_prefill_wait_gives_up_and_the_next_call_is_exact(d):
    w = Prefill("timeout_prefill", B=1, Hq=4, Hkv=2, Nq=1000, Nk=1000, d=d, causal=True, seed=90 + d)
    q, k, v = (t.cuda() for t in prefill_inputs(w))
    code, detail, secs = _stalled(lambda: binding.fwd(q, k, v, causal=True, scale=w.scale), STALL_PREFILL)
    assert code == binding.ERR_TIMEOUT, (code, detail)
    assert detail[1] == SITE_PREFILL_S_FULL and detail[2] == 0, detail
    assert secs < 0.5, f"abort took {secs:.3f} s: some wait ran to its full limit"
    # the hook disarmed itself: the next call runs normally and is exact
    o, lse = binding.fwd(q, k, v, causal=True, scale=w.scale)
    assert binding.device_status()[0] == binding.OK
    o_ref, lse_ref = oracle.attention_forward(f64(q), f64(k), f64(v), w.scale, True)
    print(compare(o, lse, o_ref, lse_ref, "after the stalled prefill"))


def test_decode_wait_gives_up_and_the_next_call_is_exact():
    w = Decode("timeout_decode", B=8, Hq=16, Hkv=4, Lmax=3000, Lmin=600, d=128, seed=97)
    q, kc, vc, sl = (t.cuda() for t in decode_inputs(w))
    ws = binding.decode_workspace(w.B, w.Hq, w.Hkv, w.Lmax, w.d)
    code, detail, secs = _stalled(lambda: binding.decode(q, kc, vc, sl, scale=w.scale, workspace=ws),
                                  STALL_DECODE)
    assert code == binding.ERR_TIMEOUT, (code, detail)
    assert detail[1] == SITE_DECODE_FULL and detail[2] == 0, detail
    assert secs < 0.5, f"abort took {secs:.3f} s: some wait ran to its full limit"
    # a fresh (zeroed) workspace: the stalled call may have left tickets behind
    o, lse = binding.decode(q, kc, vc, sl, scale=w.scale, workspace=binding.decode_workspace(w.B, w.Hq, w.Hkv,
                                                                                             w.Lmax, w.d))
    assert binding.device_status()[0] == binding.OK
    o_ref, lse_ref = oracle.attention_decode(f64(q), f64(kc), f64(vc), sl.cpu().numpy(), w.scale)
    print(compare(o, lse, o_ref, lse_ref, "after the stalled decode"))


@pytest.mark.parametrize("d", [128, 64])
def test_backward_wait_gives_up_and_the_next_call_is_exact(d):
    w = Prefill("timeout_backward", B=1, Hq=4, Hkv=2, Nq=700, Nk=700, d=d, causal=True, seed=80 + d)
    q, k, v, do = (t.cuda() for t in backward_inputs(w))
    o, lse = binding.fwd(q, k, v, causal=True, scale=w.scale)
    code, detail, secs = _stalled(lambda: binding.bwd(q, k, v, o, lse, do, causal=True, scale=w.scale),
                                  STALL_BACKWARD)
    assert code == binding.ERR_TIMEOUT, (code, detail)
    assert detail[1] == SITE_BACKWARD_S_FULL and detail[2] == 0, detail
    # the backward's elementwise and copy waits do not watch the abort flag: the
    # CTA's other roles give up at their own 1 s limit (all at about the same time)
    assert secs < 3.0, f"abort took {secs:.3f} s"
    # the hook disarmed itself: the next call runs normally and is exact
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert binding.device_status()[0] == binding.OK
    *ref, m = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), w.scale, True, magnitudes=True)
    for name, g, r, t, sd in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, (m["tq"], m["tk"], m["tv"]),
                                 (m["sq"], m["sk"], None)):
        compare_grad(g, r, t, sd, f"after the stalled backward: {name}")


def test_disarmed_hook_changes_nothing():
    w = Prefill("timeout_disarmed", B=1, Hq=2, Hkv=1, Nq=300, Nk=300, d=128, causal=True, seed=98)
    q, k, v = (t.cuda() for t in prefill_inputs(w))
    assert binding.lib().attn_test_arm_stall(STALL_PREFILL) == binding.OK
    assert binding.lib().attn_test_arm_stall(0) == binding.OK
    o, lse = binding.fwd(q, k, v, causal=True, scale=w.scale)
    assert binding.device_status()[0] == binding.OK
    o_ref, lse_ref = oracle.attention_forward(f64(q), f64(k), f64(v), w.scale, True)
    compare(o, lse, o_ref, lse_ref, "disarmed")
