"""Paged KV-cache decode with the new token appended: CUDA path vs the fp64 oracle.

The output and LSE are compared element by element within the parity bar; the
pages after the call must hold the appended K/V rows exactly and be unchanged
everywhere else (byte work: bit-exact).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_scaled_dot_03_b300 import binding
from exact_scaled_dot_03_b300.workloads import DECODE_GQA_PAGED, PagedDecode, bf16_bits, paged_decode_inputs
from tests.parity import compare, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _check(w, lens=None, poison=False):
    q, kn, vn, kp, vp, bt, sl = paged_decode_inputs(w, lens)
    if poison:  # rows no sequence may read: past each length, in unused pages
        used = set()
        P = w.page_size
        for b, L in enumerate(sl.tolist()):
            n = L + (1 if w.append else 0)
            for p in range((n + P - 1) // P):
                used.add(int(bt[b, p]))
            last = int(bt[b, (n - 1) // P]) if n else None
            if last is not None:
                kp[last, :, (n - 1) % P + 1:] = float("nan")
                vp[last, :, (n - 1) % P + 1:] = float("nan")
        for pg in range(kp.shape[0]):
            if pg not in used:
                kp[pg] = float("nan")
                vp[pg] = float("nan")
        if w.append:  # the append slot itself: stale data the kernel must not use
            for b, L in enumerate(sl.tolist()):
                kp[int(bt[b, L // P]), :, L % P] = float("nan")
                vp[int(bt[b, L // P]), :, L % P] = float("nan")
    kp_d, vp_d = kp.to(DEV), vp.to(DEV)
    o, lse = binding.decode_paged(q.to(DEV), kp_d, vp_d, bt.to(DEV), sl.to(DEV),
                                  kn.to(DEV) if kn is not None else None, vn.to(DEV) if vn is not None else None,
                                  scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref, kp_ref, vp_ref = oracle.attention_decode_paged(
        f64(q), f64(kp), f64(vp), bt.numpy(), sl.numpy(), w.scale,
        f64(kn) if kn is not None else None, f64(vn) if vn is not None else None)
    compare(o, lse, o_ref, lse_ref, w.name)
    # the appended rows land exactly; nothing else in the pages changes
    kp_after, vp_after = f64(kp_d), f64(vp_d)
    np.testing.assert_array_equal(np.isnan(kp_after), np.isnan(kp_ref))
    np.testing.assert_array_equal(np.nan_to_num(kp_after), np.nan_to_num(kp_ref))
    np.testing.assert_array_equal(np.nan_to_num(vp_after), np.nan_to_num(vp_ref))
    assert binding.device_status()[0] == binding.OK


def test_paged_decode_full_workload():
    _check(DECODE_GQA_PAGED)


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("append", [True, False])
def test_paged_decode_page_sizes_and_edges(page_size, append):
    lens = [0 if append else 1, 1, 7, 63, 64, 127, 128, 129, 255, 256, 300]
    w = PagedDecode(f"edges_p{page_size}", B=len(lens), Hq=8, Hkv=2, Lmin=1, Lmax=300, d=128,
                    page_size=page_size, append=append, seed=51)
    _check(w, lens=lens, poison=True)


@pytest.mark.parametrize("Hq,Hkv,d", [(16, 16, 64), (32, 1, 128), (12, 4, 64)], ids=["mha_d64", "mqa", "g3_d64"])
def test_paged_decode_head_layouts(Hq, Hkv, d):
    w = PagedDecode("heads", B=5, Hq=Hq, Hkv=Hkv, Lmin=0, Lmax=2000, d=d, page_size=32, append=True, seed=52)
    _check(w, poison=True)


def test_paged_decode_bad_page_id_is_flagged():
    w = PagedDecode("bad_page", B=2, Hq=8, Hkv=2, Lmin=200, Lmax=300, d=128, page_size=64, append=False, seed=53)
    q, _, _, kp, vp, bt, sl = paged_decode_inputs(w)
    bt[1, 1] = kp.shape[0] + 5
    binding.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), bt.to(DEV), sl.to(DEV), scale=w.scale)
    code, detail = binding.device_status()
    assert code == binding.ERR_DEVICE_ARG, (code, detail)
    assert binding.device_status()[0] == binding.OK
