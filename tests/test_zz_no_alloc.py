"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc or hand over a workspace (code running
inside an allocator or memory-pool callback, under a framework that owns all
device memory, or where an allocation could synchronise or fail). This entry
point keeps its split-KV scratch in a static device array inside the library
instead. Here it is called through the C ABI twice in a row, on different
problems so the second call starts from the first call's leftover scratch,
and each result is checked against the fp64 oracle (the parity bar every
other test uses) and against the workspace-taking attn_decode within the
same tolerance.

Kept in a file that pytest collects last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
from exact_scaled_dot_03_b300 import binding
from exact_scaled_dot_03_b300.workloads import DECODE_GQA, Decode, decode_inputs
from tests.parity import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, compare, f64

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 8 << 20  # ATTN_NOALLOC_SCRATCH_BYTES in include/attn.h


def _noalloc(q, kc, vc, sl, o, lse, scale):
    B, Hq, d = q.shape
    _, Hkv, Lmax, _ = kc.shape
    return binding.lib().attn_decode_noalloc(
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(), o.data_ptr(), lse.data_ptr(),
        B, Hq, Hkv, Lmax, d, ctypes.c_float(scale), torch.cuda.current_stream().cuda_stream)


def _case(w, lens=None):
    q, kc, vc, sl = decode_inputs(w)
    if lens is not None:
        sl = torch.tensor(lens, dtype=torch.int32)
    q, kc, vc, sl = (t.cuda() for t in (q, kc, vc, sl))
    return q, kc, vc, sl


def _check_against_workspace_path(w, lens=None):
    q, kc, vc, sl = _case(w, lens)
    assert binding.decode_workspace_size(w.B, w.Hq, w.Hkv, w.Lmax, w.d) <= SCRATCH_LIMIT
    o_ref, lse_ref = binding.decode(q, kc, vc, sl, scale=w.scale)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device="cuda")
    assert _noalloc(q, kc, vc, sl, o, lse, w.scale) == binding.OK
    torch.cuda.synchronize()
    # against the oracle: the plain decode definition in fp64 on the same bf16 inputs
    o64, lse64 = oracle.attention_decode(f64(q), f64(kc), f64(vc), sl.cpu().numpy(), w.scale)
    print(w.name, compare(o, lse, o64, lse64, f"noalloc {w.name}"))
    # and against the workspace-taking entry point
    err = (o.float() - o_ref.float()).abs()
    assert err.max().item() <= O_MAX_ABS and err.mean().item() <= O_MEAN_ABS
    finite = torch.isfinite(lse_ref)
    assert torch.equal(finite, torch.isfinite(lse))
    assert (lse[finite] - lse_ref[finite]).abs().max().item() <= LSE_MAX_ABS


def test_noalloc_matches_workspace_decode_twice_in_a_row():
    # first call: the bench decode shape (GQA, lengths in [1024, 8192])
    _check_against_workspace_path(DECODE_GQA)
    # second call, right after, on another shape (MQA, d = 64, empty and
    # tile-edge lengths): reuses the scratch the first call left behind
    w2 = Decode("noalloc_second", B=6, Hq=8, Hkv=1, Lmax=2100, Lmin=1, d=64, seed=41)
    _check_against_workspace_path(w2, lens=[0, 1, 64, 513, 2048, 2100])
    assert binding.device_status()[0] == binding.OK


def test_noalloc_rejects_problems_larger_than_its_scratch():
    w = Decode("too_big", B=64, Hq=32, Hkv=8, Lmax=32768, Lmin=1, d=128, seed=42)
    assert binding.decode_workspace_size(w.B, w.Hq, w.Hkv, w.Lmax, w.d) > SCRATCH_LIMIT
    q = torch.zeros(w.B, w.Hq, w.d, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, dtype=torch.bfloat16, device="cuda")   # never touched: rejected on the host
    sl = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device="cuda")
    code = binding.lib().attn_decode_noalloc(
        q.data_ptr(), kc.data_ptr(), kc.data_ptr(), sl.data_ptr(), o.data_ptr(), lse.data_ptr(),
        w.B, w.Hq, w.Hkv, w.Lmax, w.d, ctypes.c_float(w.scale), torch.cuda.current_stream().cuda_stream)
    assert code == binding.ERR_UNSUPPORTED
