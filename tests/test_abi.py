"""The C-ABI library loads, exports every symbol include/attn.h declares, and
rejects bad arguments on the host before anything is launched. No GPU needed:
only host-side entry points and argument checks run here."""
import ctypes
import os
import re

import pytest

from exact_scaled_dot_03_b300 import binding
from exact_scaled_dot_03_b300 import build as buildmod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    buildmod.build()
    return binding.lib()


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            with open(os.path.join(ROOT, "include", h)) as f:
                text = f.read()
            names += re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert len(declared) >= 8
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(binding.SIGNATURES), "binding and header disagree"


def test_host_helpers(lib):
    assert lib.attn_version().startswith(b"exact-attn-sm103")
    for code in range(6):
        assert len(binding.status_string(code)) > 0
    # score bytes ([AUT] §6) and KV cache bytes ([PW] §3.2) through the C ABI
    assert [lib.attn_score_bytes(n, 1, 4) for n in (512, 1024, 2048, 4096)] == [m * 2**20 for m in (1, 4, 16, 64)]
    assert lib.attn_score_bytes(4096, 32, 4) == 2 * 2**30
    assert lib.attn_kv_cache_bytes(1, 2048, 32, 128, 2) == 32 * 2**20
    assert lib.attn_kv_cache_bytes(32, 8192, 32, 128, 2) == 4 * 2**30
    assert lib.attn_kv_cache_bytes(-1, 1, 1, 1, 1) == 0


def test_decode_workspace_size(lib):
    ws = binding.decode_workspace_size(16, 32, 8, 8192, 128)
    # 128 units x 16 splits x 4 heads x (128 values + 1 lse) fp32 + tickets
    assert ws >= 128 * 16 * 4 * 129 * 4
    assert binding.decode_workspace_size(16, 32, 8, 8192, 96) == 0     # unsupported d
    assert binding.decode_workspace_size(16, 30, 8, 8192, 128) == 0    # Hq % Hkv != 0
    assert binding.decode_workspace_size(0, 32, 8, 8192, 128) == 0


FAKE = 0x10000  # a 16-byte-aligned non-null address: never dereferenced on these paths


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=2, Hkv=1, Nq=16, Nk=16, d=64, scale=0.125,
         causal=0):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.ERR_INVALID_ARG),
    (dict(o=None), binding.ERR_INVALID_ARG),
    (dict(k=None), binding.ERR_INVALID_ARG),
    (dict(v=None, Nq=0), binding.ERR_INVALID_ARG),
    (dict(B=0), binding.ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), binding.ERR_INVALID_ARG),
    (dict(Nq=-1), binding.ERR_INVALID_ARG),
    (dict(causal=2), binding.ERR_INVALID_ARG),
    (dict(scale=0.0), binding.ERR_INVALID_ARG),
    (dict(scale=-1.0), binding.ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.ERR_INVALID_ARG),
    (dict(q=FAKE + 8), binding.ERR_INVALID_ARG),
    (dict(lse=FAKE + 2), binding.ERR_INVALID_ARG),
    (dict(d=96), binding.ERR_UNSUPPORTED),
    (dict(d=256), binding.ERR_UNSUPPORTED),
    (dict(B=70000), binding.ERR_UNSUPPORTED),
    (dict(Nq=0), binding.OK),   # empty: nothing to do, nothing launched
])
def test_fwd_argument_checks(lib, kw, code):
    assert _fwd(lib, **kw) == code


def test_fwd_window_argument_checks(lib):
    assert lib.attn_fwd_window(FAKE, FAKE, FAKE, FAKE, None, 1, 2, 1, 16, 16, 64, 0.125, 1, -1, None) == \
        binding.ERR_INVALID_ARG
    assert lib.attn_fwd_window(FAKE, FAKE, FAKE, FAKE, None, 1, 2, 1, 0, 16, 64, 0.125, 1, 8, None) == binding.OK


def _dec(lib, q=FAKE, kc=FAKE, vc=FAKE, sl=FAKE, o=FAKE, lse=None, B=2, Hq=8, Hkv=2, Lmax=100, d=128,
         scale=0.1, ws=FAKE, wsb=1 << 30):
    return lib.attn_decode(q, kc, vc, sl, o, lse, B, Hq, Hkv, Lmax, d, scale, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(sl=None), binding.ERR_INVALID_ARG),
    (dict(ws=None), binding.ERR_INVALID_ARG),
    (dict(wsb=16), binding.ERR_INVALID_ARG),
    (dict(Lmax=0), binding.ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), binding.ERR_INVALID_ARG),
    (dict(sl=FAKE + 2), binding.ERR_INVALID_ARG),
    (dict(kc=FAKE + 4), binding.ERR_INVALID_ARG),
    (dict(scale=0.0), binding.ERR_INVALID_ARG),
    (dict(d=80), binding.ERR_UNSUPPORTED),
    (dict(B=1 << 20, Hq=32, Hkv=32), binding.ERR_UNSUPPORTED),  # more (sequence, head) units than 2^24
])
def test_decode_argument_checks(lib, kw, code):
    assert _dec(lib, **kw) == code


def _paged(lib, q=FAKE, kn=FAKE, vn=FAKE, kp=FAKE, vp=FAKE, bt=FAKE, sl=FAKE, o=FAKE, lse=None, B=2, Hq=8, Hkv=2,
           num_pages=10, page_size=64, max_pages=4, d=128, scale=0.1, ws=FAKE, wsb=1 << 30):
    return lib.attn_decode_paged(q, kn, vn, kp, vp, bt, sl, o, lse, B, Hq, Hkv, num_pages, page_size, max_pages, d,
                                 scale, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bt=None), binding.ERR_INVALID_ARG),
    (dict(kn=None), binding.ERR_INVALID_ARG),          # k_new without v_new
    (dict(vn=None), binding.ERR_INVALID_ARG),
    (dict(ws=None), binding.ERR_INVALID_ARG),
    (dict(wsb=16), binding.ERR_INVALID_ARG),
    (dict(num_pages=0), binding.ERR_INVALID_ARG),
    (dict(max_pages=0), binding.ERR_INVALID_ARG),
    (dict(bt=FAKE + 2), binding.ERR_INVALID_ARG),
    (dict(kn=FAKE + 8), binding.ERR_INVALID_ARG),
    (dict(page_size=48), binding.ERR_UNSUPPORTED),
    (dict(page_size=4), binding.ERR_UNSUPPORTED),
    (dict(page_size=192), binding.ERR_UNSUPPORTED),
    (dict(d=96), binding.ERR_UNSUPPORTED),
])
def test_paged_decode_argument_checks(lib, kw, code):
    assert _paged(lib, **kw) == code


def test_fwd_rope_argument_checks(lib):
    f = lambda **kw: lib.attn_fwd_rope(*[kw.get(n, dflt) for n, dflt in [
        ("q", FAKE), ("k", FAKE), ("v", FAKE), ("o", FAKE), ("lse", None), ("B", 1), ("Hq", 2), ("Hkv", 1),
        ("Nq", 16), ("Nk", 16), ("d", 64), ("scale", 0.125), ("causal", 1), ("window", 0), ("base", 10000.0),
        ("ws", 0x100000), ("wsb", 1 << 30), ("stream", None)]])
    assert f(base=1.0) == binding.ERR_INVALID_ARG
    assert f(base=float("nan")) == binding.ERR_INVALID_ARG
    assert f(ws=None) == binding.ERR_INVALID_ARG
    assert f(ws=0x100010) == binding.ERR_INVALID_ARG          # not 256-byte aligned
    assert f(wsb=64) == binding.ERR_INVALID_ARG
    assert f(Nk=0) == binding.ERR_INVALID_ARG
    assert f(window=-2) == binding.ERR_INVALID_ARG
    assert f(d=96) == binding.ERR_UNSUPPORTED
    assert f(Nq=0) == binding.OK
    # rotated K (1 x 1 x 16 x 64 bf16 = 2 KiB), then the 16 positions x 32 pairs
    # x 8-byte (cos, sin) table twice: position-major and pair-major
    assert lib.attn_fwd_rope_workspace_size(1, 1, 16, 16, 64) == 2048 + 2 * 16 * 32 * 8
    assert lib.attn_fwd_rope_workspace_size(1, 1, 20, 16, 64) == 2048 + 2 * 20 * 32 * 8  # queries before key 0


def test_bwd_argument_checks(lib):
    f = lambda **kw: lib.attn_bwd(*[kw.get(n, dflt) for n, dflt in [
        ("q", FAKE), ("k", FAKE), ("v", FAKE), ("o", FAKE), ("lse", FAKE), ("do", FAKE), ("dq", FAKE),
        ("dk", FAKE), ("dv", FAKE), ("B", 1), ("Hq", 4), ("Hkv", 2), ("Nq", 200), ("Nk", 300), ("d", 128),
        ("scale", 0.088), ("causal", 1), ("ws", 0x100000), ("wsb", 1 << 30), ("stream", None)]])
    assert f(lse=None) == binding.ERR_INVALID_ARG         # the forward's LSE is required
    assert f(do=None) == binding.ERR_INVALID_ARG
    assert f(dk=None) == binding.ERR_INVALID_ARG
    assert f(Hq=3) == binding.ERR_INVALID_ARG             # Hq % Hkv != 0
    assert f(causal=2) == binding.ERR_INVALID_ARG
    assert f(scale=0.0) == binding.ERR_INVALID_ARG
    assert f(dq=FAKE + 8) == binding.ERR_INVALID_ARG      # not 16-byte aligned
    assert f(ws=0x100010) == binding.ERR_INVALID_ARG      # not 256-byte aligned
    assert f(ws=None) == binding.ERR_INVALID_ARG
    assert f(wsb=4 * 256 * 72 - 1) == binding.ERR_INVALID_ARG
    assert f(d=96) == binding.ERR_UNSUPPORTED
    # per query row: lse2 and Dl (fp32) and two 32-byte seed rows; heads padded to 128 rows
    assert lib.attn_bwd_workspace_size(1, 4, 200) == 4 * 256 * 72
    assert lib.attn_bwd_workspace_size(2, 3, 128) == 6 * 128 * 72
    assert lib.attn_bwd_workspace_size(0, 4, 200) == 0


def test_paged_workspace_size(lib):
    # same plan as the contiguous decode with Lmax = pages * page_size
    assert binding.lib().attn_decode_paged_workspace_size(16, 32, 8, 128, 64, 128) == \
        binding.decode_workspace_size(16, 32, 8, 8192, 128)
    assert binding.lib().attn_decode_paged_workspace_size(16, 32, 8, 128, 48, 128) == 0


def test_product_path_has_no_fallback(monkeypatch, tmp_path):
    """Without the built library the binding raises; it never computes another way."""
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()


def test_stall_hook_host_side(lib):
    """The failure-detection test hook accepts only its kinds (and 0, which
    disarms it); nothing is launched here."""
    assert lib.attn_test_arm_stall(7) == binding.ERR_INVALID_ARG
    assert lib.attn_test_arm_stall(-1) == binding.ERR_INVALID_ARG
    assert lib.attn_test_arm_stall(4) == binding.ERR_INVALID_ARG
    assert lib.attn_test_arm_stall(3) == binding.OK   # the backward's kind
    assert lib.attn_test_arm_stall(1) == binding.OK
    assert lib.attn_test_arm_stall(0) == binding.OK   # disarmed again


def test_fwd_host_workspace_size_and_argument_checks(lib):
    # per (batch, KV head) group: K and V, twice (two K/V slots); per chunk slot (three):
    # Q and O of a whole group's query heads and their LSE, each rounded up to 256 bytes
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    B, Hq, Hkv, Nq, Nk, d = 1, 8, 2, 100, 300, 64
    G = Hq // Hkv
    want = 2 * 2 * a256(Nk * d * 2) + 3 * (2 * a256(G * Nq * d * 2) + a256(G * Nq * 4))
    assert lib.attn_fwd_host_workspace_size(B, Hq, Hkv, Nq, Nk, d) == want
    assert lib.attn_fwd_host_workspace_size(B, 6, 4, Nq, Nk, d) == 0      # Hq % Hkv != 0
    assert lib.attn_fwd_host_workspace_size(B, Hq, Hkv, Nq, Nk, 96) == 0  # unsupported d
    ws = 0x100000
    f = lambda **kw: lib.attn_fwd_host(*[kw.get(n, dflt) for n, dflt in [  # noqa: E731
        ("q", FAKE), ("k", FAKE), ("v", FAKE), ("o", FAKE), ("lse", None), ("B", B), ("Hq", Hq), ("Hkv", Hkv),
        ("Nq", Nq), ("Nk", Nk), ("d", d), ("scale", 0.125), ("causal", 1), ("ws", ws), ("wsb", want),
        ("stream", None)]])
    assert f(q=None) == binding.ERR_INVALID_ARG
    assert f(o=None) == binding.ERR_INVALID_ARG
    assert f(k=None) == binding.ERR_INVALID_ARG
    assert f(Hq=3) == binding.ERR_INVALID_ARG
    assert f(causal=2) == binding.ERR_INVALID_ARG
    assert f(scale=0.0) == binding.ERR_INVALID_ARG
    assert f(ws=None) == binding.ERR_INVALID_ARG
    assert f(ws=ws + 16) == binding.ERR_INVALID_ARG      # not 256-byte aligned
    assert f(wsb=want - 1) == binding.ERR_INVALID_ARG
    assert f(d=96) == binding.ERR_UNSUPPORTED
    # no queries: nothing to do (q and o may then be NULL), nothing queued
    assert f(Nq=0, q=None, o=None, wsb=lib.attn_fwd_host_workspace_size(B, Hq, Hkv, 0, Nk, d)) == binding.OK
