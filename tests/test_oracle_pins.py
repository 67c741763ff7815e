"""Pins for the fp64 oracle: facts that do not come from the oracle itself.

Each test would fail under a plausible slip in the oracle (a dropped scale, a
flipped sign, a wrong GQA index, a transposed operand, a wrong causal offset,
a missing rescale in the recurrence). Sources are cited by page title and
section; the key [MG-A], [MG-B], [AUT], [IMR], [PW] is spelled out in
``oracle/__init__.py``.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import (
    attention_forward_rope,
    rope_rotate,
    round_to_bf16,
    attention_decode_paged,
    attention_decode,
    attention_backward,
    attention_forward,
    bf16_bits_to_f64,
    kv_cache_bytes,
    merge_two_blocks,
    online_attention_rows,
    score_bytes,
)

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# --- worked examples (golden fixtures) -------------------------------------------------

def test_two_key_worked_example(golden_dir):
    """[MG-A] §2.4: weights exp(S_ij)/sum exp(S_ik); hand-worked 3/4, 1/4 split."""
    g = _load(golden_dir, "two_key_softmax.json")
    q = np.array(g["q"])[None, None]
    k = np.array(g["k"])[None, None]
    v = np.array(g["v"])[None, None]
    o, lse = attention_forward(q, k, v, g["scale"], causal=False)
    np.testing.assert_allclose(o[0, 0], g["o"], atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], g["lse"], atol=1e-12)


def test_causal_three_token_worked_example(golden_dir):
    """[IMR] masking: token t sees positions <= t; hand-worked weights 1, 1:2, 1:2:3."""
    g = _load(golden_dir, "causal_three_tokens.json")
    q = np.array(g["q"])[None, None]
    k = np.array(g["k"])[None, None]
    v = np.array(g["v"])[None, None]
    o, lse = attention_forward(q, k, v, g["scale"], causal=True)
    np.testing.assert_allclose(o[0, 0], g["o"], atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], g["lse"], atol=1e-12)
    # the online recurrence must give the same numbers at every tiling
    for tile in (1, 2, 3):
        o2, l2 = online_attention_rows(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]),
                                       g["scale"], tile, causal_offset=0)
        np.testing.assert_allclose(o2, g["o"], atol=1e-12)
        np.testing.assert_allclose(l2, g["lse"], atol=1e-12)


def test_score_matrix_bytes_match_pages(golden_dir):
    """[AUT] §6: 1/4/16/64 MiB at N = 512..4096; [PW] §2.1: 32 heads at 4096 ~ 2 GB."""
    g = _load(golden_dir, "score_bytes.json")
    for n, mib in g["per_head_fp32_mib"].items():
        assert score_bytes(int(n)) == mib * 2**20
    assert score_bytes(4096, heads=32) == g["n4096_heads32_fp32_gib"] * 2**30
    # quadratic growth: doubling n quadruples the bytes ([AUT] §4)
    assert score_bytes(2048) == 4 * score_bytes(1024)


def test_kv_cache_bytes_match_pages(golden_dir):
    """[PW] §3.2 / §7.3 LLaMA-7B cache sizes from [AUT] §9 M_KV = 2 L n h_kv d_h b."""
    g = _load(golden_dir, "kv_cache_bytes.json")
    for c in g["cases"]:
        got = kv_cache_bytes(c["layers"], c["n"], c["h_kv"], c["d_h"], c["b"])
        want = c["mib"] * 2**20 if "mib" in c else c["gib"] * 2**30
        assert got == want
    assert 16 * kv_cache_bytes(32, 2048, 32, 128, 2) == g["batch16_n2048_layers32_gib"] * 2**30
    r = g["gqa_ratio"]
    assert kv_cache_bytes(1, 1, r["h_q"], 128, 2) == r["shrink"] * kv_cache_bytes(1, 1, r["h_kv"], 128, 2)


# --- closed forms and invariants ----------------------------------------------------------

def test_bf16_decoding_exact():
    """bf16 is the top half of binary32: check named patterns and all 65536 against torch."""
    named = {0x3F80: 1.0, 0xC000: -2.0, 0x3FC0: 1.5, 0x0000: 0.0, 0x7F80: np.inf,
             0xFF80: -np.inf, 0x0001: 2.0**-133, 0x4049: 3.140625}
    for bits, val in named.items():
        assert bf16_bits_to_f64(np.array([bits], np.uint16))[0] == val
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = bf16_bits_to_f64(allbits)
    ref = torch.from_numpy(allbits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_rows_are_probability_distributions():
    """[MG-A] §2.4: each row of weights sums to 1; with V = I the output IS the weight row,
    and weight ratios follow exp of score differences."""
    rng = np.random.default_rng(1)
    n, d = 9, 5
    q, k = _rand(rng, 1, 1, n, d), _rand(rng, 1, 1, n, d)
    scale = 0.37
    P, _ = attention_forward(q, k, np.eye(n)[None, None], scale, causal=False)
    P = P[0, 0]
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
    assert (P > 0).all()
    s = scale * q[0, 0] @ k[0, 0].T
    np.testing.assert_allclose(np.log(P[:, 1:] / P[:, :1]), s[:, 1:] - s[:, :1], atol=1e-10)
    # causal: weights above the diagonal are exactly 0, rows still sum to 1
    Pc, _ = attention_forward(q, k, np.eye(n)[None, None], scale, causal=True)
    assert (np.triu(Pc[0, 0], 1) == 0).all()
    np.testing.assert_allclose(Pc[0, 0].sum(axis=1), 1.0, atol=1e-12)


def test_identical_keys_give_mean_of_values():
    """All keys equal => uniform weights => O = mean(V), LSE = s + ln Nk ([MG-A] §2.4)."""
    rng = np.random.default_rng(2)
    Nk, d = 37, 8
    q = _rand(rng, 1, 1, 5, d)
    k = np.repeat(_rand(rng, 1, 1, 1, d), Nk, axis=2)
    v = _rand(rng, 1, 1, Nk, d)
    scale = 0.25
    o, lse = attention_forward(q, k, v, scale, causal=False)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (5, d)), atol=1e-12)
    s = scale * (q[0, 0] @ k[0, 0, 0])
    np.testing.assert_allclose(lse[0, 0], s + math.log(Nk), atol=1e-12)


def test_causal_row_zero_is_first_value():
    """[IMR] masking: row 0 sees only key 0 => O_0 = v_0 exactly, LSE_0 = scale q_0.k_0."""
    rng = np.random.default_rng(3)
    q, k, v = (_rand(rng, 2, 3, 16, 8) for _ in range(3))
    o, lse = attention_forward(q, k, v, 0.5, causal=True)
    assert np.array_equal(o[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], 0.5 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]),
                               atol=1e-12)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 1, 2, 6, 4), _rand(rng, 1, 2, 1, 4), _rand(rng, 1, 2, 1, 4)
    o, _ = attention_forward(q, k, v, 1.0, causal=False)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), atol=1e-15)


def test_affine_in_values():
    """O is a convex combination of value rows ([MG-A] §2.4), hence affine in V."""
    rng = np.random.default_rng(5)
    q, k, v = (_rand(rng, 1, 2, 11, 6) for _ in range(3))
    for causal in (False, True):
        o, _ = attention_forward(q, k, v, 0.4, causal)
        o2, _ = attention_forward(q, k, 3.0 * v - 2.0, 0.4, causal)
        np.testing.assert_allclose(o2, 3.0 * o - 2.0, atol=1e-12)


def test_permutation_invariance_non_causal():
    """Permuting (K, V) rows together changes nothing; permuting Q rows permutes O."""
    rng = np.random.default_rng(6)
    q, k, v = _rand(rng, 1, 1, 10, 5), _rand(rng, 1, 1, 13, 5), _rand(rng, 1, 1, 13, 3)
    o, lse = attention_forward(q, k, v, 0.7, causal=False)
    pk = rng.permutation(13)
    o2, lse2 = attention_forward(q, k[:, :, pk], v[:, :, pk], 0.7, causal=False)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)
    pq = rng.permutation(10)
    o3, _ = attention_forward(q[:, :, pq], k, v, 0.7, causal=False)
    np.testing.assert_allclose(o3, o[:, :, pq], atol=1e-12)


def test_large_scale_selects_best_matching_key():
    """As the scale grows, softmax concentrates on the largest score: O -> v_argmax.
    (A sign slip would select the smallest score instead.)"""
    rng = np.random.default_rng(7)
    q, k, v = _rand(rng, 1, 1, 6, 4), _rand(rng, 1, 1, 9, 4), _rand(rng, 1, 1, 9, 3)
    s = q[0, 0] @ k[0, 0].T
    o, _ = attention_forward(q, k, v, 1e4, causal=False)
    np.testing.assert_allclose(o[0, 0], v[0, 0][s.argmax(axis=1)], atol=1e-9)


def test_cross_attention_bottom_right_causal_alignment():
    """Nq != Nk causal: the last query sees every key, query i sees keys j <= i + Nk - Nq;
    the no-key rows (Nq > Nk) give O = 0, LSE = -inf."""
    rng = np.random.default_rng(8)
    q, k, v = _rand(rng, 1, 1, 4, 3), _rand(rng, 1, 1, 7, 3), _rand(rng, 1, 1, 7, 2)
    o, lse = attention_forward(q, k, v, 1.0, causal=True)
    full, fl = attention_forward(q[:, :, 3:], k, v, 1.0, causal=False)
    np.testing.assert_allclose(o[:, :, 3:], full, atol=1e-12)
    np.testing.assert_allclose(lse[:, :, 3:], fl, atol=1e-12)
    first, f0 = attention_forward(q[:, :, :1], k[:, :, :4], v[:, :, :4], 1.0, causal=False)
    np.testing.assert_allclose(o[:, :, :1], first, atol=1e-12)
    q2 = _rand(rng, 1, 1, 6, 3)
    o2, l2 = attention_forward(q2, k[:, :, :2], v[:, :, :2], 1.0, causal=True)
    assert (o2[0, 0, :4] == 0).all() and np.isneginf(l2[0, 0, :4]).all()
    np.testing.assert_allclose(o2[0, 0, 5], attention_forward(q2[:, :, 5:], k[:, :, :2], v[:, :, :2],
                                                              1.0, False)[0][0, 0, 0], atol=1e-12)


# --- independent library routine ----------------------------------------------------------

@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,dv,causal", [
    (2, 4, 4, 33, 33, 16, 16, False),
    (1, 6, 2, 40, 40, 8, 8, True),       # GQA: contiguous groups of 3
    (1, 4, 1, 17, 29, 8, 12, False),     # MQA, rectangular, d != dv
    (2, 8, 2, 21, 50, 16, 16, True),     # GQA, causal rectangular (bottom-right)
])
def test_matches_torch_sdpa_fp64(B, Hq, Hkv, Nq, Nk, d, dv, causal):
    """torch's scaled_dot_product_attention (CPU, fp64) is an independent implementation."""
    rng = np.random.default_rng(9 + Nq)
    q, k, v = _rand(rng, B, Hq, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, dv)
    scale = 1.0 / math.sqrt(d)
    o, lse = attention_forward(q, k, v, scale, causal)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    g = Hq // Hkv
    tk, tv = tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1)
    mask = None
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        mask = j <= i + (Nk - Nq)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)
    s = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
    if mask is not None:
        s = s.masked_fill(~mask, -math.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


def test_row_subset_is_exact():
    rng = np.random.default_rng(10)
    q, k, v = _rand(rng, 1, 2, 50, 8), _rand(rng, 1, 1, 50, 8), _rand(rng, 1, 1, 50, 8)
    o, lse = attention_forward(q, k, v, 0.3, True, row_block=7)
    rows = np.array([0, 3, 17, 49])
    o2, lse2 = attention_forward(q, k, v, 0.3, True, rows=rows)
    np.testing.assert_allclose(o2, o[:, :, rows], atol=1e-13)
    np.testing.assert_allclose(lse2, lse[:, :, rows], atol=1e-13)


# --- the online recurrence equals the two-pass definition ([AUT] §8; [PW] §4.2) -----------

def _adversarial_keys(rng, n, d, kind):
    q = _rand(rng, 1, d)
    base = _rand(rng, n, d)
    if kind == "random":
        return q, base
    # scores that rise (new max every tile) or fall (max fixed by the first key)
    direction = q[0] / np.linalg.norm(q[0])
    ramp = np.linspace(-6, 6, n) if kind == "rising" else np.linspace(6, -6, n)
    return q, base * 0.1 + ramp[:, None] * direction[None, :] * 3


@pytest.mark.parametrize("kind", ["random", "rising", "falling"])
def test_online_recurrence_equals_two_pass_all_tilings(kind):
    rng = np.random.default_rng(11)
    for n_keys in (1, 2, 5, 16):
        for d in (1, 3, 8):
            q1, k = _adversarial_keys(rng, n_keys, d, kind)
            q = np.concatenate([q1, _rand(rng, 3, d)])
            v = _rand(rng, n_keys, d)
            ref_o, ref_l = attention_forward(q[None, None], k[None, None], v[None, None], 0.9, False)
            for tile in range(1, n_keys + 1):
                o, lse = online_attention_rows(q, k, v, 0.9, tile)
                np.testing.assert_allclose(o, ref_o[0, 0], atol=1e-12, rtol=1e-12)
                np.testing.assert_allclose(lse, ref_l[0, 0], atol=1e-12, rtol=1e-12)


def test_online_recurrence_causal_and_empty_rows():
    rng = np.random.default_rng(12)
    n, Nk, d = 6, 9, 4
    q, k, v = _rand(rng, n, d), _rand(rng, Nk, d), _rand(rng, Nk, d)
    for offset in (-3, 0, 3):   # Nk - Nq offsets; -3 leaves rows with no visible key
        Nq = Nk - offset
        qq = _rand(rng, Nq, d) if Nq != n else q
        ref_o, ref_l = attention_forward(qq[None, None], k[None, None], v[None, None], 1.1, True)
        for tile in range(1, Nk + 1):
            o, lse = online_attention_rows(qq, k, v, 1.1, tile, causal_offset=offset)
            np.testing.assert_allclose(o, ref_o[0, 0], atol=1e-12)
            np.testing.assert_allclose(lse, ref_l[0, 0], atol=1e-12)


def test_equivalence_check_catches_a_missing_rescale():
    """Plant a mistake in a copy of the recurrence (drop the exp(m - m') factor on u):
    the equivalence check above must then fail on keys whose max keeps rising."""
    rng = np.random.default_rng(15)
    q, k = _adversarial_keys(rng, 8, 4, "rising")
    v = _rand(rng, 8, 4)

    def broken(tile):
        m, l, u = -np.inf, 0.0, np.zeros(4)
        for t0 in range(0, 8, tile):
            s = [float(q[0] @ k[j]) for j in range(t0, t0 + tile)]
            m_new = max([m] + s)
            corr = np.exp(m - m_new)
            p = [np.exp(x - m_new) for x in s]
            l = corr * l + sum(p)
            u = u + sum(pj * v[t0 + i] for i, pj in enumerate(p))   # planted: no corr
            m = m_new
        return u / l

    ref, _ = attention_forward(q[None, None], k[None, None], v[None, None], 1.0, False)
    good, _ = online_attention_rows(q, k, v, 1.0, 2)
    np.testing.assert_allclose(good[0], ref[0, 0, 0], atol=1e-12)
    assert np.abs(broken(2) - ref[0, 0, 0]).max() > 1e-3


def test_two_block_merge_equals_full_softmax():
    """[MG-A] §6.3: merging (m, l, O) of two key blocks reproduces the full result,
    at every split point, including a block that sees nothing."""
    rng = np.random.default_rng(13)
    Nq, Nk, d = 7, 12, 5
    q, k, v = _rand(rng, Nq, d), _rand(rng, Nk, d), _rand(rng, Nk, d)
    ref_o, ref_l = attention_forward(q[None, None], k[None, None], v[None, None], 0.8, False)
    for cut in range(1, Nk):
        stats = []
        for sl in (slice(0, cut), slice(cut, Nk)):
            o_b, lse_b = attention_forward(q[None, None], k[None, None, sl], v[None, None, sl], 0.8, False)
            m_b = (0.8 * q @ k[sl].T).max(axis=1)
            stats.append((m_b, np.exp(lse_b[0, 0] - m_b), o_b[0, 0]))
        m, l, o = merge_two_blocks(*stats[0], *stats[1])
        np.testing.assert_allclose(o, ref_o[0, 0], atol=1e-12)
        np.testing.assert_allclose(m + np.log(l), ref_l[0, 0], atol=1e-12)
    empty = (np.full(Nq, -np.inf), np.zeros(Nq), np.zeros((Nq, d)))
    m_full = (0.8 * q @ k.T).max(axis=1)
    full = (m_full, np.exp(ref_l[0, 0] - m_full), ref_o[0, 0])
    for a, b in ((empty, full), (full, empty)):
        m, l, o = merge_two_blocks(*a, *b)
        np.testing.assert_allclose(o, ref_o[0, 0], atol=1e-12)
    m, l, o = merge_two_blocks(*empty, *empty)
    assert (l == 0).all() and (o == 0).all()


# --- decode -------------------------------------------------------------------------------

def test_decode_matches_prefix_attention_and_sdpa():
    """Decode = one query over the cached prefix [0, L) ([IMR] prefill/decode; [PW] §3.1)."""
    rng = np.random.default_rng(14)
    B, Hq, Hkv, Lmax, d = 3, 8, 2, 40, 16
    q, kc, vc = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, Lmax, d), _rand(rng, B, Hkv, Lmax, d)
    seqlens = np.array([1, 23, 40])
    scale = 1 / math.sqrt(d)
    o, lse = attention_decode(q, kc, vc, seqlens, scale)
    for b in range(B):
        L = seqlens[b]
        tq = torch.from_numpy(q[b][:, None, :])
        tk = torch.from_numpy(kc[b, :, :L]).repeat_interleave(Hq // Hkv, dim=0)
        tv = torch.from_numpy(vc[b, :, :L]).repeat_interleave(Hq // Hkv, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
        np.testing.assert_allclose(o[b], ref[:, 0].numpy(), atol=1e-12)
        s = torch.einsum("hd,hjd->hj", tq[:, 0], tk) * scale
        np.testing.assert_allclose(lse[b], torch.logsumexp(s, -1).numpy(), atol=1e-12)
    # the cache tail past seqlens is never read
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[0, :, 1:] = 1e30
    vc2[1, :, 23:] = np.nan
    o2, lse2 = attention_decode(q, kc2, vc2, seqlens, scale)
    np.testing.assert_array_equal(o2, o)
    np.testing.assert_array_equal(lse2, lse)
    # length 1: the only cached value; length 0: zero output, -inf lse
    np.testing.assert_allclose(o[0], vc[0].repeat(Hq // Hkv, axis=0)[:, 0], atol=1e-15)
    o0, l0 = attention_decode(q, kc, vc, np.array([0, 0, 5]), scale)
    assert (o0[:2] == 0).all() and np.isneginf(l0[:2]).all()
    with pytest.raises(ValueError):
        attention_decode(q, kc, vc, np.array([1, 41, 2]), scale)


# --- paged decode with the new token appended -----------------------------------------------

def _sdpa_decode(q_b, keys, vals, scale, G):
    """torch SDPA (fp64) for one sequence: q_b [Hq, d], keys/vals [Hkv, L, d]."""
    tq = torch.from_numpy(q_b[:, None, :])
    tk = torch.from_numpy(keys).repeat_interleave(G, dim=0)
    tv = torch.from_numpy(vals).repeat_interleave(G, dim=0)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[:, 0].numpy()
    lse = torch.logsumexp(torch.einsum("hd,hjd->hj", tq[:, 0], tk) * scale, -1).numpy()
    return o, lse


@pytest.mark.parametrize("page_size", [4, 8, 16])
def test_paged_decode_gathers_pages_through_the_block_table(page_size):
    """Blocks of the KV cache need not be contiguous ([IMR] PagedAttention section;
    [PW] §3.3): position p of sequence b is row p % P of physical page
    block_table[b][p // P]. Checked against SDPA on keys gathered by that rule,
    with a shuffled page pool; permuting the physical pages (and the table) changes nothing."""
    rng = np.random.default_rng(31)
    B, Hq, Hkv, d, num_pages = 3, 8, 2, 16, 24
    seqlens = np.array([1, page_size * 2, page_size * 3 + 1])
    kp, vp = _rand(rng, num_pages, Hkv, page_size, d), _rand(rng, num_pages, Hkv, page_size, d)
    perm = rng.permutation(num_pages)
    bt = perm[: B * 6].reshape(B, 6)
    q = _rand(rng, B, Hq, d)
    scale = 1 / math.sqrt(d)
    o, lse, kp2, vp2 = attention_decode_paged(q, kp, vp, bt, seqlens, scale)
    np.testing.assert_array_equal(kp2, kp)  # no append: pages untouched
    for b in range(B):
        L = seqlens[b]
        keys = np.stack([kp[bt[b][p // page_size], :, p % page_size] for p in range(L)], axis=1)
        vals = np.stack([vp[bt[b][p // page_size], :, p % page_size] for p in range(L)], axis=1)
        ro, rl = _sdpa_decode(q[b], keys, vals, scale, Hq // Hkv)
        np.testing.assert_allclose(o[b], ro, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl, atol=1e-12)
    # relabel physical pages: same attention
    relabel = rng.permutation(num_pages)
    kp3, vp3 = np.empty_like(kp), np.empty_like(vp)
    kp3[relabel], vp3[relabel] = kp, vp
    o3, lse3, _, _ = attention_decode_paged(q, kp3, vp3, relabel[bt], seqlens, scale)
    np.testing.assert_allclose(o3, o, atol=1e-15)
    np.testing.assert_allclose(lse3, lse, atol=1e-15)


def test_paged_decode_appends_the_new_token_before_attending():
    """The new token's K/V is written at position seqlens[b] and attended to
    together with the cache ([PW] §3.1: the new token's K/V joins the cache)."""
    rng = np.random.default_rng(32)
    B, Hq, Hkv, d, P, num_pages = 4, 4, 1, 8, 4, 16
    seqlens = np.array([0, 3, 4, 7])  # 4: the append opens a new page
    kp, vp = _rand(rng, num_pages, Hkv, P, d), _rand(rng, num_pages, Hkv, P, d)
    bt = rng.permutation(num_pages)[: B * 3].reshape(B, 3)
    q, kn, vn = _rand(rng, B, Hq, d), _rand(rng, B, Hkv, d), _rand(rng, B, Hkv, d)
    scale = 0.7
    o, lse, kp2, vp2 = attention_decode_paged(q, kp, vp, bt, seqlens, scale, kn, vn)
    for b in range(B):
        L = seqlens[b]
        pg, row = bt[b][L // P], L % P
        np.testing.assert_array_equal(kp2[pg, :, row], kn[b])
        np.testing.assert_array_equal(vp2[pg, :, row], vn[b])
        gather = lambda pages: (np.stack([pages[bt[b][p // P], :, p % P] for p in range(L)], axis=1) if L
                                else np.zeros((Hkv, 0, d)))
        keys = np.concatenate([gather(kp), kn[b][:, None]], axis=1)
        vals = np.concatenate([gather(vp), vn[b][:, None]], axis=1)
        ro, rl = _sdpa_decode(q[b], keys, vals, scale, Hq // Hkv)
        np.testing.assert_allclose(o[b], ro, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl, atol=1e-12)
    # a cache of length 0 plus the appended token: the output is that token's value
    np.testing.assert_allclose(o[0], np.repeat(vn[0], Hq // Hkv, axis=0), atol=1e-15)
    # every other page row is left as it was
    changed = np.zeros(kp.shape[:1] + kp.shape[2:3], bool)
    for b in range(B):
        changed[bt[b][seqlens[b] // P], seqlens[b] % P] = True
    np.testing.assert_array_equal(kp2[~changed[:, None, :].repeat(Hkv, 1)], kp[~changed[:, None, :].repeat(Hkv, 1)])


# --- local (sliding-window) attention --------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Nq,Nk,window", [(20, 20, 5), (12, 30, 7), (30, 12, 4), (16, 16, 1), (16, 16, 40)])
def test_window_matches_sdpa_with_an_explicit_mask(causal, Nq, Nk, window):
    """Local window ([AUT] §2 Longformer; [PW] §6.1): query i sees key j iff
    |j - (i + Nk - Nq)| < w (and j <= i + Nk - Nq when causal). Checked
    against torch SDPA with a boolean mask built from that rule."""
    rng = np.random.default_rng(40 + window)
    B, Hq, Hkv, d = 1, 4, 2, 8
    q, k, v = _rand(rng, B, Hq, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, d)
    o, lse = attention_forward(q, k, v, 0.5, causal, window=window)
    i = np.arange(Nq)[:, None] + (Nk - Nq)
    j = np.arange(Nk)[None, :]
    allowed = np.abs(j - i) < window
    if causal:
        allowed &= j <= i
    rows = allowed.any(axis=1)
    tk = torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=1)
    tv = torch.from_numpy(v).repeat_interleave(Hq // Hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[:, :, rows]), tk, tv, attn_mask=torch.from_numpy(allowed[rows]), scale=0.5)
    np.testing.assert_allclose(o[:, :, rows], ref.numpy(), atol=1e-12)
    assert (o[:, :, ~rows] == 0).all() and np.isneginf(lse[:, :, ~rows]).all()
    if window >= Nq + Nk:  # a window wider than everything is no window
        o0, l0 = attention_forward(q, k, v, 0.5, causal)
        np.testing.assert_array_equal(o, o0)


def test_window_of_one_sees_only_the_aligned_key():
    rng = np.random.default_rng(47)
    q, k, v = _rand(rng, 1, 2, 10, 4), _rand(rng, 1, 2, 10, 4), _rand(rng, 1, 2, 10, 4)
    o, lse = attention_forward(q, k, v, 1.0, True, window=1)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    np.testing.assert_allclose(lse[0], np.einsum("hid,hid->hi", q[0], k[0]), atol=1e-12)


# --- rotary position embedding -----------------------------------------------------------------

def test_rope_scores_depend_only_on_relative_position():
    """[PW] §5.3: with RoPE the score of a query at m and a key at n depends
    only on m - n. Shift both positions by the same amount: same scores."""
    rng = np.random.default_rng(70)
    d = 16
    q, k = _rand(rng, 1, d), _rand(rng, 1, d)
    for m, n in [(5, 2), (100, 40), (7, 7)]:
        s0 = rope_rotate(q, [m]) @ rope_rotate(k, [n]).T
        for shift in (1, 37, 1000):
            s1 = rope_rotate(q, [m + shift]) @ rope_rotate(k, [n + shift]).T
            np.testing.assert_allclose(s1, s0, atol=1e-10)


def test_rope_is_a_pairwise_rotation():
    """Position 0 is the identity; each pair keeps its norm; pair 0 at position 1
    turns by exactly one radian (omega_0 = 1); a quarter turn maps (x, y) to (-y, x)."""
    rng = np.random.default_rng(71)
    x = _rand(rng, 3, 8)
    np.testing.assert_array_equal(rope_rotate(x, [0, 0, 0]), x)
    r = rope_rotate(x, [3, 9, 250])
    np.testing.assert_allclose(np.hypot(r[:, 0::2], r[:, 1::2]), np.hypot(x[:, 0::2], x[:, 1::2]), atol=1e-12)
    e = np.zeros((1, 8)); e[0, 0] = 1.0
    np.testing.assert_allclose(rope_rotate(e, [1])[0, :2], [math.cos(1.0), math.sin(1.0)], atol=1e-15)
    # base chosen so that pair 1 of d=4 turns by pi/2 at position 1: base^(-2/4) = pi/2
    b = (math.pi / 2) ** -2
    v = np.array([[0.0, 0.0, 3.0, 5.0]])
    np.testing.assert_allclose(rope_rotate(v, [1], base=b)[0, 2:], [-5.0, 3.0], atol=1e-12)


@pytest.mark.parametrize("Nq,Nk,window", [(40, 40, 0), (30, 45, 0), (40, 40, 7)])
def test_rope_row_subset_is_exact(Nq, Nk, window):
    """Asking for a subset of query rows gives those rows of the full result
    (the rows keep their positions: the rotation uses each row's own position)."""
    rng = np.random.default_rng(11)
    q, k, v = _rand(rng, 1, 2, Nq, 8), _rand(rng, 1, 1, Nk, 8), _rand(rng, 1, 1, Nk, 8)
    o, lse = attention_forward_rope(q, k, v, 0.3, True, base=100.0, window=window)
    rows = np.array([0, 1, Nq // 2, Nq - 1])
    o2, lse2 = attention_forward_rope(q, k, v, 0.3, True, base=100.0, window=window, rows=rows)
    np.testing.assert_allclose(o2, o[:, :, rows], atol=1e-13)
    np.testing.assert_allclose(lse2, lse[:, :, rows], atol=1e-13)


def test_rope_attention_matches_rotating_by_hand_and_rounding():
    rng = np.random.default_rng(72)
    B, Hq, Hkv, Nq, Nk, d = 1, 4, 2, 9, 13, 8
    q, k, v = _rand(rng, B, Hq, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, d)
    o, lse = attention_forward_rope(q, k, v, 0.3, True)
    theta_q = (np.arange(Nq) + Nk - Nq)[:, None] * 10000.0 ** (-np.arange(0, d, 2) / d)[None, :]
    qr = q.copy()
    qr[..., 0::2] = q[..., 0::2] * np.cos(theta_q) - q[..., 1::2] * np.sin(theta_q)
    qr[..., 1::2] = q[..., 0::2] * np.sin(theta_q) + q[..., 1::2] * np.cos(theta_q)
    qr = _nearest_bf16_by_table(qr)  # the rounding is pinned on its own below
    kr = _nearest_bf16_by_table(rope_rotate(k, np.arange(Nk)))
    o2, lse2 = attention_forward(qr, kr, v, 0.3, True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


# --- rounding fp64 -> bf16 (the RoPE reading: rotated operands are rounded once, to nearest, ties to even)

def _bf16_table():
    """Every finite non-negative bf16 value in increasing order, from the bit
    patterns (bf16_bits_to_f64 is pinned against all 65 536 patterns)."""
    vals = bf16_bits_to_f64(np.arange(0, 0x7F80, dtype=np.uint16))
    assert np.all(np.diff(vals) > 0)
    return vals


def _nearest_bf16_by_table(x):
    """Brute force: look |x| up between its two bf16 neighbours, pick the
    nearer one, on a tie the one whose bit pattern is even."""
    x = np.asarray(x, dtype=np.float64)
    tab = _bf16_table()
    ax = np.abs(x)
    i = np.clip(np.searchsorted(tab, ax, side="right") - 1, 0, tab.size - 1)  # tab[i] <= ax
    lo = tab[i]
    hi = np.where(i + 1 < tab.size, tab[np.minimum(i + 1, tab.size - 1)], np.inf)
    d_lo, d_hi = ax - lo, hi - ax
    # above the largest finite value the upper neighbour is +inf at distance "one more step"
    top = i + 1 >= tab.size
    d_hi = np.where(top, (tab[-1] - tab[-2]) - d_lo, d_hi)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (i % 2 == 1))
    return np.copysign(np.where(pick_hi, hi, lo), x)


def test_round_to_bf16_hand_cases():
    """Cases fixed by round-to-nearest-even alone (no conversion library in between):
    bf16 keeps 8 significant bits, so next to 1 its spacing is 2^-7."""
    u = 2.0 ** -7
    cases = [
        (1 + u / 2 + 2.0 ** -30, 1 + u),  # just above the midpoint: up (a detour through fp32 gives 1.0)
        (1 + u / 2, 1.0),                 # the midpoint: to the even neighbour 1.0
        (1 + u / 2 - 2.0 ** -40, 1.0),    # just below: down
        (1 + 3 * u / 2, 1 + 2 * u),       # midpoint between odd 1+u and even 1+2u: up to even
        (1 + u, 1 + u),                   # representable values stay
        (2 - u / 4, 2.0),                 # rounding up carries into the next binade
        (0.0, 0.0),
    ]
    for scale in (1.0, -1.0, 2.0 ** -100, -(2.0 ** 90), 2.0 ** 120):
        for x, want in cases:
            got = round_to_bf16(np.array([x * scale]))[0]
            assert got == want * scale, (x, scale, got, want * scale)


def test_round_to_bf16_extremes():
    big = (2 - 2.0 ** -7) * 2.0 ** 127  # largest finite bf16
    half_step = 2.0 ** (127 - 8)
    tiny = 2.0 ** -133                  # smallest subnormal bf16
    x = np.array([big, big + half_step * 0.99, big + half_step, -(big + half_step), 1.5 * tiny, 2.5 * tiny,
                  0.5 * tiny, 0.5 * tiny * (1 + 2.0 ** -20), np.inf, -np.inf, 1e-300])
    want = np.array([big, big, np.inf, -np.inf, 2 * tiny, 2 * tiny, 0.0, tiny, np.inf, -np.inf, 0.0])
    np.testing.assert_array_equal(round_to_bf16(x), want)
    assert np.isnan(round_to_bf16(np.array([np.nan]))[0])
    assert np.signbit(round_to_bf16(np.array([-1e-300]))[0])


def test_round_to_bf16_matches_brute_force_between_every_pair_of_neighbours():
    """For every pair of adjacent finite bf16 values: points at 1/4, just below,
    at, and just above the midpoint, and at 3/4 of the gap, both signs."""
    tab = _bf16_table()
    lo, hi = tab[:-1], tab[1:]
    gap = hi - lo
    pts = [lo + gap * f for f in (0.25, 0.75)]
    mid = lo + gap / 2
    pts += [mid, np.nextafter(mid, -np.inf), np.nextafter(mid, np.inf)]
    x = np.concatenate(pts)
    x = np.concatenate([x, -x])
    np.testing.assert_array_equal(round_to_bf16(x), _nearest_bf16_by_table(x))
    # and random magnitudes over the whole range
    rng = np.random.default_rng(73)
    y = rng.standard_normal(200000) * 2.0 ** rng.uniform(-140, 127, 200000)
    np.testing.assert_array_equal(round_to_bf16(y), _nearest_bf16_by_table(y))


# ---------------------------------------------------------------- backward pass


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 2, 2, 9, 9, 4, False),
    (2, 4, 2, 13, 13, 8, True),      # GQA: the group's dK, dV contributions add
    (1, 3, 1, 6, 11, 5, True),       # MQA, bottom-right causal with Nq < Nk
    (1, 2, 1, 12, 7, 8, False),      # cross-attention, Nq > Nk
])
def test_backward_matches_torch_autograd_fp64(B, Hq, Hkv, Nq, Nk, d, causal):
    """torch autograd through its own matmul / masked softmax (fp64) is an
    independent derivation of the same gradients."""
    rng = np.random.default_rng(40 + Nq)
    q, k, v = _rand(rng, B, Hq, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, d)
    do = _rand(rng, B, Hq, Nq, d)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = attention_backward(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    g = Hq // Hkv
    s = torch.einsum("bhid,bhjd->bhij", tq, tk.repeat_interleave(g, dim=1)) * scale
    if causal:
        keep = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
        s = s.masked_fill(~keep, -math.inf)
    o = torch.softmax(s, dim=-1) @ tv.repeat_interleave(g, dim=1)
    o.backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_backward_equals_central_finite_differences():
    """Brute force: perturb every input entry of L = sum(dO * O) and difference
    the forward definition."""
    rng = np.random.default_rng(41)
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 3, 4, 3
    q, k, v = _rand(rng, B, Hq, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, d)
    do = _rand(rng, B, Hq, Nq, d)
    scale = 0.7
    dq, dk, dv = attention_backward(q, k, v, do, scale, True)

    def loss(qq, kk, vv):
        return float((attention_forward(qq, kk, vv, scale, True)[0] * do).sum())

    eps = 1e-6
    for x, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += eps
            args_m[which][idx] -= eps
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(grad, num, atol=1e-8)


def test_backward_shift_and_sum_invariants():
    """Adding one vector to every key leaves each softmax row unchanged, so
    sum_j dK_j = 0; each row of P sums to 1, so sum_j dV_j = sum_i dO_i over
    rows that see a key; identical keys make every row uniform, so dQ = 0."""
    rng = np.random.default_rng(42)
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 17, 23, 8
    q, k, v = _rand(rng, B, Hq, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, d)
    do = _rand(rng, B, Hq, Nq, d)
    for causal in (False, True):
        dq, dk, dv = attention_backward(q, k, v, do, 0.4, causal)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
        do_sum = do.reshape(B, Hkv, Hq // Hkv, Nq, d).sum(axis=(2, 3))
        np.testing.assert_allclose(dv.sum(axis=2), do_sum, atol=1e-12)
    k_same = np.broadcast_to(k[:, :, :1], k.shape).copy()
    dq, _, _ = attention_backward(q, k_same, v, do, 0.4, False)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)


def test_backward_empty_rows_and_linearity_in_do():
    rng = np.random.default_rng(43)
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 9, 5, 4   # causal, Nq > Nk: rows 0..3 see no key
    q, k, v = _rand(rng, B, Hq, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, d)
    do1, do2 = _rand(rng, B, Hq, Nq, d), _rand(rng, B, Hq, Nq, d)
    g1 = attention_backward(q, k, v, do1, 0.5, True)
    np.testing.assert_array_equal(g1[0][:, :, :Nq - Nk], 0.0)
    g2 = attention_backward(q, k, v, do2, 0.5, True)
    g12 = attention_backward(q, k, v, 2.0 * do1 - 3.0 * do2, 0.5, True)
    for a, b_, c in zip(g1, g2, g12):
        np.testing.assert_allclose(c, 2.0 * a - 3.0 * b_, atol=1e-12)


def test_backward_row_subsets_are_exact():
    rng = np.random.default_rng(44)
    q, k, v = _rand(rng, 1, 4, 40, 8), _rand(rng, 1, 2, 40, 8), _rand(rng, 1, 2, 40, 8)
    do = _rand(rng, 1, 4, 40, 8)
    full = attention_backward(q, k, v, do, 0.35, True, row_block=9)
    qr, kr = np.array([0, 5, 39]), np.array([1, 20, 38, 39])
    dq, dk, dv = attention_backward(q, k, v, do, 0.35, True, q_rows=qr, k_rows=kr, row_block=16)
    np.testing.assert_allclose(dq, full[0][:, :, qr], atol=1e-13)
    np.testing.assert_allclose(dk, full[1][:, :, kr], atol=1e-13)
    np.testing.assert_allclose(dv, full[2][:, :, kr], atol=1e-13)


def test_sum_invariant_catches_a_dropped_softmax_correction():
    """The invariants above are sensitive: leaving out the row term of the
    softmax Jacobian (dS = P * dP) breaks sum_j dK_j = 0."""
    rng = np.random.default_rng(45)
    q, k, v = _rand(rng, 1, 1, 6, 4), _rand(rng, 1, 1, 6, 4), _rand(rng, 1, 1, 6, 4)
    do = _rand(rng, 1, 1, 6, 4)
    S = 0.5 * q[0, 0] @ k[0, 0].T
    P = np.exp(S - S.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    wrong_dk = 0.5 * (P * (do[0, 0] @ v[0, 0].T)).T @ q[0, 0]
    assert np.abs(wrong_dk.sum(axis=0)).max() > 1e-3
    _, dk, _ = attention_backward(q, k, v, do, 0.5, False)
    assert np.abs(dk[0, 0].sum(axis=0)).max() < 1e-12


def test_backward_term_magnitudes():
    """The magnitude sums bound the gradients (triangle inequality), equal them
    where every term is non-negative, and do not change the gradients; the
    Dl sensitivities bound the first-order move of dq, dk when O's
    components are perturbed by at most e_it relatively."""
    rng = np.random.default_rng(46)
    q, k, v = _rand(rng, 1, 4, 21, 8), _rand(rng, 1, 2, 21, 8), _rand(rng, 1, 2, 21, 8)
    do = _rand(rng, 1, 4, 21, 8)
    plain = attention_backward(q, k, v, do, 0.4, True)
    dq, dk, dv, m = attention_backward(q, k, v, do, 0.4, True, magnitudes=True)
    for a, b_ in zip(plain, (dq, dk, dv)):
        np.testing.assert_array_equal(a, b_)
    for g, t in ((dq, m["tq"]), (dk, m["tk"]), (dv, m["tv"])):
        assert (t >= np.abs(g) - 1e-12).all()
    _, _, dv_pos, m_pos = attention_backward(q, k, v, np.abs(do), 0.4, True, magnitudes=True)
    np.testing.assert_allclose(m_pos["tv"], dv_pos, atol=1e-12)   # P >= 0 and dO >= 0: no cancellation
    # one key per row: dS = 0, so dq has no terms; Dl still moves dq
    _, _, _, m1 = attention_backward(q, k[:, :, :1], v[:, :, :1], do, 0.4, False, magnitudes=True)
    np.testing.assert_allclose(m1["tq"], 0.0, atol=1e-12)
    assert (m1["sq"] > 0).all()
    # dO = 0: nothing moves
    _, _, _, m0 = attention_backward(q, k, v, np.zeros_like(do), 0.4, True, magnitudes=True)
    assert np.abs(m0["sq"]).max() == 0 and np.abs(m0["sk"]).max() == 0
    # brute force for one row: perturbing Dl by its bound r moves dq by at most sq
    B, H, N, d = 1, 1, 6, 4
    q1, k1, v1, do1 = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d), _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    S = 0.5 * q1[0, 0] @ k1[0, 0].T
    P = np.exp(S - S.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    e = np.sqrt((P ** 2) @ (v1[0, 0] ** 2)) + np.abs(P @ v1[0, 0])
    r = np.sqrt(((do1[0, 0] * e) ** 2).sum(axis=1))
    moved = 0.5 * (P * r[:, None]) @ k1[0, 0]            # dq change for Dl -> Dl - r
    _, _, _, mm = attention_backward(q1, k1, v1, do1, 0.5, False, magnitudes=True)
    assert (np.abs(moved) <= mm["sq"][0, 0] + 1e-12).all()
