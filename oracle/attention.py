"""Plain fp64 definition of exact scaled-dot-product attention. TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU arms import this file.
Source key ([MG-A], [MG-B], [AUT], [IMR], [PW]) is spelled out in
``oracle/__init__.py``; each function names the passage it follows.

Readings taken where the pages are silent:
  * the score scale is applied before the mask; masked scores are -inf;
  * causal with Nq != Nk aligns the last query with the last key: query i sees
    key j iff j <= i + (Nk - Nq) (equal to the pages' j <= i when Nq == Nk);
  * a query row that sees no key has O = 0 and LSE = -inf;
  * LSE is the natural log of the sum of exp over the visible *scaled* scores;
  * GQA groups are contiguous: query head h reads K/V head h // (Hq // Hkv);
  * decode attends to cache rows [0, seqlens[b]) with no mask (the caller has
    already appended the new token's K/V).
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode raw bf16 bit patterns exactly.

    bf16 is the upper 16 bits of an IEEE-754 binary32 value, so shifting the
    pattern into the high half of a 32-bit word and widening is exact.
    """
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _kv_head(h: int, Hq: int, Hkv: int) -> int:
    """Query head h shares the K/V head of its group ([PW] §2.3, MQA/GQA)."""
    return h // (Hq // Hkv)


def _two_pass_softmax(S: np.ndarray):
    """Row softmax of a fully materialised score block ([MG-A] §2.4).

    Pass 1 takes each row's max m and Z = sum_j exp(S_ij - m); pass 2 forms
    P_ij = exp(S_ij - m) / Z. Subtracting the row max only changes the
    representation, not the probabilities ([AUT] §8). Returns (P, lse) with
    lse = m + ln Z. Rows whose scores are all -inf give P = 0, lse = -inf.
    """
    m = S.max(axis=1, initial=-np.inf)  # a row with no keys at all has max -inf
    live = np.isfinite(m)
    P = np.zeros_like(S)
    Z = np.zeros_like(m)
    E = np.exp(S[live] - m[live, None])  # masked entries: exp(-inf) = 0
    Z[live] = E.sum(axis=1)
    P[live] = E / Z[live, None]
    lse = np.full(m.shape, -np.inf)
    lse[live] = m[live] + np.log(Z[live])
    return P, lse


def attention_forward(q, k, v, scale: float, causal: bool, rows=None, row_block: int = 1024, window: int = 0):
    """O = softmax(scale * Q K^T + mask) V per (batch, query head), and the LSE.

    q: [B, Hq, Nq, d]; k, v: [B, Hkv, Nk, d] (float64). Returns o [B, Hq, R, d]
    and lse [B, Hq, R] where R = Nq, or len(rows) when a subset of query rows
    is asked for (the definition is row-wise, so a subset is exact).

    Steps ([MG-A] §2.2-§2.4, §4.1; [PW] §2.1): materialise
    S_ij = scale * q_i . k_j for every visible pair; put -inf where the causal
    rule hides key j from query i ([IMR], masking section); two-pass softmax
    per row; O = P V. Rows are processed in blocks of ``row_block`` only to
    bound memory: each row's full score vector is materialised before its
    softmax, which is the same definition.

    window > 0 adds a local window (Longformer-style local attention, [AUT]
    §2 Longformer comparison; [PW] §6.1 sliding-window attention, O(n*w)):
    query i, aligned with key i + (Nk - Nq), sees key j only if
    |j - (i + Nk - Nq)| < window; with causal also j <= i + Nk - Nq.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, dv = v.shape
    assert k.shape == (B, Hkv, Nk, d) and Hq % Hkv == 0
    rows = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.zeros((B, Hq, rows.size, dv))
    lse = np.full((B, Hq, rows.size), -np.inf)
    keys = np.arange(Nk)
    for b in range(B):
        for h in range(Hq):
            kh = k[b, _kv_head(h, Hq, Hkv)]
            vh = v[b, _kv_head(h, Hq, Hkv)]
            for r0 in range(0, rows.size, row_block):
                ri = rows[r0:r0 + row_block]
                S = scale * (q[b, h, ri] @ kh.T)
                diag = ri[:, None] + (Nk - Nq)  # the key each query row is aligned with
                if causal:
                    S = np.where(keys[None, :] > diag, -np.inf, S)
                if window > 0:
                    S = np.where(np.abs(keys[None, :] - diag) >= window, -np.inf, S)
                P, l = _two_pass_softmax(S)
                o[b, h, r0:r0 + ri.size] = P @ vh
                lse[b, h, r0:r0 + ri.size] = l
    return o, lse


def attention_backward(q, k, v, do, scale: float, causal: bool, q_rows=None, k_rows=None, row_block: int = 1024,
                       magnitudes: bool = False):
    """Gradients of O = softmax(scale * Q K^T + mask) V with respect to Q, K, V.

    Given dO = dL/dO for some loss L, returns (dq, dk, dv) = dL/dQ, dL/dK,
    dL/dV. The pages name the backward pass as the reason the score matrix is
    stored in standard attention ([MG-A] §3.3) and say the tiled method
    instead recomputes it from Q and K ([MG-B] §3.2, engineering results);
    the exact tiled method is to be checked on its gradients as well as its
    outputs ([AUT] method table, exact tiled attention row; verification
    protocol, second step). They give no formulas, so this is the chain rule
    through the forward definition, written out:

      S = scale * Q K^T (masked entries -inf), P = row softmax(S), O = P V
      dV = P^T dO                      (O is linear in V)
      dP = dO V^T
      dS_ij = P_ij * (dP_ij - sum_k P_ik dP_ik)   (Jacobian of a row softmax)
      dQ = scale * dS K,  dK = scale * dS^T Q

    With GQA the query heads of a group share one K/V head, so their dK and
    dV contributions add. Masked entries have P = 0, hence dS = 0; a row with
    no visible key contributes nothing and gets dq = 0.

    q, do: [B, Hq, Nq, d]; k, v: [B, Hkv, Nk, d] (float64). q_rows / k_rows
    select which query rows of dq and which key rows of dk, dv are returned
    (all by default); every query row's full score vector is still
    materialised, in blocks of ``row_block`` rows, before its softmax.

    magnitudes=True returns (dq, dk, dv, mags), mags holding the scales that
    rounding errors of an implementation are measured against (test use):
      tq, tk, tv  per element, the sum of the absolute values of the terms it
                  adds up (scale |dS| |K|, scale |dS|^T |Q|, P^T |dO|); a sum
                  of large cancelling terms can be much smaller than this.
      sq, sk      how far dq, dk move when Dl is formed from an O whose
                  components carry relative errors of size one (first order):
                  with e_it = sqrt(sum_j P_ij^2 v_jt^2) + |O_it| (the size of
                  O_it and of the spread of its terms), Dl_i moves by about
                  r_i = sqrt(sum_t dO_it^2 e_it^2), so dq_it by
                  scale r_i sum_j P_ij |k_jt| and dk_jt by
                  scale sum_i P_ij r_i |q_it|.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, dv_ = v.shape
    assert k.shape == (B, Hkv, Nk, d) and do.shape == (B, Hq, Nq, dv_) and Hq % Hkv == 0
    q_rows = np.arange(Nq) if q_rows is None else np.asarray(q_rows, dtype=np.int64)
    k_rows = np.arange(Nk) if k_rows is None else np.asarray(k_rows, dtype=np.int64)
    dq = np.zeros((B, Hq, q_rows.size, d))
    dk = np.zeros((B, Hkv, k_rows.size, d))
    dv = np.zeros((B, Hkv, k_rows.size, dv_))
    tq, tk, tv = np.zeros_like(dq), np.zeros_like(dk), np.zeros_like(dv)
    sq, sk = np.zeros_like(dq), np.zeros_like(dk)
    keys = np.arange(Nk)
    want_q = np.zeros(Nq, dtype=bool)
    want_q[q_rows] = True
    q_pos = np.full(Nq, -1)
    q_pos[q_rows] = np.arange(q_rows.size)
    for b in range(B):
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            kh, vh = k[b, g], v[b, g]
            for r0 in range(0, Nq, row_block):
                ri = np.arange(r0, min(Nq, r0 + row_block))
                if k_rows.size == 0 and not want_q[ri].any():
                    continue
                S = scale * (q[b, h, ri] @ kh.T)
                if causal:
                    S = np.where(keys[None, :] > ri[:, None] + (Nk - Nq), -np.inf, S)
                P, _ = _two_pass_softmax(S)
                dP = do[b, h, ri] @ vh.T
                dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                if magnitudes:
                    e = np.sqrt((P ** 2) @ (vh ** 2)) + np.abs(P @ vh)
                    r = np.sqrt(((do[b, h, ri] * e) ** 2).sum(axis=1))
                sel = want_q[ri]
                if sel.any():
                    dq[b, h, q_pos[ri[sel]]] = scale * (dS[sel] @ kh)
                    if magnitudes:
                        tq[b, h, q_pos[ri[sel]]] = scale * (np.abs(dS[sel]) @ np.abs(kh))
                        sq[b, h, q_pos[ri[sel]]] = scale * r[sel, None] * (P[sel] @ np.abs(kh))
                if k_rows.size:
                    dv[b, g] += P[:, k_rows].T @ do[b, h, ri]
                    dk[b, g] += scale * (dS[:, k_rows].T @ q[b, h, ri])
                    if magnitudes:
                        tv[b, g] += P[:, k_rows].T @ np.abs(do[b, h, ri])
                        tk[b, g] += scale * (np.abs(dS[:, k_rows]).T @ np.abs(q[b, h, ri]))
                        sk[b, g] += scale * ((P[:, k_rows] * r[:, None]).T @ np.abs(q[b, h, ri]))
    if magnitudes:
        return dq, dk, dv, {"tq": tq, "tk": tk, "tv": tv, "sq": sq, "sk": sk}
    return dq, dk, dv


def attention_decode(q, k_cache, v_cache, seqlens, scale: float):
    """One decode step: each sequence's new query attends to its cached keys.

    q: [B, Hq, d]; k_cache, v_cache: [B, Hkv, Lmax, d]; seqlens: [B] ints in
    [0, Lmax]. The new token's query reads the cached K/V of positions
    0..seqlens[b]-1 ([IMR], prefill/decode section; [PW] §3.1), with GQA head
    sharing ([PW] §3.2). Returns o [B, Hq, d] and lse [B, Hq]; a sequence of
    length 0 gives o = 0 and lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    _, Hkv, Lmax, dv = v_cache.shape
    o = np.zeros((B, Hq, dv))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        L = int(seqlens[b])
        if not 0 <= L <= Lmax:
            raise ValueError(f"seqlens[{b}]={L} outside [0, {Lmax}]")
        for h in range(Hq):
            kvh = _kv_head(h, Hq, Hkv)
            S = scale * (q[b, h][None, :] @ np.asarray(k_cache[b, kvh, :L], np.float64).T)
            P, l = _two_pass_softmax(S)
            o[b, h] = (P @ np.asarray(v_cache[b, kvh, :L], np.float64))[0]
            lse[b, h] = l[0]
    return o, lse


def rope_rotate(x, positions, base: float = 10000.0):
    """Rotary position embedding of [..., n, d] vectors ([PW] §5.3).

    The d components are split into pairs (2i, 2i+1); the pair of a vector at
    position m is rotated by the angle m * base**(-2i/d):
        x'_{2i}   = x_{2i} cos(theta) - x_{2i+1} sin(theta)
        x'_{2i+1} = x_{2i} sin(theta) + x_{2i+1} cos(theta)
    so that the score of a query at m and a key at n depends on m - n only.
    positions: [n] integers. fp64 throughout.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    i = np.arange(d // 2)
    theta = np.asarray(positions, dtype=np.float64)[:, None] * base ** (-2.0 * i / d)[None, :]
    c, s = np.cos(theta), np.sin(theta)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return out


def round_to_bf16(x):
    """fp64 -> nearest bf16 value (ties to even), returned as fp64.

    One rounding, straight from fp64: bf16 keeps 8 significant bits, so in the
    binade [2^(e-1), 2^e) of |x| its values are the integer multiples of
    2^(e-8) (below the smallest normal, 2^-126, the spacing stays 2^-133). The
    result is the multiple nearest |x|; an exact half goes to the even
    multiple. Magnitudes that round to 2^128 or more become infinite (the
    largest finite bf16 is (2 - 2^-7) 2^127); NaN, +-inf and +-0 pass through.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    fin = np.isfinite(x) & (x != 0.0)
    ax = np.abs(x[fin])
    _, e = np.frexp(ax)                          # ax = frac * 2^e, 0.5 <= frac < 1
    spacing = np.ldexp(1.0, np.maximum(e, -125) - 8)
    t = ax / spacing                             # exact: a power-of-two scaling
    n = np.floor(t)
    rem = t - n                                  # exact fraction in [0, 1)
    up = (rem > 0.5) | ((rem == 0.5) & (np.fmod(n, 2.0) == 1.0))
    mag = (n + up) * spacing
    mag = np.where(mag >= 2.0 ** 128, np.inf, mag)
    out[fin] = np.copysign(mag, x[fin])
    return out


def attention_forward_rope(q, k, v, scale: float, causal: bool, base: float = 10000.0, window: int = 0, rows=None):
    """Prefill with RoPE applied to Q and K first ([PW] §5.3: it acts on Q
    and K, not on the input). Key j sits at position j and query i at
    position i + (Nk - Nq), the same alignment as the causal rule. The
    rotated Q and K are rounded to bf16 (the inputs' type) before the scores,
    then the plain definition (attention_forward) is applied, on the query
    rows ``rows`` only when given (as there)."""
    Nq, Nk = q.shape[-2], k.shape[-2]
    qr = round_to_bf16(rope_rotate(q, np.arange(Nq) + (Nk - Nq), base))
    kr = round_to_bf16(rope_rotate(k, np.arange(Nk), base))
    return attention_forward(qr, kr, v, scale, causal, rows=rows, window=window)


def attention_decode_paged(q, k_pages, v_pages, block_table, seqlens, scale: float, k_new=None, v_new=None):
    """Decode step over a paged KV cache, with the new token's K/V appended first.

    The KV cache is cut into fixed-size blocks ("pages") that are allocated on
    demand and need not be contiguous; a per-sequence block table maps the
    logical page number to the physical page ([IMR], section "FlashAttention 和
    PagedAttention 不是同一种答案"; [PW] §3.3).

    k_pages, v_pages: [num_pages, Hkv, page_size, d]; token position p of
    sequence b lives in physical page block_table[b][p // page_size], row
    p % page_size. seqlens[b] is the number of tokens already cached.
    If k_new / v_new ([B, Hkv, d]) are given, they are first written at
    position seqlens[b] (the caller has reserved that page) and the query
    attends to positions 0..seqlens[b]; otherwise to 0..seqlens[b]-1.

    Written as: apply the append to copies of the pages, gather each
    sequence's positions page by page into a contiguous cache, then take the
    plain decode definition (attention_decode). Returns (o, lse, k_pages_after,
    v_pages_after).
    """
    kp = np.array(k_pages, dtype=np.float64, copy=True)
    vp = np.array(v_pages, dtype=np.float64, copy=True)
    num_pages, Hkv, page_size, d = kp.shape
    B = len(seqlens)
    lens = [int(x) for x in seqlens]
    if k_new is not None:
        for b in range(B):
            pos = lens[b]
            page = int(block_table[b][pos // page_size])
            kp[page, :, pos % page_size] = np.asarray(k_new[b], np.float64)
            vp[page, :, pos % page_size] = np.asarray(v_new[b], np.float64)
        lens = [x + 1 for x in lens]
    Lmax = max(1, max(lens))
    kc = np.zeros((B, Hkv, Lmax, d))
    vc = np.zeros((B, Hkv, Lmax, vp.shape[-1]))
    for b in range(B):
        for pos in range(lens[b]):
            page = int(block_table[b][pos // page_size])
            kc[b, :, pos] = kp[page, :, pos % page_size]
            vc[b, :, pos] = vp[page, :, pos % page_size]
    o, lse = attention_decode(q, kc, vc, np.array(lens), scale)
    return o, lse, kp, vp


def online_attention_rows(q, k, v, scale: float, tile: int, causal_offset=None):
    """The blockwise recurrence of [AUT] §8 (its first two equations), literally.

    q: [n, d]; k, v: [Nk, d]. Keys are visited in tiles of ``tile``. Per query
    row the state is the running max m, the denominator l and the
    un-normalised weighted sum u. For each tile with scores s_j:
        m' = max(m, max_j s_j)
        l' = exp(m - m') l + sum_j exp(s_j - m')
        u' = exp(m - m') u + sum_j exp(s_j - m') v_j
    and finally o = u / l, lse = m + ln l. ``causal_offset`` (if given) hides
    key j from query i when j > i + causal_offset. Starting state m = -inf,
    l = 0, u = 0; a tile in which nothing is visible yet leaves the state
    unchanged (exp(-inf - -inf) is never formed). Pure Python loops: meant
    only for the tiny brute-force equivalence tests.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, Nk = q.shape[0], k.shape[0]
    o = np.zeros((n, v.shape[1]))
    lse = np.full(n, -np.inf)
    for i in range(n):
        m, l, u = -np.inf, 0.0, np.zeros(v.shape[1])
        for t0 in range(0, Nk, tile):
            js = range(t0, min(t0 + tile, Nk))
            s = [(-np.inf if causal_offset is not None and j > i + causal_offset
                  else scale * float(q[i] @ k[j])) for j in js]
            m_new = max([m] + s)
            if m_new == -np.inf:
                continue
            corr = np.exp(m - m_new)
            p = [np.exp(sj - m_new) for sj in s]
            l = corr * l + sum(p)
            u = corr * u + sum(pj * v[j] for pj, j in zip(p, js))
            m = m_new
        if l > 0:
            o[i] = u / l
            lse[i] = m + np.log(l)
    return o, lse


def merge_two_blocks(m1, l1, o1, m2, l2, o2):
    """Combine the softmax statistics of two key blocks ([MG-A] §6.3 steps 2-4).

    Each block carries its row max m, its local exp-sum l (relative to m) and
    its block-normalised output o. With m_new = max(m1, m2):
        l_new = l1 exp(m1 - m_new) + l2 exp(m2 - m_new)
        o_new = (l1 o1 exp(m1 - m_new) + l2 o2 exp(m2 - m_new)) / l_new
    A block that saw no key (m = -inf, l = 0) contributes nothing. Works on
    scalars or on aligned arrays of rows (o has one more trailing axis).
    """
    m1, l1, m2, l2 = (np.asarray(x, np.float64) for x in (m1, l1, m2, l2))
    o1, o2 = np.asarray(o1, np.float64), np.asarray(o2, np.float64)
    m_new = np.maximum(m1, m2)
    live = np.isfinite(m_new)
    safe = np.where(live, m_new, 0.0)
    a1 = np.where(np.isfinite(m1), np.exp(np.where(np.isfinite(m1), m1, 0.0) - safe), 0.0) * l1
    a2 = np.where(np.isfinite(m2), np.exp(np.where(np.isfinite(m2), m2, 0.0) - safe), 0.0) * l2
    l_new = a1 + a2
    denom = np.where(l_new > 0, l_new, 1.0)
    o_new = (a1[..., None] * o1 + a2[..., None] * o2) / denom[..., None]
    return m_new, l_new, o_new


def score_bytes(n: int, heads: int = 1, bytes_per_score: int = 4) -> int:
    """Bytes of an explicitly stored score matrix: heads * n^2 * bytes ([AUT] §4, §6)."""
    return heads * n * n * bytes_per_score


def kv_cache_bytes(layers: int, n: int, h_kv: int, d_h: int, bytes_per_scalar: int) -> int:
    """KV cache size 2 * L * n * h_kv * d_h * b ([AUT] §9, third equation; [PW] §3.2)."""
    return 2 * layers * n * h_kv * d_h * bytes_per_scalar
