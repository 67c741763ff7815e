"""Shared helpers for the GPU-vs-oracle parity tests.

The bar (one set of numbers for every case): compared against the fp64
oracle on the same bf16 inputs, the bf16 output must have max-abs error
<= 1e-2 and mean-abs error <= 1e-3, and the fp32 LSE max-abs error <= 1e-3.
Rows the oracle marks as seeing no key must come back as o = 0, lse = -inf.

Gradients (dQ, dK, dV) have no stated bar; the one used is derived from the
arithmetic of the backward path, with u = 2^-8 the unit roundoff of bf16.
Each gradient element g is a sum of terms in which one factor (P or dS) was
rounded to bf16 (error <= u |term|), Dl comes from the bf16 forward output
(an error of the same order), and g is rounded to bf16 (<= u |g|). With T the
sum of the terms' absolute values (the oracle returns it: a sum of large
cancelling terms, e.g. a causal row that sees few keys, can be much smaller
than T) and S the oracle's first-order sensitivity of g to errors of relative
size one in the components of O (Dl = sum_t dO_t O_t uses the bf16 forward
output, whose components are off by about u; S is 0 for dV), every element
must satisfy
    |g - g_ref| <= 4u (T + S) + u |g_ref| + 2^-16
(2^-16 covers the fp32 accumulation residue where T and S vanish), and over
a tensor mean |g - g_ref| <= u mean(T + S).
"""
import numpy as np
import torch

import oracle
from exact_scaled_dot_03_b300.workloads import bf16_bits

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3
BF16_U = 2.0 ** -8
GRAD_TERMS = 4 * BF16_U
GRAD_FLOOR = 2.0 ** -16


def f64(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> exact fp64 numpy, decoded by the oracle."""
    return oracle.bf16_bits_to_f64(bf16_bits(t.detach().cpu()))


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Assert the parity bar; returns the measured errors for reporting."""
    o = f64(o_gpu) if o_gpu.dtype == torch.bfloat16 else o_gpu.detach().cpu().double().numpy()
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    res = {"o_max_abs": float(err.max()) if err.size else 0.0,
           "o_mean_abs": float(err.mean()) if err.size else 0.0,
           # what bf16 rounding of the exact answer alone would cost (a floor, not a failure)
           "bf16_floor": float(np.abs(oracle.bf16_bits_to_f64(bf16_bits(torch.from_numpy(o_ref).to(torch.bfloat16)))
                                      - o_ref).max()) if err.size else 0.0}
    assert res["o_max_abs"] <= O_MAX_ABS, f"{what}: {res}"
    assert res["o_mean_abs"] <= O_MEAN_ABS, f"{what}: {res}"
    if lse_gpu is not None:
        lse = lse_gpu.detach().cpu().double().numpy()
        empty = np.isneginf(lse_ref)
        assert (np.isneginf(lse) == empty).all(), f"{what}: -inf pattern of the LSE differs"
        assert (o[empty] == 0).all(), f"{what}: rows with no key must be 0"
        lerr = np.abs(lse[~empty] - lse_ref[~empty])
        res["lse_max_abs"] = float(lerr.max()) if lerr.size else 0.0
        assert res["lse_max_abs"] <= LSE_MAX_ABS, f"{what}: {res}"
    return res


def compare_any_shape(o_gpu, lse_gpu, o_ref, lse_ref, a_ref, what=""):
    """The forward bar for shapes of any kind (the randomised sweep).

    The stated bar (max-abs 1e-2, mean-abs 1e-3) is met by the workloads,
    whose outputs average many keys. With only a few keys, |o| approaches the
    |v| it averages, and the arithmetic cannot meet an absolute 1e-2 there. The
    kernels round each probability p_j to bf16 before the P.V product (relative
    error <= u = 2^-8). The denominator stays fp32. Rounding o to bf16 adds
    another <= u |o|. So every element satisfies
        |o - o_ref| <= u (|o_ref| + a_ref)
    up to fp32 residue (2^-14 covers it), where a_ref = sum_j w_j |v_j| are
    the same softmax weights applied to |V|; the oracle returns a_ref when
    called with |V|. Each element must meet the larger of that bound and the
    stated 1e-2. The mean error must meet the larger of the stated 1e-3 and
    u mean|o_ref|. Rounding o to bf16 alone averages up to u/2 |o|; with one
    key that is about 1e-3 for N(0, 1) values. The P terms' errors have
    independent signs, so their mean stays within the other u/2. With many
    keys u mean|o_ref| is far below 1e-3, so the stated bar holds there. The
    LSE bar and the empty-row pattern are as stated."""
    o = f64(o_gpu)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    res = {}
    if err.size:
        scale = np.abs(o_ref) + a_ref
        bound = np.maximum(BF16_U * scale + 2.0 ** -14, O_MAX_ABS)
        res = {"o_max_abs": float(err.max()), "worst_of_bound": float((err / bound).max()),
               "o_mean_abs": float(err.mean()),
               "mean_of_bound": float(err.mean() / max(O_MEAN_ABS, BF16_U * float(np.abs(o_ref).mean())))}
        assert res["worst_of_bound"] <= 1.0, f"{what}: {res}"
        assert res["mean_of_bound"] <= 1.0, f"{what}: {res}"
    lse = lse_gpu.detach().cpu().double().numpy()
    empty = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == empty).all(), f"{what}: -inf pattern of the LSE differs"
    assert (o[empty] == 0).all(), f"{what}: rows with no key must be 0"
    lerr = np.abs(lse[~empty] - lse_ref[~empty])
    res["lse_max_abs"] = float(lerr.max()) if lerr.size else 0.0
    assert res["lse_max_abs"] <= LSE_MAX_ABS, f"{what}: {res}"
    return res


def compare_grad(g_gpu, g_ref, t_ref, s_ref=None, what=""):
    """Assert the gradient bar (module docstring) given the oracle's gradient
    g_ref, its term magnitudes t_ref and its Dl sensitivity s_ref (None for
    dV); returns the measured errors."""
    g = f64(g_gpu)
    assert g.shape == g_ref.shape == t_ref.shape, f"{what}: shape {g.shape} vs {g_ref.shape}"
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    if g.size == 0:
        return {}
    scale = t_ref if s_ref is None else t_ref + s_ref
    err = np.abs(g - g_ref)
    bound = GRAD_TERMS * scale + BF16_U * np.abs(g_ref) + GRAD_FLOOR
    res = {"max_abs": float(err.max()), "worst_of_bound": float((err / bound).max()),
           "mean_abs": float(err.mean()), "mean_of_bound": float(err.mean() / max(BF16_U * scale.mean(), GRAD_FLOOR))}
    assert res["worst_of_bound"] <= 1.0, f"{what}: {res}"
    assert res["mean_of_bound"] <= 1.0, f"{what}: {res}"
    return res
