"""Shared helpers for the GPU-vs-oracle parity tests.

The bar (one set of numbers for every case): compared against the fp64
oracle on the same bf16 inputs, the bf16 output must have max-abs error
<= 1e-2 and mean-abs error <= 1e-3, and the fp32 LSE max-abs error <= 1e-3.
Rows the oracle marks as seeing no key must come back as o = 0, lse = -inf.
"""
import numpy as np
import torch

import oracle
from exact_scaled_dot_03_b300.workloads import bf16_bits

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


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
