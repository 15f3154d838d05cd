"""Comparison helpers for the GPU parity tests (data handling only)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances of the method's floating-point outputs against the fp64 oracle:
# bf16 O within 1e-2 + 1e-2 |O_ref|, fp32 LSE within 1e-3 absolute.
O_ATOL = 1e-2
O_RTOL = 1e-2
LSE_ATOL = 1e-3


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def diagnostics(got, ref) -> dict:
    g, r = to64(got).ravel(), to64(ref).ravel()
    err = np.abs(g - r)
    denom = np.linalg.norm(g) * np.linalg.norm(r)
    return {
        "max_abs_err": float(err.max()) if err.size else 0.0,
        "max_rel_err": float((err / np.maximum(np.abs(r), 1e-30)).max()) if err.size else 0.0,
        "cosine": float(g @ r / denom) if denom > 0 else 1.0,
    }


def assert_o_close(got, ref, what=""):
    g, r = to64(got), to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    bad = ~(np.abs(g - r) <= O_ATOL + O_RTOL * np.abs(r))
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; {diagnostics(g, r)}"


def assert_lse_close(got, ref, what=""):
    g, r = to64(got), to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    both_neg_inf = np.isneginf(g) & np.isneginf(r)
    bad = ~((np.abs(g - r) <= LSE_ATOL) | both_neg_inf)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} LSE outside {LSE_ATOL}; max {np.nanmax(np.abs(g - r))}"
