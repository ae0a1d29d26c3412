"""Comparison helpers shared by the parity tests (no method arithmetic here).

Tolerances (elementwise |gpu - oracle| <= atol + rtol * |oracle|):
  bf16 inputs with fp32 accumulation: atol 1e-2, rtol 2e-2;
  the all-fp32 mode: atol 1e-5, rtol 1e-5.
Argmax: where the oracle's top-2 margin exceeds the tolerance at the top
value, the GPU slot must equal the oracle's; elsewhere any slot whose oracle
score is within the tolerance of the maximum is accepted.
"""
from __future__ import annotations

import numpy as np
import torch

TOL = {"bf16": (1e-2, 2e-2), "f32": (1e-5, 1e-5)}


def tdtype(dtype: str):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def dev(t, dtype=None, device="cuda"):
    """Copy an fp32 host tensor holding storage-dtype values to the device."""
    if t is None:
        return None
    if dtype is None:
        return t.to(device).contiguous()
    return t.to(tdtype(dtype)).to(device).contiguous()


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype != torch.int32 else \
        t.detach().cpu().numpy()


def assert_close(gpu, ref, dtype, what=""):
    atol, rtol = TOL[dtype]
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    err = np.abs(g - r)
    lim = atol + rtol * np.abs(r)
    bad = err > lim
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance (atol={atol}, rtol={rtol}); "
            f"max err {err.max():.3e}; first {[(tuple(i), g[tuple(i)], r[tuple(i)]) for i in idx]}")
    return float(err.max()) if err.size else 0.0


def assert_argmax(gpu_slot, ref_edges, ref_slot, dtype, what=""):
    """Check the readout against the oracle's full edge matrix [..., K, K]."""
    atol, rtol = TOL[dtype]
    gs = np.asarray(gpu_slot).reshape(-1)
    E = np.asarray(ref_edges, dtype=np.float64).reshape(gs.size, -1)
    rs = np.asarray(ref_slot).reshape(-1)
    if gs.size == 0:
        return 0
    K = E.shape[1]
    top = E.max(axis=1)
    tol = atol + rtol * np.abs(top)
    if K > 1:
        second = np.partition(E, K - 2, axis=1)[:, K - 2]
    else:
        second = np.full_like(top, -np.inf)
    strict = (top - second) > tol
    bad_strict = strict & (gs != rs)
    assert not bad_strict.any(), \
        f"{what}: {int(bad_strict.sum())} argmax mismatches above the margin"
    picked = E[np.arange(gs.size), np.clip(gs, 0, K - 1)]
    in_range = (gs >= 0) & (gs < K)
    ok_loose = in_range & (np.abs(picked - top) <= tol)
    assert ok_loose.all(), f"{what}: {int((~ok_loose).sum())} slots not within tolerance of max"
    return int((~strict).sum())
