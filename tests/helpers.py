"""Shared test helpers: moving synthetic inputs to the GPU and the parity metric."""
from __future__ import annotations

import numpy as np

# Tolerances.  bf16 streams with fp32 state: max |g - r| / max(1, |r|) <= 2e-2
# and ||g - r|| / ||r|| <= 1e-2 per tensor; fp32 streams: both <= 1e-4.  The
# max-abs bound is taken relative to max(1, |r|) because a bf16 output of
# magnitude >= 8 has a half-ulp of 0.031 > 2e-2: a plain absolute 2e-2 would
# fail even a correctly rounded output.
TOL = {"bf16": (2e-2, 1e-2), "fp32": (1e-4, 1e-4)}


def parity(got, ref, dtype: str, what: str = ""):
    """Assert the per-tensor tolerances; returns (max_rel, rel_l2, max_abs)."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    mask = ~np.isnan(r)
    g, r = g[mask], r[mask]
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - r)
    max_rel = float(np.max(err / np.maximum(1.0, np.abs(r)))) if err.size else 0.0
    denom = float(np.linalg.norm(r))
    rel_l2 = float(np.linalg.norm(g - r) / denom) if denom > 0 else float(np.linalg.norm(g - r))
    max_abs = float(err.max()) if err.size else 0.0
    tmax, tl2 = TOL[dtype]
    assert max_rel <= tmax and rel_l2 <= tl2, (
        f"{what}: max|d|/max(1,|r|) = {max_rel:.3e} (tol {tmax}), rel-L2 = {rel_l2:.3e} (tol {tl2}), "
        f"max|d| = {max_abs:.3e}")
    return max_rel, rel_l2, max_abs


def to_torch(inp: dict, bf16: bool, device="cuda"):
    """numpy workload -> torch tensors on `device` (streams bf16 or fp32)."""
    import torch
    sdt = torch.bfloat16 if bf16 else torch.float32
    out = {}
    for key in ("x_q", "x_k", "x_v", "z", "a", "b", "conv_state"):
        if key in inp and inp[key] is not None:
            out[key] = torch.from_numpy(np.ascontiguousarray(inp[key])).to(device=device, dtype=sdt)
    for key in ("conv_w", "A_log", "dt_bias", "norm_w", "init_state", "state"):
        if key in inp and inp[key] is not None:
            out[key] = torch.from_numpy(np.ascontiguousarray(inp[key])).to(device=device, dtype=torch.float32)
    if "cu_seqlens" in inp:
        out["cu_seqlens"] = torch.from_numpy(inp["cu_seqlens"]).to(device=device, dtype=torch.int32)
    return out

