"""Shared test helpers: moving synthetic inputs to the GPU and the parity metric."""
from __future__ import annotations

import numpy as np

# Tolerances.  bf16 streams with fp32 state: max |g - r| / max(1, |r|) <= 2e-2
# and ||g - r|| / ||r|| <= 1e-2 per tensor; fp32 streams: both <= 1e-4.  The
# max-abs bound is taken relative to max(1, |r|) because a bf16 output of
# magnitude >= 8 has a half-ulp of 0.031 > 2e-2: a plain absolute 2e-2 would
# fail even a correctly rounded output.  The plain max-abs error is reported
# beside it, both against the fp64 reference and against the reference rounded
# to bf16 (the grid the output lives on), with the bf16 ulp of |r| allowed.
TOL = {"bf16": (2e-2, 1e-2), "fp32": (1e-4, 1e-4)}


def _round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 (ties to even), as fp64 values."""
    f = np.asarray(x, dtype=np.float32).copy()
    u = f.view(np.uint32)
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    u &= np.uint32(0xFFFF0000)
    return f.astype(np.float64)


def _ulp_bf16(r: np.ndarray) -> np.ndarray:
    """Spacing of the bf16 grid at |r| (7 stored mantissa bits)."""
    a = np.maximum(np.abs(r), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7.0)


class Parity:
    """Accumulates the parity figures of one tensor over several slices (so a
    full-size output can be compared sequence by sequence without holding the
    whole fp64 reference), then asserts the tolerances once."""

    def __init__(self, dtype: str, what: str = "", normwise: bool = False):
        self.dtype, self.what, self.normwise = dtype, what, normwise
        self.max_rel = 0.0
        self.max_abs = 0.0
        self.max_abs_rounded = 0.0      # |g - bf16(r)|
        self.max_excess_ulp = 0.0       # |g - bf16(r)| - ulp(r), bf16 only
        self.sq_err = 0.0
        self.sq_ref = 0.0
        self.count = 0

    def add(self, got, ref):
        g = np.asarray(got, dtype=np.float64)
        r = np.asarray(ref, dtype=np.float64)
        assert g.shape == r.shape, (self.what, g.shape, r.shape)
        mask = ~np.isnan(r)
        g, r = g[mask], r[mask]
        if g.size == 0:
            return self
        assert np.all(np.isfinite(g)), f"{self.what}: non-finite values"
        err = np.abs(g - r)
        if self.normwise:  # relative to the tensor's largest magnitude (see parity_sum)
            self.max_rel = max(self.max_rel, float(err.max()) / max(1.0, float(np.abs(r).max())))
        else:
            self.max_rel = max(self.max_rel, float(np.max(err / np.maximum(1.0, np.abs(r)))))
        self.max_abs = max(self.max_abs, float(err.max()))
        if self.dtype == "bf16":
            er = np.abs(g - _round_bf16(r))
            self.max_abs_rounded = max(self.max_abs_rounded, float(er.max()))
            self.max_excess_ulp = max(self.max_excess_ulp, float(np.max(er - _ulp_bf16(r))))
        self.sq_err += float(np.sum((g - r) ** 2))
        self.sq_ref += float(np.sum(r ** 2))
        self.count += g.size
        return self

    @property
    def rel_l2(self) -> float:
        return float(np.sqrt(self.sq_err / self.sq_ref)) if self.sq_ref > 0 else float(np.sqrt(self.sq_err))

    def summary(self) -> str:
        s = (f"{self.what}: {self.count} values, max|d|/max(1,|r|) = {self.max_rel:.3e}, "
             f"rel-L2 = {self.rel_l2:.3e}, max|d| = {self.max_abs:.3e}")
        if self.dtype == "bf16":
            s += (f", max|g - bf16(r)| = {self.max_abs_rounded:.3e} "
                  f"(largest excess over one bf16 ulp of |r|: {self.max_excess_ulp:.3e})")
        return s

    def check(self):
        tmax, tl2 = TOL[self.dtype]
        assert self.max_rel <= tmax and self.rel_l2 <= tl2, f"{self.summary()} (tol {tmax}, {tl2})"
        return self.max_rel, self.rel_l2, self.max_abs


def parity(got, ref, dtype: str, what: str = ""):
    """Assert the per-tensor tolerances; returns (max_rel, rel_l2, max_abs)."""
    return Parity(dtype, what).add(got, ref).check()


def parity_sum(got, ref, dtype: str, what: str = ""):
    """The tolerances for a tensor each of whose elements is a sum over every
    token and head (the parameter gradients): the max-abs measure is taken
    relative to max(1, the tensor's largest |r|) instead of each element's own
    |r|.  An element summed from n terms in fp32 carries an error of order
    n * 2^-24 * sum |term|, which is of the tensor's scale, not of an element
    that the signs of its terms cancel down; the rel-L2 bound is unchanged."""
    return Parity(dtype, what, normwise=True).add(got, ref).check()


def to_torch(inp: dict, bf16: bool, device="cuda"):
    """numpy workload -> torch tensors on `device` (streams bf16 or fp32)."""
    import torch
    sdt = torch.bfloat16 if bf16 else torch.float32
    out = {}
    for key in ("x_q", "x_k", "x_v", "z", "a", "b", "conv_state", "init_conv"):
        if key in inp and inp[key] is not None:
            out[key] = torch.from_numpy(np.ascontiguousarray(inp[key])).to(device=device, dtype=sdt)
    for key in ("conv_w", "A_log", "dt_bias", "norm_w", "init_state", "state"):
        if key in inp and inp[key] is not None:
            out[key] = torch.from_numpy(np.ascontiguousarray(inp[key])).to(device=device, dtype=torch.float32)
    if "cu_seqlens" in inp:
        out["cu_seqlens"] = torch.from_numpy(inp["cu_seqlens"]).to(device=device, dtype=torch.int32)
    return out
