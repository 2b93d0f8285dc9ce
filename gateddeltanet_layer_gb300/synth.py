"""Seeded synthetic inputs for the GatedDeltaNet layer.

This module holds none of the layer's arithmetic: it draws random numbers,
rounds them to the I/O dtype and lays them out.  It is the one module that both
the CUDA path's tests/benchmark and the oracle's tests read inputs from.

Draw order (fixed, numpy PCG64 seeded with ``seed``): sequence lengths (packed
varlen only), x_q, x_k, x_v, z, a, b, conv_w, dt_bias, A_log, norm_w, then
init_state (prefill) or conv cache and state (decode).  Values are drawn in
fp32; streams of a bf16 workload are rounded to bf16 (round to nearest even)
and kept as fp32 arrays holding bf16-representable values, so every consumer
reads exactly the same numbers.

Distributions (second argument of N is the standard deviation):
  x_q, x_k, x_v, z ~ N(0, 1);  a, b ~ N(0, 1);  conv_w ~ N(0, 0.25)
  dt_bias ~ U(-1, 1);  A_log = log U(lo, hi) with (lo, hi) = (1, 16) by default
  norm_w = 1 + N(0, 0.1);  init_state ~ N(0, init_std) or zeros
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns fp32."""
    x = np.array(x, dtype=np.float32, copy=True, order="C")
    u = x.view(np.uint32)
    # finite inputs: u + 0x8000 <= 0xFF807FFF, so 32-bit arithmetic cannot wrap
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    u &= np.uint32(0xFFFF0000)
    return x


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    lengths: tuple            # per-sequence token counts (packed in this order)
    h_qk: int = 16
    h_v: int = 32
    d_k: int = 128
    d_v: int = 128
    dtype: str = "bf16"       # "bf16" or "fp32" streams; parameters and state are fp32
    init_std: float = 0.0     # 0 = zero initial state (passed as NULL)
    a_log_range: tuple = (1.0, 16.0)
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def T(self) -> int:
        return int(sum(self.lengths))

    @property
    def N(self) -> int:
        return len(self.lengths)

    @property
    def channels(self) -> int:
        return 2 * self.h_qk * self.d_k + self.h_v * self.d_v


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    h_qk: int = 16
    h_v: int = 32
    d_k: int = 128
    d_v: int = 128
    dtype: str = "bf16"
    state_std: float = 0.02
    a_log_range: tuple = (1.0, 16.0)
    seed: int = 0

    @property
    def channels(self) -> int:
        return 2 * self.h_qk * self.d_k + self.h_v * self.d_v


def varlen_lengths(total: int, lo: int, hi: int, rng: np.random.Generator) -> tuple:
    """Integers uniform on [lo, hi], drawn until they sum to ``total``; the last
    one is cut to the remainder."""
    out, acc = [], 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return tuple(out)


def _varlen_32k(seed: int = 0) -> tuple:
    return varlen_lengths(32768, 256, 8192, np.random.default_rng(seed))


# The five workloads.
TINY = PrefillConfig("tiny_T64_fp32", (64,), h_qk=2, h_v=2, d_k=16, d_v=16, dtype="fp32")
SINGLE_4K = PrefillConfig("prefill_T4096", (4096,))
VARLEN_32K = PrefillConfig("prefill_varlen_T32768", _varlen_32k(), init_std=0.02)
DECODE_256 = DecodeConfig("decode_B256", 256)
LONG_128K = PrefillConfig("prefill_long_T131072", (8192,) * 16, a_log_range=(1.0, 4.0))

CONFIGS = {c.name: c for c in (TINY, SINGLE_4K, VARLEN_32K, DECODE_256, LONG_128K)}

# Few chains: one 16384-token sequence with the heads one GPU holds when the
# layer's 16/32 heads are split 8 ways by tensor parallelism (2 q/k, 4 value
# heads): the case the segment-parallel prefill is for.
FEW_CHAINS_16K = PrefillConfig("prefill_T16384_hv4", (16384,), h_qk=2, h_v=4)


def _stream(rng, shape, dtype):
    x = rng.standard_normal(shape, dtype=np.float32)
    return round_bf16(x) if dtype == "bf16" else x


def make_prefill(cfg: PrefillConfig, seed: int | None = None) -> dict:
    """Draw one prefill workload.  Returns a dict of numpy arrays:
    x_q, x_k [T, h_qk, d_k]; x_v, z [T, h_v, d_v]; a, b [T, h_v]; conv_w [Cc, 4];
    A_log, dt_bias [h_v]; norm_w [d_v]; init_state [N, h_v, d_k, d_v] or None;
    cu_seqlens int32 [N+1]."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    T, hq, hv, dk, dv, dt = cfg.T, cfg.h_qk, cfg.h_v, cfg.d_k, cfg.d_v, cfg.dtype
    inp = {}
    inp["x_q"] = _stream(rng, (T, hq, dk), dt)
    inp["x_k"] = _stream(rng, (T, hq, dk), dt)
    inp["x_v"] = _stream(rng, (T, hv, dv), dt)
    inp["z"] = _stream(rng, (T, hv, dv), dt)
    inp["a"] = _stream(rng, (T, hv), dt)
    inp["b"] = _stream(rng, (T, hv), dt)
    inp["conv_w"] = (0.25 * rng.standard_normal((cfg.channels, 4))).astype(np.float32)
    inp["dt_bias"] = rng.uniform(-1.0, 1.0, hv).astype(np.float32)
    lo, hi = cfg.a_log_range
    inp["A_log"] = np.log(rng.uniform(lo, hi, hv)).astype(np.float32)
    inp["norm_w"] = (1.0 + 0.1 * rng.standard_normal(dv)).astype(np.float32)
    if cfg.init_std > 0:
        inp["init_state"] = (cfg.init_std * rng.standard_normal((cfg.N, hv, dk, dv), dtype=np.float32))
    else:
        inp["init_state"] = None
    inp["cu_seqlens"] = np.concatenate([[0], np.cumsum(cfg.lengths)]).astype(np.int32)
    return inp


def make_decode(cfg: DecodeConfig, seed: int | None = None) -> dict:
    """Draw one decode-step workload: the prefill streams with T = batch (token
    b belongs to sequence b), plus conv_state [B, Cc, 3] (I/O dtype, oldest
    input first) and state [B, h_v, d_k, d_v] fp32."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    B, hq, hv, dk, dv, dt = cfg.batch, cfg.h_qk, cfg.h_v, cfg.d_k, cfg.d_v, cfg.dtype
    inp = {}
    inp["x_q"] = _stream(rng, (B, hq, dk), dt)
    inp["x_k"] = _stream(rng, (B, hq, dk), dt)
    inp["x_v"] = _stream(rng, (B, hv, dv), dt)
    inp["z"] = _stream(rng, (B, hv, dv), dt)
    inp["a"] = _stream(rng, (B, hv), dt)
    inp["b"] = _stream(rng, (B, hv), dt)
    inp["conv_w"] = (0.25 * rng.standard_normal((cfg.channels, 4))).astype(np.float32)
    inp["dt_bias"] = rng.uniform(-1.0, 1.0, hv).astype(np.float32)
    lo, hi = cfg.a_log_range
    inp["A_log"] = np.log(rng.uniform(lo, hi, hv)).astype(np.float32)
    inp["norm_w"] = (1.0 + 0.1 * rng.standard_normal(dv)).astype(np.float32)
    inp["conv_state"] = _stream(rng, (B, cfg.channels, 3), dt)
    inp["state"] = (cfg.state_std * rng.standard_normal((B, hv, dk, dv), dtype=np.float32))
    return inp


def scaled(cfg, **changes):
    """A copy of a workload with some fields changed (smaller parity cases)."""
    return replace(cfg, **changes)
