"""fp64 CPU oracle of the GatedDeltaNet layer -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this module.  The CUDA product path never does, and the
two share no code: this file marshals numpy arrays into the plain C of
``gdn_oracle.c`` (compiled here with gcc), one (sequence, value-head) chain per
call, and composes the layer's stages in the order the layer defines them:

    conv1d(width 4) + SiLU on q, k, v  ->  L2-normalise q, k  ->  gates g, beta
    ->  gated delta rule  ->  RMSNormGated

(the layer named "GatedDeltaNet" / "RMSNormGated" on the page "[Qwen3.5 MoE]
Add hybrid decoder model (GatedDeltaNet + full attention + MoE)", Summary;
packed varlen sequences via cu_seqlens per "feat(models): dense Qwen3.5 custom
attention", Summary, and "Support Qwen35 SFT", XTuner changes).  The formulas
are written out in the header of ``gdn_oracle.c``.

Conventions (the readings the pages leave open; each is listed with its reason
in the design notes):
  * conv weights ``conv_w[c, j]``, ``j = 3`` multiplies the current token;
    channels ordered [q heads | k heads | v heads], each head-major then dim;
    no conv bias; zero history at each sequence start in prefill.
  * value head ``h`` reads query/key head ``h // (h_v // h_qk)``.
  * state ``[n, h, i, j]`` = S[j, i] (i over d_k, j over d_v).
  * eps_l2 = eps_rms = 1e-6; ``norm_w`` is a plain [d_v] weight shared by heads.

Threads: chains are independent, and ctypes releases the GIL during each C
call, so ``threads > 1`` runs chains in parallel on the host cores.
"""
from __future__ import annotations

import concurrent.futures as _cf
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

EPS_L2 = 1e-6
EPS_RMS = 1e-6

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into oracle/libgdn_oracle.so with gcc (plain C, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d = ctypes.c_int, ctypes.c_double
            lib.gdn_ref_conv_silu.argtypes = [i, i, _dp, _dp, _dp, _dp]
            lib.gdn_ref_l2norm.argtypes = [i, i, d, _dp]
            lib.gdn_ref_gates.argtypes = [i, _dp, _dp, d, d, _dp, _dp]
            lib.gdn_ref_recurrence.argtypes = [i, i, i, d, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.gdn_ref_recurrence_chunked.argtypes = [i, i, i, i, d, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.gdn_ref_rmsnorm_gated.argtypes = [i, i, d, _dp, _dp, _dp, _dp]
            lib.gdn_ref_rmsnorm_gated_backward.argtypes = [i, i, d, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.gdn_ref_recurrence_backward.argtypes = [i, i, i, d] + [_dp] * 14
            lib.gdn_ref_l2norm_backward.argtypes = [i, i, d, _dp, _dp, _dp]
            lib.gdn_ref_conv_silu_backward.argtypes = [i, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.gdn_ref_gates_backward.argtypes = [i, _dp, _dp, d, d, _dp, _dp, _dp, _dp, _dp, _dp]
            for f in ("gdn_ref_conv_silu", "gdn_ref_l2norm", "gdn_ref_gates", "gdn_ref_recurrence",
                      "gdn_ref_recurrence_chunked", "gdn_ref_rmsnorm_gated", "gdn_ref_rmsnorm_gated_backward",
                      "gdn_ref_recurrence_backward", "gdn_ref_l2norm_backward", "gdn_ref_conv_silu_backward",
                      "gdn_ref_gates_backward"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    return None if x is None else x.ctypes.data_as(_dp)


# ---------------------------------------------------------------- stages
def conv_silu(x, w, hist=None) -> np.ndarray:
    """x [L, C], w [C, 4], hist [3, C] (inputs at t=-3,-2,-1) or None -> silu(conv) [L, C]."""
    x, w = _f64(x), _f64(w)
    L, C = x.shape
    assert w.shape == (C, 4)
    h = None if hist is None else _f64(hist)
    if h is not None:
        assert h.shape == (3, C)
    y = np.empty((L, C), np.float64)
    _load().gdn_ref_conv_silu(L, C, _ptr(x), _ptr(w), _ptr(h), _ptr(y))
    return y


def l2norm(x, eps: float = EPS_L2) -> np.ndarray:
    """Row-wise x / sqrt(sum x^2 + eps) of x [L, D]."""
    y = _f64(x).copy()
    L, D = y.shape
    _load().gdn_ref_l2norm(L, D, eps, _ptr(y))
    return y


def gates(a, b, A_log: float, dt_bias: float):
    """a, b [L] of one value head -> (g [L], beta [L])."""
    a, b = _f64(a), _f64(b)
    L = a.shape[0]
    g, beta = np.empty(L), np.empty(L)
    _load().gdn_ref_gates(L, _ptr(a), _ptr(b), float(A_log), float(dt_bias), _ptr(g), _ptr(beta))
    return g, beta


def recurrence(q, k, v, g, beta, H0=None, scale=None, chunk: int | None = None):
    """Gated delta rule over one chain.  q, k [L, dk]; v [L, dv]; g, beta [L];
    H0 [dk, dv] or None.  Returns (o [L, dv] scaled, H_final [dk, dv]).
    ``chunk=None`` runs the token-by-token definition, an integer the chunked
    (WY/UT) reformulation with that chunk length."""
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    L, dk = k.shape
    dv = v.shape[1]
    if scale is None:
        scale = dk ** -0.5
    H0 = None if H0 is None else _f64(H0)
    o = np.empty((L, dv), np.float64)
    Hf = np.empty((dk, dv), np.float64)
    lib = _load()
    if chunk is None:
        lib.gdn_ref_recurrence(L, dk, dv, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                               _ptr(H0), _ptr(o), _ptr(Hf))
    else:
        lib.gdn_ref_recurrence_chunked(L, dk, dv, int(chunk), float(scale), _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(g), _ptr(beta), _ptr(H0), _ptr(o), _ptr(Hf))
    return o, Hf


def rmsnorm_gated(o, z, w, eps: float = EPS_RMS) -> np.ndarray:
    """RMSNormGated: o / sqrt(mean(o^2) + eps) * w * silu(z), rows of o, z [L, dv]; w [dv]."""
    o, z, w = _f64(o), _f64(z), _f64(w)
    L, dv = o.shape
    y = np.empty((L, dv), np.float64)
    _load().gdn_ref_rmsnorm_gated(L, dv, eps, _ptr(o), _ptr(z), _ptr(w), _ptr(y))
    return y


# ---------------------------------------------------------------- the layer, one chain
def _channels(h_qk, h_v, dk, dv, hq, hv):
    """conv_w rows of q head hq, k head hq and v head hv."""
    qc = np.arange(hq * dk, (hq + 1) * dk)
    kc = h_qk * dk + qc
    vc = 2 * h_qk * dk + np.arange(hv * dv, (hv + 1) * dv)
    return qc, kc, vc


def chain(inp: dict, s0: int, s1: int, hv: int, H0=None, hist=None, *, chunk=None,
          eps_l2=EPS_L2, eps_rms=EPS_RMS, scale=None):
    """The layer for tokens [s0, s1) of one packed sequence and value head hv.

    ``inp`` holds x_q, x_k [T, h_qk, dk]; x_v, z [T, h_v, dv]; a, b [T, h_v];
    conv_w [Cc, 4]; A_log, dt_bias [h_v]; norm_w [dv].  ``hist`` (optional)
    is a dict with "q", "k" [3, dk] and "v" [3, dv]: the raw inputs of the three
    tokens before s0 (decode); None means zeros (start of a prefill sequence).
    Returns dict(y [L, dv], o [L, dv], H [dk, dv], q, k, v, g, beta).
    """
    h_qk, dk = inp["x_q"].shape[1:]
    h_v, dv = inp["x_v"].shape[1:]
    hq = hv // (h_v // h_qk)
    qc, kc, vc = _channels(h_qk, h_v, dk, dv, hq, hv)
    w = _f64(inp["conv_w"])
    hq_, hk_, hv_ = (None, None, None) if hist is None else (hist["q"], hist["k"], hist["v"])
    q = l2norm(conv_silu(inp["x_q"][s0:s1, hq, :], w[qc], hq_), eps_l2)
    k = l2norm(conv_silu(inp["x_k"][s0:s1, hq, :], w[kc], hk_), eps_l2)
    v = conv_silu(inp["x_v"][s0:s1, hv, :], w[vc], hv_)
    g, beta = gates(inp["a"][s0:s1, hv], inp["b"][s0:s1, hv], float(inp["A_log"][hv]),
                    float(inp["dt_bias"][hv]))
    o, Hf = recurrence(q, k, v, g, beta, H0, scale=scale, chunk=chunk)
    y = rmsnorm_gated(o, inp["z"][s0:s1, hv, :], inp["norm_w"], eps_rms)
    return dict(y=y, o=o, H=Hf, q=q, k=k, v=v, g=g, beta=beta)


def _pool_map(fn, items, threads):
    if threads is None:
        threads = os.cpu_count() or 1
    if threads <= 1 or len(items) <= 1:
        return [fn(it) for it in items]
    with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))


def _hist_of(conv, h_qk, h_v, dk, dv, hv):
    """The conv history of value head hv from a [Cc, 3] conv cache (raw inputs
    of the three tokens before, oldest first): dict of q, k [3, dk] and v [3, dv]."""
    hq = hv // (h_v // h_qk)
    qc, kc, vc = _channels(h_qk, h_v, dk, dv, hq, hv)
    c = _f64(conv)
    return {"q": c[qc].T, "k": c[kc].T, "v": c[vc].T}


def prefill(inp: dict, cu_seqlens, init_state=None, chains=None, threads=None, init_conv=None, **kw):
    """Prefill over packed sequences.

    cu_seqlens [N+1] (int); init_state [N, h_v, dk, dv] or None; init_conv
    [N, Cc, 3] (the raw inputs of the three tokens before each sequence, oldest
    first, channels as conv_w) or None (= zeros: a sequence start).
    chains: list of (n, hv) to compute (None = all).  Returns dict with
    y [T, h_v, dv] and o [T, h_v, dv] (NaN outside the computed chains) and
    final_state [N, h_v, dk, dv] (NaN for chains not computed).
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    T, h_v, dv = inp["x_v"].shape
    dk = inp["x_k"].shape[2]
    if chains is None:
        chains = [(n, h) for n in range(N) for h in range(h_v)]
    y = np.full((T, h_v, dv), np.nan)
    o = np.full((T, h_v, dv), np.nan)
    fs = np.full((N, h_v, dk, dv), np.nan)

    h_qk = inp["x_q"].shape[1]

    def run(nh):
        n, h = nh
        H0 = None if init_state is None else init_state[n, h]
        hist = None if init_conv is None else _hist_of(init_conv[n], h_qk, h_v, dk, dv, h)
        return nh, chain(inp, int(cu[n]), int(cu[n + 1]), h, H0, hist, **kw)

    for (n, h), r in _pool_map(run, list(chains), threads):
        y[cu[n]:cu[n + 1], h] = r["y"]
        o[cu[n]:cu[n + 1], h] = r["o"]
        fs[n, h] = r["H"]
    return dict(y=y, o=o, final_state=fs)


def decode_step(inp: dict, conv_state, state, threads=None, **kw):
    """One token per sequence.  inp as in ``chain`` with T = B (token b belongs
    to sequence b); conv_state [B, Cc, 3] (oldest first); state [B, h_v, dk, dv].
    Returns dict(y [B, h_v, dv], state [B, h_v, dk, dv], conv_state [B, Cc, 3])
    with the state and conv cache as they are after the step."""
    B, h_v, dv = inp["x_v"].shape
    h_qk, dk = inp["x_q"].shape[1:]
    cs = _f64(conv_state)
    y = np.empty((B, h_v, dv))
    new_state = np.empty((B, h_v, dk, dv))

    def run(bh):
        b, h = bh
        hq = h // (h_v // h_qk)
        qc, kc, vc = _channels(h_qk, h_v, dk, dv, hq, h)
        hist = {"q": cs[b][qc].T, "k": cs[b][kc].T, "v": cs[b][vc].T}
        return bh, chain(inp, b, b + 1, h, state[b, h], hist, **kw)

    for (b, h), r in _pool_map(run, [(b, h) for b in range(B) for h in range(h_v)], threads):
        y[b, h] = r["y"][0]
        new_state[b, h] = r["H"]
    # the cache keeps the last three raw inputs, oldest first
    x_all = np.concatenate([np.asarray(inp["x_q"], np.float64).reshape(B, -1),
                            np.asarray(inp["x_k"], np.float64).reshape(B, -1),
                            np.asarray(inp["x_v"], np.float64).reshape(B, -1)], axis=1)
    new_cs = np.concatenate([cs[:, :, 1:], x_all[:, :, None]], axis=2)
    return dict(y=y, state=new_state, conv_state=new_cs)


def conv_cache_after_prefill(inp: dict, cu_seqlens, init_conv=None):
    """The decode conv cache [N, Cc, 3] a prefill leaves: per sequence and conv
    channel ([q | k | v], as conv_w) the raw inputs of its last three tokens,
    oldest first; before the sequence start the carried history ``init_conv``
    ([N, Cc, 3], token s0 - 3 + m at m) or zero (the zero conv history of a
    prefill, reading of the depthwise-conv bullet of "[Qwen3.5 MoE] Add hybrid
    decoder model ...", Summary).  Plain slicing, written from that definition."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T = inp["x_q"].shape[0]
    x_all = np.concatenate([np.asarray(inp["x_q"], np.float64).reshape(T, -1),
                            np.asarray(inp["x_k"], np.float64).reshape(T, -1),
                            np.asarray(inp["x_v"], np.float64).reshape(T, -1)], axis=1)
    N, Cc = len(cu) - 1, x_all.shape[1]
    cache = np.zeros((N, Cc, 3))
    for n in range(N):
        for j in range(3):
            t = cu[n + 1] - 3 + j
            if t >= cu[n]:
                cache[n, :, j] = x_all[t]
            elif init_conv is not None:
                cache[n, :, j] = np.asarray(init_conv[n], np.float64)[:, t - cu[n] + 3]
    return cache


# ---------------------------------------------------------------- backward (reverse mode)
# The gradient of a scalar loss  sum(dy * y) + sum(dfinal * final_state)  with
# respect to every input of the layer, by the stages' reverse-mode functions
# of gdn_oracle.c applied in the reverse of the forward order.  Training
# frameworks run this layer ("[Qwen3.5 MoE] Add hybrid decoder model ...",
# "Support Qwen35 SFT", "feat(models): dense Qwen3.5 custom attention": all
# train it); the pages state no backward, so this is the chain rule of the
# forward definitions, pinned to finite differences of the forward oracle.
def chain_backward(inp: dict, s0: int, s1: int, hv: int, dy, H0=None, hist=None, dHf=None, *,
                   eps_l2=EPS_L2, eps_rms=EPS_RMS, scale=None):
    """Gradients for tokens [s0, s1) of one sequence and value head hv.
    dy [L, dv] (gradient of y), dHf [dk, dv] or None (gradient of the final state).
    Returns dict: x_q, x_k [L, dk] and x_v, z [L, dv] (raw stream gradients of
    this chain's heads), a, b [L], conv_w_q, conv_w_k [dk, 4], conv_w_v [dv, 4],
    A_log, dt_bias (scalars), norm_w [dv], H0 [dk, dv], hist (dict q, k [3, dk],
    v [3, dv]: gradient of the carried conv history)."""
    lib = _load()
    h_qk, dk = inp["x_q"].shape[1:]
    h_v, dv = inp["x_v"].shape[1:]
    hq = hv // (h_v // h_qk)
    qc, kc, vc = _channels(h_qk, h_v, dk, dv, hq, hv)
    w = _f64(inp["conv_w"])
    L = s1 - s0
    if scale is None:
        scale = dk ** -0.5
    hq_, hk_, hv_ = (None, None, None) if hist is None else (_f64(hist["q"]), _f64(hist["k"]), _f64(hist["v"]))
    xq, xk, xv = _f64(inp["x_q"][s0:s1, hq, :]), _f64(inp["x_k"][s0:s1, hq, :]), _f64(inp["x_v"][s0:s1, hv, :])
    zz, aa, bb = _f64(inp["z"][s0:s1, hv, :]), _f64(inp["a"][s0:s1, hv]), _f64(inp["b"][s0:s1, hv])
    A_log, dt_bias = float(inp["A_log"][hv]), float(inp["dt_bias"][hv])
    nw = _f64(inp["norm_w"])
    # forward, keeping what the reverse steps read
    qr, kr, v = conv_silu(xq, w[qc], hq_), conv_silu(xk, w[kc], hk_), conv_silu(xv, w[vc], hv_)
    q, k = l2norm(qr, eps_l2), l2norm(kr, eps_l2)
    g, beta = gates(aa, bb, A_log, dt_bias)
    H0 = None if H0 is None else _f64(H0)
    o, _ = recurrence(q, k, v, g, beta, H0, scale=scale)
    # reverse
    dyy = _f64(dy)
    d_o, dz, dnw = np.empty((L, dv)), np.empty((L, dv)), np.zeros(dv)
    lib.gdn_ref_rmsnorm_gated_backward(L, dv, eps_rms, _ptr(o), _ptr(zz), _ptr(nw), _ptr(dyy), _ptr(d_o), _ptr(dz),
                                       _ptr(dnw))
    dq, dkk, dvv = np.empty((L, dk)), np.empty((L, dk)), np.empty((L, dv))
    dg, dbeta, dH0 = np.empty(L), np.empty(L), np.empty((dk, dv))
    dHf_ = None if dHf is None else _f64(dHf)
    lib.gdn_ref_recurrence_backward(L, dk, dv, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    _ptr(H0), _ptr(d_o), _ptr(dHf_), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dg),
                                    _ptr(dbeta), _ptr(dH0))
    dqr, dkr = np.empty((L, dk)), np.empty((L, dk))
    lib.gdn_ref_l2norm_backward(L, dk, eps_l2, _ptr(qr), _ptr(dq), _ptr(dqr))
    lib.gdn_ref_l2norm_backward(L, dk, eps_l2, _ptr(kr), _ptr(dkk), _ptr(dkr))
    res = {}
    for name, x, wc, hh, dyx in (("q", xq, w[qc], hq_, dqr), ("k", xk, w[kc], hk_, dkr), ("v", xv, w[vc], hv_, dvv)):
        C = x.shape[1]
        dx, dw, dh = np.zeros((L, C)), np.zeros((C, 4)), np.zeros((3, C))
        wc = _f64(wc)
        lib.gdn_ref_conv_silu_backward(L, C, _ptr(x), _ptr(wc), _ptr(hh), _ptr(_f64(dyx)), _ptr(dx), _ptr(dh),
                                       _ptr(dw))
        res["x_" + name], res["conv_w_" + name], res["hist_" + name] = dx, dw, dh
    da, db = np.empty(L), np.empty(L)
    dA, ddt = ctypes.c_double(0.0), ctypes.c_double(0.0)
    lib.gdn_ref_gates_backward(L, _ptr(aa), _ptr(bb), A_log, dt_bias, _ptr(dg), _ptr(dbeta), _ptr(da), _ptr(db),
                               ctypes.byref(dA), ctypes.byref(ddt))
    res.update(z=dz, a=da, b=db, A_log=dA.value, dt_bias=ddt.value, norm_w=dnw, H0=dH0,
               hist={"q": res.pop("hist_q"), "k": res.pop("hist_k"), "v": res.pop("hist_v")})
    return res


def prefill_backward(inp: dict, cu_seqlens, dy, init_state=None, dfinal_state=None, threads=None, init_conv=None,
                     **kw):
    """Gradients of  sum(dy * y) + sum(dfinal_state * final_state)  of a prefill
    with respect to every input: dict with x_q, x_k [T, h_qk, dk]; x_v, z
    [T, h_v, dv]; a, b [T, h_v]; conv_w [Cc, 4]; A_log, dt_bias [h_v];
    norm_w [dv]; init_state [N, h_v, dk, dv]; init_conv [N, Cc, 3]."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    T, h_v, dv = inp["x_v"].shape
    h_qk, dk = inp["x_q"].shape[1:]
    Cc = 2 * h_qk * dk + h_v * dv
    dy = _f64(dy)
    gr = {"x_q": np.zeros((T, h_qk, dk)), "x_k": np.zeros((T, h_qk, dk)), "x_v": np.zeros((T, h_v, dv)),
          "z": np.zeros((T, h_v, dv)), "a": np.zeros((T, h_v)), "b": np.zeros((T, h_v)),
          "conv_w": np.zeros((Cc, 4)), "A_log": np.zeros(h_v), "dt_bias": np.zeros(h_v), "norm_w": np.zeros(dv),
          "init_state": np.zeros((N, h_v, dk, dv)), "init_conv": np.zeros((N, Cc, 3))}

    def run(nh):
        n, h = nh
        H0 = None if init_state is None else init_state[n, h]
        hist = None if init_conv is None else _hist_of(init_conv[n], h_qk, h_v, dk, dv, h)
        dHf = None if dfinal_state is None else dfinal_state[n, h]
        return nh, chain_backward(inp, int(cu[n]), int(cu[n + 1]), h, dy[cu[n]:cu[n + 1], h], H0, hist, dHf, **kw)

    for (n, h), r in _pool_map(run, [(n, h) for n in range(N) for h in range(h_v)], threads):
        s0, s1 = cu[n], cu[n + 1]
        hq = h // (h_v // h_qk)
        qc, kc, vc = _channels(h_qk, h_v, dk, dv, hq, h)
        gr["x_q"][s0:s1, hq] += r["x_q"]
        gr["x_k"][s0:s1, hq] += r["x_k"]
        gr["x_v"][s0:s1, h] += r["x_v"]
        gr["z"][s0:s1, h] = r["z"]
        gr["a"][s0:s1, h] = r["a"]
        gr["b"][s0:s1, h] = r["b"]
        gr["conv_w"][qc] += r["conv_w_q"]
        gr["conv_w"][kc] += r["conv_w_k"]
        gr["conv_w"][vc] += r["conv_w_v"]
        gr["A_log"][h] += r["A_log"]
        gr["dt_bias"][h] += r["dt_bias"]
        gr["norm_w"] += r["norm_w"]
        gr["init_state"][n, h] = r["H0"]
        gr["init_conv"][n][qc] += r["hist"]["q"].T
        gr["init_conv"][n][kc] += r["hist"]["k"].T
        gr["init_conv"][n][vc] += r["hist"]["v"].T
    return gr
