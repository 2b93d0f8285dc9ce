"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test checks a stage or the whole layer against a closed form, a library
routine, an invariant of the gated delta rule, a hand-worked example under
tests/golden/, or a brute-force restatement in a different algebraic form.
Together they are chosen so that a plausible slip in the oracle (reversed conv
taps, a missing SiLU, a wrong eps, a sign or placement error in the gates, a
transposed state, alpha or beta applied at the wrong place, the output read
before the state update, a wrong GQA head, a mis-ordered conv cache) fails at
least one of them.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import expit

from gateddeltanet_layer_gb300 import synth
from oracle import oracle as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


# ------------------------------------------------------------------ conv + SiLU
def test_conv_matches_numpy_convolve():
    """Causal width-4 depthwise conv = np.convolve with the taps reversed (w[c,3]
    multiplies the current token), followed by SiLU; history = the 3 inputs before t=0."""
    rng = _rng(1)
    L, C = 11, 5
    x = rng.standard_normal((L, C))
    w = rng.standard_normal((C, 4))
    hist = rng.standard_normal((3, C))
    for h in (None, hist):
        y = ref.conv_silu(x, w, h)
        for c in range(C):
            xx = x[:, c] if h is None else np.concatenate([h[:, c], x[:, c]])
            pre = np.convolve(xx, w[c, ::-1])[: len(xx)][-L:]
            np.testing.assert_allclose(y[:, c], pre * expit(pre), rtol=1e-13, atol=1e-14)


def test_conv_impulse_response():
    """A unit impulse at t0 gives pre-activations w[c, 3-(t-t0)] for t0 <= t <= t0+3, 0 elsewhere."""
    L, C, t0 = 10, 3, 2
    w = _rng(2).standard_normal((C, 4))
    x = np.zeros((L, C))
    x[t0] = 1.0
    y = ref.conv_silu(x, w)
    for c in range(C):
        for t in range(L):
            pre = w[c, 3 - (t - t0)] if 0 <= t - t0 <= 3 else 0.0
            assert abs(y[t, c] - pre * expit(pre)) < 1e-15


# ------------------------------------------------------------------ L2 norm
def test_l2norm_unit_and_eps():
    rng = _rng(3)
    x = rng.standard_normal((6, 16))
    y = ref.l2norm(x, eps=0.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(y * np.linalg.norm(x, axis=1, keepdims=True), x, rtol=1e-13)
    # with eps = 1e-6 and a row of squared norm s = 1e-6, ||y||^2 = s / (s + eps) = 1/2
    small = np.full((1, 4), 0.5e-3)  # s = 4 * 0.25e-6 = 1e-6
    y = ref.l2norm(small)
    assert abs(np.sum(y ** 2) - 0.5) < 1e-12


# ------------------------------------------------------------------ gates
@pytest.mark.parametrize("A_log,a,dt,b,g_exp,beta_exp", [
    (0.0, 0.0, 0.0, 0.0, -np.log(2.0), 0.5),                    # softplus(0) = ln 2
    (np.log(2.0), 1.0, -1.0, np.log(3.0), -2 * np.log(2.0), 0.75),  # dt_bias is added to a
    (np.log(3.0), 60.0, 0.0, -np.log(3.0), -180.0, 0.25),       # softplus(x) = x + O(e^-x)
    (0.0, 0.0, np.log(np.e - 1.0), 0.0, -1.0, 0.5),  # softplus(ln(e-1)) = 1
])
def test_gates_closed_forms(A_log, a, dt, b, g_exp, beta_exp):
    g, beta = ref.gates(np.array([a]), np.array([b]), A_log, dt)
    assert abs(g[0] - g_exp) < 1e-12 * max(1.0, abs(g_exp))
    assert abs(beta[0] - beta_exp) < 1e-15


# ------------------------------------------------------------------ recurrence
def _brute_force(q, k, v, g, beta, S0, scale):
    """The rule exactly as written with explicit matrices, S (dv x dk):
    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = S_t q_t scale."""
    L, dk = k.shape
    S = S0.copy()
    o = []
    for t in range(L):
        P = np.eye(dk) - beta[t] * np.outer(k[t], k[t])
        S = np.exp(g[t]) * S @ P + beta[t] * np.outer(v[t], k[t])
        o.append(S @ q[t] * scale)
    return np.array(o), S


def test_golden_worked_example():
    """Hand-worked two-token example (tests/golden/delta_rule_2x2.json)."""
    with open(os.path.join(GOLDEN, "delta_rule_2x2.json")) as f:
        gd = json.load(f)
    g = np.log(np.array(gd["alpha"]))
    o, H = ref.recurrence(np.array(gd["q"]), np.array(gd["k"]), np.array(gd["v"]), g,
                          np.array(gd["beta"]), None)
    np.testing.assert_allclose(o * np.sqrt(2.0), gd["o_times_sqrt2"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(H, gd["H_final"], rtol=0, atol=1e-14)


def test_recurrence_vs_explicit_transition_matrices():
    """Token form (H = S^T, rank-1 updates) vs the rule's matrix-product form."""
    rng = _rng(4)
    L, dk, dv = 9, 5, 3
    q = _unit_rows(rng.standard_normal((L, dk)))
    k = _unit_rows(rng.standard_normal((L, dk)))
    v = rng.standard_normal((L, dv))
    g = -rng.uniform(0.0, 1.5, L)
    beta = rng.uniform(0.05, 0.95, L)
    S0 = rng.standard_normal((dv, dk))
    o, H = ref.recurrence(q, k, v, g, beta, S0.T, scale=0.37)
    o_bf, S_bf = _brute_force(q, k, v, g, beta, S0, 0.37)
    np.testing.assert_allclose(o, o_bf, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(H, S_bf.T, rtol=1e-12, atol=1e-13)


def test_zero_beta_zero_gate_keeps_state():
    """beta = 0, g = 0: the state never changes and o_t = S0 q_t scale."""
    rng = _rng(5)
    L, dk, dv = 7, 6, 4
    q = _unit_rows(rng.standard_normal((L, dk)))
    k = _unit_rows(rng.standard_normal((L, dk)))
    v = rng.standard_normal((L, dv))
    H0 = rng.standard_normal((dk, dv))
    o, H = ref.recurrence(q, k, v, np.zeros(L), np.zeros(L), H0)
    np.testing.assert_array_equal(H, H0)
    np.testing.assert_allclose(o, q @ H0 * dk ** -0.5, rtol=1e-13)


def test_pure_decay():
    """beta = 0: H_t = exp(g_1 + ... + g_t) H0 and o_t = exp(G_t) H0^T q_t scale."""
    rng = _rng(6)
    L, dk, dv = 8, 4, 3
    q = _unit_rows(rng.standard_normal((L, dk)))
    k = _unit_rows(rng.standard_normal((L, dk)))
    g = -rng.uniform(0, 0.7, L)
    H0 = rng.standard_normal((dk, dv))
    o, H = ref.recurrence(q, k, rng.standard_normal((L, dv)), g, np.zeros(L), H0)
    G = np.cumsum(g)
    np.testing.assert_allclose(H, np.exp(G[-1]) * H0, rtol=1e-13)
    np.testing.assert_allclose(o, np.exp(G)[:, None] * (q @ H0) * dk ** -0.5, rtol=1e-12)


def test_single_token_from_zero_state():
    """One token from S0 = 0: o = beta (k . q) v scale (the output reads the updated state)."""
    rng = _rng(7)
    dk, dv = 8, 5
    q = _unit_rows(rng.standard_normal((1, dk)))
    k = _unit_rows(rng.standard_normal((1, dk)))
    v = rng.standard_normal((1, dv))
    o, H = ref.recurrence(q, k, v, np.array([-0.3]), np.array([0.7]), None)
    np.testing.assert_allclose(o[0], 0.7 * (k[0] @ q[0]) * v[0] * dk ** -0.5, rtol=1e-13)
    np.testing.assert_allclose(H, 0.7 * np.outer(k[0], v[0]), rtol=1e-13)


def test_zero_alpha_forgets_everything():
    """alpha = 0 (g -> -inf): each token behaves as the first token of a fresh state."""
    rng = _rng(8)
    L, dk, dv = 6, 5, 4
    q = _unit_rows(rng.standard_normal((L, dk)))
    k = _unit_rows(rng.standard_normal((L, dk)))
    v = rng.standard_normal((L, dv))
    beta = rng.uniform(0.1, 0.9, L)
    o, H = ref.recurrence(q, k, v, np.full(L, -1e4), beta, rng.standard_normal((dk, dv)))
    exp_o = (beta * np.sum(k * q, axis=1))[:, None] * v * dk ** -0.5
    np.testing.assert_allclose(o, exp_o, rtol=1e-13)
    np.testing.assert_allclose(H, beta[-1] * np.outer(k[-1], v[-1]), rtol=1e-13)


def test_orthonormal_keys_exact_recall():
    """alpha = 1, beta = 1, orthonormal keys from zero: the state recalls every pair,
    S_L k_s = v_s, and a fresh write overwrites exactly (S k_t = v_t after each step)."""
    rng = _rng(9)
    dk, dv, L = 6, 4, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:, :L].T
    v = rng.standard_normal((L, dv))
    _, H = ref.recurrence(k, k, v, np.zeros(L), np.ones(L), None)
    np.testing.assert_allclose(k @ H, v, atol=1e-13)
    # overwrite with a non-orthogonal key: S k = v for the newest pair
    k2 = np.vstack([k, _unit_rows(rng.standard_normal((1, dk)))])
    v2 = np.vstack([v, rng.standard_normal((1, dv))])
    _, H2 = ref.recurrence(k2, k2, v2, np.zeros(L + 1), np.ones(L + 1), None)
    np.testing.assert_allclose(k2[-1] @ H2, v2[-1], atol=1e-13)


def test_superposition_in_state_and_values():
    """With q, k, g, beta fixed, (o, H_final) is linear in (S0, v)."""
    rng = _rng(10)
    L, dk, dv = 12, 6, 5
    q = _unit_rows(rng.standard_normal((L, dk)))
    k = _unit_rows(rng.standard_normal((L, dk)))
    g = -rng.uniform(0, 1, L)
    beta = rng.uniform(0, 1, L)
    v = rng.standard_normal((L, dv))
    H0 = rng.standard_normal((dk, dv))
    o_a, H_a = ref.recurrence(q, k, v, g, beta, H0)
    o_s, H_s = ref.recurrence(q, k, np.zeros_like(v), g, beta, H0)
    o_v, H_v = ref.recurrence(q, k, v, g, beta, None)
    np.testing.assert_allclose(o_a, o_s + o_v, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(H_a, H_s + H_v, rtol=1e-12, atol=1e-14)


def test_segments_joined_by_their_affine_state_maps():
    """The reading behind the segment-parallel prefill: over a stretch of
    tokens the state map is affine, H_out = M H_in + B, with B the run from a
    zero state and M the run of the same tokens on the identity with v = 0 (the
    linear part alone).  Joining segments by H_in(s + 1) = M_s H_in(s) + B_s and
    rerunning each segment from its H_in gives the single run's outputs and
    final state (segments of 10 tokens and a ragged 7-token one)."""
    rng = _rng(12)
    L, dk, dv = 37, 6, 5
    q = _unit_rows(rng.standard_normal((L, dk)))
    k = _unit_rows(rng.standard_normal((L, dk)))
    g = -rng.uniform(0, 1, L)
    beta = rng.uniform(0, 1, L)
    v = rng.standard_normal((L, dv))
    H0 = rng.standard_normal((dk, dv))
    o_full, H_full = ref.recurrence(q, k, v, g, beta, H0)
    cuts = [0, 10, 20, 30, L]
    H_in, outs = H0, []
    for s0, s1 in zip(cuts[:-1], cuts[1:]):
        sl = slice(s0, s1)
        _, B = ref.recurrence(q[sl], k[sl], v[sl], g[sl], beta[sl], None)
        _, M = ref.recurrence(q[sl], k[sl], np.zeros((s1 - s0, dk)), g[sl], beta[sl], np.eye(dk))
        o_seg, H_seg = ref.recurrence(q[sl], k[sl], v[sl], g[sl], beta[sl], H_in)
        np.testing.assert_allclose(H_seg, M @ H_in + B, rtol=1e-12, atol=1e-13)
        outs.append(o_seg)
        H_in = M @ H_in + B
    np.testing.assert_allclose(np.vstack(outs), o_full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(H_in, H_full, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("chunk", [1, 7, 16, 64])
@pytest.mark.parametrize("memory", ["config", "long"])
def test_chunked_equals_token_form(chunk, memory):
    """The chunked WY/UT reformulation equals the token-by-token rule (ragged last chunk)."""
    rng = _rng(11)
    L, dk, dv = 150, 16, 12
    q = _unit_rows(rng.standard_normal((L, dk)))
    k = _unit_rows(rng.standard_normal((L, dk)))
    v = rng.standard_normal((L, dv))
    if memory == "config":   # the workloads' gates: A_log = log U(1,16), dt_bias ~ U(-1,1)
        g = -rng.uniform(1, 16) * np.log1p(np.exp(rng.standard_normal(L) + rng.uniform(-1, 1)))
    else:                    # long memory: dt_bias = -6
        g = -1.0 * np.log1p(np.exp(rng.standard_normal(L) - 6.0))
    beta = expit(rng.standard_normal(L))
    H0 = 0.02 * rng.standard_normal((dk, dv))
    o1, H1 = ref.recurrence(q, k, v, g, beta, H0)
    o2, H2 = ref.recurrence(q, k, v, g, beta, H0, chunk=chunk)
    np.testing.assert_allclose(o2, o1, rtol=1e-11, atol=1e-13 * np.abs(o1).max())
    np.testing.assert_allclose(H2, H1, rtol=1e-11, atol=1e-13 * np.abs(H1).max())


# ------------------------------------------------------------------ RMSNormGated
def test_rmsnorm_gated_unit_rms():
    """eps = 0: y / (w silu(z)) has RMS exactly 1 per row and is parallel to o."""
    rng = _rng(12)
    o = rng.standard_normal((4, 10)) * 1e-3
    z = rng.standard_normal((4, 10))
    w = 1 + 0.1 * rng.standard_normal(10)
    y = ref.rmsnorm_gated(o, z, w, eps=0.0)
    r = y / (w * z * expit(z))
    np.testing.assert_allclose(np.sqrt(np.mean(r ** 2, axis=1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(r * np.sqrt(np.mean(o ** 2, axis=1, keepdims=True)), o, rtol=1e-12)


def test_rmsnorm_eps_effect():
    """A row with mean(o^2) = eps is scaled by 1/sqrt(2 eps)."""
    o = np.full((1, 8), 1e-3)  # mean(o^2) = 1e-6 = eps
    z = np.full((1, 8), 30.0)  # silu(30) = 30 (1 - 9.4e-14)
    y = ref.rmsnorm_gated(o, z, np.ones(8), eps=1e-6)
    np.testing.assert_allclose(y, 1e-3 / np.sqrt(2e-6) * 30.0 * expit(30.0), rtol=1e-14)


# ------------------------------------------------------------------ the whole layer
def _tiny_inputs(T_lengths=(64,), h_qk=2, h_v=2, d=16, seed=0, init_std=0.0):
    cfg = synth.scaled(synth.TINY, lengths=tuple(T_lengths), h_qk=h_qk, h_v=h_v, d_k=d, d_v=d,
                       seed=seed, init_std=init_std)
    return synth.make_prefill(cfg)


def test_layer_first_token_closed_form():
    """T = 1 from a zero state, computed independently: pre = w[:,3] x (no history),
    k = silu(pre_k)/|.|, ..., o = beta (k.q) v scale, y = RMSNormGated(o)."""
    inp = _tiny_inputs((1,), h_qk=1, h_v=1, d=16, seed=3)
    r = ref.prefill(inp, inp["cu_seqlens"])
    d = 16
    w = inp["conv_w"].astype(np.float64)

    def silu(x):
        return x * expit(x)

    q = silu(w[:d, 3] * inp["x_q"][0, 0])
    k = silu(w[d:2 * d, 3] * inp["x_k"][0, 0])
    v = silu(w[2 * d:, 3] * inp["x_v"][0, 0])
    q, k = q / np.sqrt(q @ q + 1e-6), k / np.sqrt(k @ k + 1e-6)
    beta = expit(float(inp["b"][0, 0]))
    c = beta * (k @ q) * d ** -0.5
    o = c * v
    z = inp["z"][0, 0].astype(np.float64)
    y = o / np.sqrt(np.mean(o ** 2) + 1e-6) * inp["norm_w"] * silu(z)
    np.testing.assert_allclose(r["o"][0, 0], o, rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(r["y"][0, 0], y, rtol=1e-11, atol=1e-14)


def test_varlen_split_equals_independent_runs():
    """Packing sequences with cu_seqlens = running each one alone (bitwise)."""
    inp = _tiny_inputs((37, 64, 5), seed=1, init_std=0.02)
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"])
    cu = inp["cu_seqlens"]
    for n in range(3):
        sub = {k_: (v_[cu[n]:cu[n + 1]] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_)
               for k_, v_ in inp.items()}
        rs = ref.prefill(sub, [0, cu[n + 1] - cu[n]], inp["init_state"][n:n + 1])
        np.testing.assert_array_equal(r["y"][cu[n]:cu[n + 1]], rs["y"])
        np.testing.assert_array_equal(r["final_state"][n], rs["final_state"][0])


def test_no_conv_leak_across_sequence_boundary():
    """Changing the last tokens of sequence 0 leaves sequence 1 untouched."""
    inp = _tiny_inputs((20, 20), seed=2)
    r0 = ref.prefill(inp, inp["cu_seqlens"])
    for key in ("x_q", "x_k", "x_v"):
        inp[key] = inp[key].copy()
        inp[key][17:20] += 5.0
    r1 = ref.prefill(inp, inp["cu_seqlens"])
    np.testing.assert_array_equal(r0["y"][20:], r1["y"][20:])
    assert not np.array_equal(r0["y"][:20], r1["y"][:20])


def test_gqa_head_mapping():
    """Value head h reads query/key head h // (h_v / h_qk): with h_qk = 2, h_v = 4, value
    heads 0, 1 depend on qk head 0 only and heads 2, 3 on qk head 1 only."""
    inp = _tiny_inputs((16,), h_qk=2, h_v=4, seed=4)
    r0 = ref.prefill(inp, inp["cu_seqlens"])
    for key in ("x_q", "x_k"):
        inp[key] = inp[key].copy()
        inp[key][:, 1] = np.roll(inp[key][:, 1], 1, axis=0)   # perturb qk head 1
    r1 = ref.prefill(inp, inp["cu_seqlens"])
    np.testing.assert_array_equal(r0["y"][:, :2], r1["y"][:, :2])
    assert not np.allclose(r0["y"][:, 2:], r1["y"][:, 2:])


def test_identical_value_heads_give_identical_outputs():
    """Two value heads of one qk head with identical data and parameters agree exactly."""
    inp = _tiny_inputs((24,), h_qk=1, h_v=2, seed=5)
    d = 16
    for key in ("x_v", "z", "a", "b"):
        inp[key] = inp[key].copy()
        inp[key][:, 1] = inp[key][:, 0]
    inp["conv_w"] = inp["conv_w"].copy()
    inp["conv_w"][3 * d:4 * d] = inp["conv_w"][2 * d:3 * d]
    for key in ("A_log", "dt_bias"):
        inp[key] = inp[key].copy()
        inp[key][1] = inp[key][0]
    r = ref.prefill(inp, inp["cu_seqlens"])
    np.testing.assert_array_equal(r["y"][:, 0], r["y"][:, 1])
    np.testing.assert_array_equal(r["final_state"][0, 0], r["final_state"][0, 1])


def test_decode_continues_prefill():
    """prefill(T) + conv cache of the last 3 raw inputs + decode(token T) == prefill(T+1)."""
    inp = _tiny_inputs((21,), h_qk=1, h_v=2, seed=6)
    T = 20
    full = ref.prefill(inp, [0, T + 1])
    head = ref.prefill({k_: (v_[:T] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_)
                        for k_, v_ in inp.items()}, [0, T])
    xs = np.concatenate([inp["x_q"].reshape(T + 1, -1), inp["x_k"].reshape(T + 1, -1),
                         inp["x_v"].reshape(T + 1, -1)], axis=1)
    conv_state = xs[T - 3:T].T[None]          # [1, Cc, 3], oldest first
    dec = {k_: (v_[T:T + 1] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_)
           for k_, v_ in inp.items()}
    r = ref.decode_step(dec, conv_state, head["final_state"])
    np.testing.assert_allclose(r["y"][0], full["y"][T], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["state"][0], full["final_state"][0], rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(r["conv_state"][0], xs[T - 2:T + 1].T)


def test_synth_bf16_rounding():
    """The generator's bf16 rounding is round-to-nearest-even (checked against torch)."""
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32) * 100
    x[:4] = [1.00390625, 1.01171875, -1.00390625, 3.0e-39]  # ties and a subnormal
    np.testing.assert_array_equal(synth.round_bf16(x),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_conv_cache_after_prefill_equals_stepping_decode():
    """The conv cache a prefill leaves (the last three raw inputs, zeros before
    the sequence start) equals the cache that decoding the same tokens one by
    one from an empty cache builds up -- for sequences of 0, 1, 2 and 5 tokens."""
    lengths = (0, 1, 2, 5)
    inp = _tiny_inputs(lengths, h_qk=1, h_v=2, seed=8)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    cache = ref.conv_cache_after_prefill(inp, cu)
    h_qk, dk = inp["x_q"].shape[1:]
    h_v, dv = inp["x_v"].shape[1:]
    Cc = 2 * h_qk * dk + h_v * dv
    for n, L in enumerate(lengths):
        cs = np.zeros((1, Cc, 3))
        st = np.zeros((1, h_v, dk, dv))
        for t in range(cu[n], cu[n + 1]):
            tok = {k_: (v_[t:t + 1] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_) for k_, v_ in inp.items()}
            r = ref.decode_step(tok, cs, st)
            cs, st = r["conv_state"], r["state"]
        np.testing.assert_array_equal(cache[n], cs[0])


def test_short_sequence_prefill_then_decode():
    """A 2-token prefill leaves a cache with one zero entry; decoding the third
    token from it reproduces the 3-token prefill."""
    inp = _tiny_inputs((3,), h_qk=1, h_v=2, seed=9)
    T = 2
    full = ref.prefill(inp, [0, T + 1])
    head_inp = {k_: (v_[:T] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_) for k_, v_ in inp.items()}
    head = ref.prefill(head_inp, [0, T])
    cache = ref.conv_cache_after_prefill(head_inp, [0, T])
    assert np.all(cache[0, :, 0] == 0)
    dec = {k_: (v_[T:T + 1] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_) for k_, v_ in inp.items()}
    r = ref.decode_step(dec, cache, head["final_state"])
    np.testing.assert_allclose(r["y"][0], full["y"][T], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["state"][0], full["final_state"][0], rtol=1e-12, atol=1e-15)


def _segment(inp, cu, bounds):
    """Tokens [bounds[n][0], bounds[n][1]) of every sequence n, as one packed workload."""
    idx = np.concatenate([np.arange(cu[n] + b0, cu[n] + b1) for n, (b0, b1) in enumerate(bounds)]).astype(np.int64)
    seg = {k_: (v_[idx] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_) for k_, v_ in inp.items()}
    seg["cu_seqlens"] = np.concatenate([[0], np.cumsum([b1 - b0 for b0, b1 in bounds])]).astype(np.int64)
    return seg, idx


def test_split_prefill_with_carried_state_and_conv_equals_one_run():
    """Running every sequence as consecutive segments, each started from the
    previous segment's final state and conv history (the last three raw inputs,
    carried through conv_cache_after_prefill), equals one run over the whole
    sequence, bitwise -- including segments of 1 and 2 tokens, whose conv
    history reaches back through more than one segment, and empty ones."""
    lengths = (37, 64, 9)
    inp = _tiny_inputs(lengths, h_qk=1, h_v=2, seed=10, init_std=0.02)
    cu = inp["cu_seqlens"].astype(np.int64)
    full = ref.prefill(inp, cu, inp["init_state"])
    cuts = [(0, 20, 21, 23, 37), (0, 0, 64, 64, 64), (0, 1, 2, 4, 9)]   # segment boundaries per sequence
    state, conv = inp["init_state"], None
    for s in range(4):
        bounds = [(c[s], c[s + 1]) for c in cuts]
        seg, idx = _segment(inp, cu, bounds)
        r = ref.prefill(seg, seg["cu_seqlens"], state, init_conv=conv)
        np.testing.assert_array_equal(r["y"], full["y"][idx])
        conv = ref.conv_cache_after_prefill(seg, seg["cu_seqlens"], init_conv=conv)
        state = r["final_state"]
    np.testing.assert_array_equal(state, full["final_state"])
    np.testing.assert_array_equal(conv, ref.conv_cache_after_prefill(inp, cu))


def test_split_prefill_without_conv_history_differs():
    """The control: the same split with the state carried but the conv history
    dropped (zeros, as a plain prefill takes) changes the first three tokens
    after the split and none before it."""
    inp = _tiny_inputs((30,), h_qk=1, h_v=2, seed=11)
    full = ref.prefill(inp, [0, 30])
    head, _ = _segment(inp, np.array([0, 30]), [(0, 12)])
    tail, _ = _segment(inp, np.array([0, 30]), [(12, 30)])
    rh = ref.prefill(head, head["cu_seqlens"])
    rt = ref.prefill(tail, tail["cu_seqlens"], rh["final_state"])
    np.testing.assert_array_equal(rh["y"], full["y"][:12])
    assert not np.allclose(rt["y"][:3], full["y"][12:15])
    rc = ref.prefill(tail, tail["cu_seqlens"], rh["final_state"],
                     init_conv=ref.conv_cache_after_prefill(head, head["cu_seqlens"]))
    np.testing.assert_array_equal(rc["y"], full["y"][12:])
