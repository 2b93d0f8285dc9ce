"""Pins of the oracle's backward pass: central finite differences of the
forward oracle, on every element of every input of a tiny layer.

The loss is  sum(dy * y) + sum(dfinal * final_state)  for fixed random dy and
dfinal; its gradient with respect to each input (the raw streams, the gates'
inputs, every parameter, the initial state and the carried conv history) from
oracle.prefill_backward must equal (loss(x + h) - loss(x - h)) / 2h.  Two
packed sequences, two value heads on one q/k head (so the q/k gradients add
up over heads), one head with slow decay so that gradients flow through many
steps of the state, nonzero initial states and conv history.
"""
import numpy as np
import pytest

from gateddeltanet_layer_gb300 import synth
from oracle import oracle as ref


def _problem(seed=0, lengths=(6, 4), d=4):
    cfg = synth.scaled(synth.TINY, lengths=lengths, h_qk=1, h_v=2, d_k=d, d_v=d, init_std=0.3, seed=seed)
    inp = {k: (None if v is None else np.asarray(v, dtype=np.float64)) for k, v in synth.make_prefill(cfg).items()}
    inp["cu_seqlens"] = np.asarray(inp["cu_seqlens"], dtype=np.int64)
    inp["dt_bias"] = np.array([-2.0, 0.5])      # value head 0 decays slowly, head 1 fast
    inp["A_log"] = np.log(np.array([1.2, 6.0]))
    rng = np.random.default_rng(seed + 100)
    Cc = cfg.channels
    inp["init_conv"] = rng.standard_normal((cfg.N, Cc, 3))
    dy = rng.standard_normal((cfg.T, 2, d))
    dfinal = rng.standard_normal((cfg.N, 2, d, d))
    return inp, dy, dfinal


def _loss(inp, dy, dfinal):
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"], init_conv=inp["init_conv"], threads=1)
    return float(np.sum(dy * r["y"]) + np.sum(dfinal * r["final_state"]))


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_equals_central_differences_everywhere(seed):
    inp, dy, dfinal = _problem(seed)
    gr = ref.prefill_backward(inp, inp["cu_seqlens"], dy, inp["init_state"], dfinal, threads=1,
                              init_conv=inp["init_conv"])
    for key in ("x_q", "x_k", "x_v", "z", "a", "b", "conv_w", "A_log", "dt_bias", "norm_w", "init_state",
                "init_conv"):
        x = inp[key]
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            h = 1e-6 * max(1.0, abs(x[idx]))
            keep = x[idx]
            x[idx] = keep + h
            lp = _loss(inp, dy, dfinal)
            x[idx] = keep - h
            lm = _loss(inp, dy, dfinal)
            x[idx] = keep
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(gr[key], fd, rtol=2e-6, atol=2e-8, err_msg=key)
        assert np.any(gr[key] != 0), key


def test_backward_of_a_split_equals_backward_of_one_run():
    """Reverse mode through a split: the gradient of the second segment's
    initial state and conv history, fed back as the gradient of the first
    segment's final state and final conv history, reproduces the unsplit
    gradient of the first segment's streams (the hand-off is differentiable
    the same way as the forward)."""
    inp, dy, _ = _problem(seed=3, lengths=(10,))
    inp["init_conv"] = None
    cut = 6
    full = ref.prefill_backward(inp, [0, 10], dy, inp["init_state"], threads=1)
    head = {k: (v[:cut] if k in ("x_q", "x_k", "x_v", "z", "a", "b") else v) for k, v in inp.items()}
    tail = {k: (v[cut:] if k in ("x_q", "x_k", "x_v", "z", "a", "b") else v) for k, v in inp.items()}
    rh = ref.prefill(head, [0, cut], inp["init_state"], threads=1)
    conv = ref.conv_cache_after_prefill(head, [0, cut])
    gt = ref.prefill_backward(tail, [0, 10 - cut], dy[cut:], rh["final_state"], threads=1, init_conv=conv)
    # the conv history of the tail is the head's last three raw inputs: its gradient lands on those rows
    hg = ref.prefill_backward(head, [0, cut], dy[:cut], inp["init_state"], gt["init_state"], threads=1)
    d = inp["x_q"].shape[2]
    dxq = hg["x_q"].copy()
    dxq[cut - 3:cut, 0] += gt["init_conv"][0, :d].T
    np.testing.assert_allclose(dxq, full["x_q"][:cut], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(gt["x_q"], full["x_q"][cut:], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(hg["init_state"], full["init_state"], rtol=1e-10, atol=1e-13)
