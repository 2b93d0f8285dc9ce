"""GPU parity of gdn_decode_step against the fp64 oracle, and the prefill ->
decode hand-off (prefill of T tokens, then one decode step, equals the oracle's
prefill of T+1 tokens)."""
import numpy as np
import pytest

from gateddeltanet_layer_gb300 import synth
from oracle import oracle as ref
from tests.helpers import parity, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _gdn():
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    return gdn


def run_decode(inp, bf16):
    gdn = _gdn()
    t = to_torch(inp, bf16)
    out = gdn.decode_step(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                          t["dt_bias"], t["norm_w"], t["conv_state"], t["state"])
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), t["state"].cpu().numpy(), t["conv_state"].float().cpu().numpy()


@pytest.mark.parametrize("cfg", [
    synth.scaled(synth.DECODE_256, batch=5, h_qk=2, h_v=4),
    synth.scaled(synth.DECODE_256, batch=3, h_qk=2, h_v=2, d_k=16, d_v=16, dtype="fp32"),
    synth.scaled(synth.DECODE_256, batch=4, h_qk=1, h_v=2, d_k=64, d_v=128, seed=2),
], ids=["bf16_d128", "fp32_d16", "bf16_dk64"])
def test_decode_small(cfg):
    inp = synth.make_decode(cfg)
    y, st, cs = run_decode(inp, cfg.dtype == "bf16")
    r = ref.decode_step(inp, inp["conv_state"], inp["state"])
    parity(y, r["y"], cfg.dtype, "out")
    parity(st, r["state"], cfg.dtype, "state")
    np.testing.assert_array_equal(cs, r["conv_state"])  # a byte move: exact


@pytest.mark.slow
def test_decode_full_config():
    """B=256, H=16/32, d=128: every sequence and head (the oracle is cheap for one token)."""
    cfg = synth.DECODE_256
    inp = synth.make_decode(cfg)
    y, st, cs = run_decode(inp, True)
    r = ref.decode_step(inp, inp["conv_state"], inp["state"])
    parity(y, r["y"], "bf16", "out")
    parity(st, r["state"], "bf16", "state")
    np.testing.assert_array_equal(cs, r["conv_state"])


def test_prefill_then_decode_continues_the_sequence():
    gdn = _gdn()
    T = 133
    cfg = synth.scaled(synth.SINGLE_4K, lengths=(T + 1,), h_qk=2, h_v=4, init_std=0.02, seed=21)
    inp = synth.make_prefill(cfg)
    full = ref.prefill(inp, [0, T + 1], inp["init_state"])
    head = {k_: (v_[:T] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_) for k_, v_ in inp.items()}
    head["cu_seqlens"] = np.array([0, T], dtype=np.int32)
    th = to_torch(head, True)
    _, fs = gdn.prefill(th["x_q"], th["x_k"], th["x_v"], th["a"], th["b"], th["z"], th["conv_w"], th["A_log"],
                        th["dt_bias"], th["norm_w"], th["cu_seqlens"], th["init_state"])
    xs = np.concatenate([inp["x_q"].reshape(T + 1, -1), inp["x_k"].reshape(T + 1, -1),
                         inp["x_v"].reshape(T + 1, -1)], axis=1)
    dec = {k_: (v_[T:T + 1] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_) for k_, v_ in inp.items()}
    dec["conv_state"] = np.ascontiguousarray(xs[T - 3:T].T[None])
    td = to_torch(dec, True)
    out = gdn.decode_step(td["x_q"], td["x_k"], td["x_v"], td["a"], td["b"], td["z"], td["conv_w"],
                          td["A_log"], td["dt_bias"], td["norm_w"], td["conv_state"], fs)
    torch.cuda.synchronize()
    parity(out.float().cpu().numpy()[0], full["y"][T], "bf16", "decoded token")
    parity(fs.cpu().numpy(), full["final_state"], "bf16", "state after decode")
