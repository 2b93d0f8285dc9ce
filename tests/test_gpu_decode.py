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


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_conv_cache_from_prefill_is_exact(dtype):
    """The library's conv cache after a prefill equals the oracle's (a byte move)
    for sequences of 0, 1, 2, 5 and 130 tokens."""
    gdn = _gdn()
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(0, 1, 2, 5, 130), h_qk=2, h_v=4, seed=31, dtype=dtype,
                       d_k=16 if dtype == "fp32" else 128, d_v=16 if dtype == "fp32" else 128)
    inp = synth.make_prefill(cfg)
    t = to_torch(inp, dtype == "bf16")
    cache = gdn.conv_cache_from_prefill(t["x_q"], t["x_k"], t["x_v"], t["cu_seqlens"])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cache.float().cpu().numpy(), ref.conv_cache_after_prefill(inp, inp["cu_seqlens"]))


def test_prefill_hand_off_to_decode_through_the_library():
    """prefill of two sequences, the library's conv cache and final state, one
    decode step: equals the oracle's prefill of one more token per sequence."""
    gdn = _gdn()
    L = (70, 2)
    cfg = synth.scaled(synth.VARLEN_32K, lengths=tuple(x + 1 for x in L), h_qk=2, h_v=4, init_std=0.02, seed=32)
    inp = synth.make_prefill(cfg)
    cu_full = inp["cu_seqlens"]
    full = ref.prefill(inp, cu_full, inp["init_state"])
    keep = np.concatenate([np.arange(cu_full[n], cu_full[n + 1] - 1) for n in range(len(L))])
    last = cu_full[1:] - 1
    seq = ("x_q", "x_k", "x_v", "z", "a", "b")
    head = {k_: (v_[keep] if k_ in seq else v_) for k_, v_ in inp.items()}
    head["cu_seqlens"] = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    th = to_torch(head, True)
    _, fs = gdn.prefill(th["x_q"], th["x_k"], th["x_v"], th["a"], th["b"], th["z"], th["conv_w"], th["A_log"],
                        th["dt_bias"], th["norm_w"], th["cu_seqlens"], th["init_state"])
    cache = gdn.conv_cache_from_prefill(th["x_q"], th["x_k"], th["x_v"], th["cu_seqlens"])
    dec = {k_: (v_[last] if k_ in seq else v_) for k_, v_ in inp.items()}
    td = to_torch(dec, True)
    out = gdn.decode_step(td["x_q"], td["x_k"], td["x_v"], td["a"], td["b"], td["z"], td["conv_w"],
                          td["A_log"], td["dt_bias"], td["norm_w"], cache, fs)
    torch.cuda.synchronize()
    parity(out.float().cpu().numpy(), full["y"][last], "bf16", "decoded tokens")
    parity(fs.cpu().numpy(), full["final_state"], "bf16", "states after decode")


def _pool_case(seed=33, P=7, slots=(5, 0, 3, 6)):
    cfg = synth.scaled(synth.DECODE_256, batch=len(slots), h_qk=2, h_v=4, seed=seed)
    inp = synth.make_decode(cfg)
    rng = np.random.default_rng(seed)
    h_v, dk, dv = inp["state"].shape[1:]
    Cc = inp["conv_state"].shape[1]
    pool_state = (0.02 * rng.standard_normal((P, h_v, dk, dv))).astype(np.float32)
    pool_cs = synth.round_bf16(rng.standard_normal((P, Cc, 3)).astype(np.float32))
    return inp, pool_state, pool_cs, np.asarray(slots, dtype=np.int32)


def test_decode_slots_reads_and_updates_pool_entries():
    gdn = _gdn()
    inp, pool_state, pool_cs, slots = _pool_case()
    t = to_torch(inp, True)
    ps = torch.from_numpy(pool_state).cuda()
    pc = torch.from_numpy(pool_cs).cuda().to(torch.bfloat16)
    sl = torch.from_numpy(slots).cuda()
    out = gdn.decode_step_slots(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                                t["dt_bias"], t["norm_w"], pc, ps, sl)
    torch.cuda.synchronize()
    r = ref.decode_step(inp, pool_cs[slots], pool_state[slots])
    parity(out.float().cpu().numpy(), r["y"], "bf16", "out")
    got_s, got_c = ps.cpu().numpy(), pc.float().cpu().numpy()
    parity(got_s[slots], r["state"], "bf16", "pool states in use")
    np.testing.assert_array_equal(got_c[slots], r["conv_state"])
    untouched = np.setdiff1d(np.arange(len(pool_state)), slots)
    np.testing.assert_array_equal(got_s[untouched], pool_state[untouched])
    np.testing.assert_array_equal(got_c[untouched], pool_cs[untouched])


def test_decode_slots_out_of_range_is_reported():
    gdn = _gdn()
    inp, pool_state, pool_cs, slots = _pool_case(seed=34, P=5, slots=(1, 5, 4))  # 5 is outside the pool
    t = to_torch(inp, True)
    ps = torch.from_numpy(pool_state).cuda()
    pc = torch.from_numpy(pool_cs).cuda().to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gdn.decode_step_slots(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                                t["dt_bias"], t["norm_w"], pc, ps, torch.from_numpy(slots).cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    y = out.float().cpu().numpy()
    assert np.all(y[1] == 0)
    ok = np.array([0, 2])
    r = ref.decode_step({k_: (v_[ok] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_) for k_, v_ in inp.items()},
                        pool_cs[slots[ok]], pool_state[slots[ok]])
    parity(y[ok], r["y"], "bf16", "valid sequences")
    got_s = ps.cpu().numpy()
    np.testing.assert_array_equal(got_s[[0, 2, 3]], pool_state[[0, 2, 3]])  # entries no valid slot names
