"""A seeded sweep of small random workloads through the chunked prefill, the
segment-parallel prefill and the carried-conv prefill, every chain against the
oracle: random sequence counts and lengths (empty, 1-token, chunk-edge and
multi-chunk sequences), q/k and value head counts (1 to 16 value heads per q/k
head, so one or several chunk-prep groups and both state-pass forms), initial
states present or not, the final state written over the initial one, and
random segment lengths; the backward and the decode step on random small
workloads; and (slow) random medium packed batches at the graded head counts."""
import numpy as np
import pytest

from gateddeltanet_layer_gb300 import synth
from oracle import oracle as ref
from tests.helpers import parity, parity_sum, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EDGE_LENGTHS = (0, 1, 2, 3, 63, 64, 65, 127, 128, 129)


def _draw(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 7))
    lengths = tuple(int(rng.choice(EDGE_LENGTHS)) if rng.random() < 0.5 else int(rng.integers(0, 400))
                    for _ in range(n))
    if sum(lengths) == 0:
        lengths = lengths[:-1] + (70,)
    h_qk = int(rng.choice([1, 2, 4]))
    rep = int(rng.choice([1, 2, 3, 4, 8, 12, 16]))
    init_std = float(rng.choice([0.0, 0.02]))
    cfg = synth.scaled(synth.VARLEN_32K, lengths=lengths, h_qk=h_qk, h_v=h_qk * rep, init_std=init_std,
                       seed=1000 + seed)
    return cfg, rng


@pytest.mark.parametrize("seed", range(12))
def test_random_workload(seed):
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    cfg, rng = _draw(seed)
    inp = synth.make_prefill(cfg)
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"])
    t = to_torch(inp, True)
    args = (t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"], t["dt_bias"],
            t["norm_w"], t["cu_seqlens"])
    what = f"seed {seed} (lengths {cfg.lengths}, {cfg.h_qk}/{cfg.h_v} heads)"

    # the chunked prefill; with an initial state, in place every other seed
    init = t.get("init_state")
    in_place = init is not None and seed % 2 == 0
    out, fs = gdn.prefill(*args, None if init is None else init.clone() if not in_place else init,
                          final_state=init if in_place else None)
    torch.cuda.synchronize()
    parity(out.float().cpu().numpy(), r["y"], "bf16", f"{what} out")
    parity(fs.cpu().numpy(), r["final_state"], "bf16", f"{what} final_state")

    # the segment-parallel prefill with a random segment length
    seg = int(rng.choice([1, 2, 3, 5]))
    init2 = None if inp["init_state"] is None else to_torch({"init_state": inp["init_state"]}, True)["init_state"]
    out2, fs2 = gdn.prefill_segmented(*args, init2, seg_chunks=seg)
    torch.cuda.synchronize()
    parity(out2.float().cpu().numpy(), r["y"], "bf16", f"{what} segmented({seg}) out")
    parity(fs2.cpu().numpy(), r["final_state"], "bf16", f"{what} segmented({seg}) final_state")

    # the carried-conv prefill with a random conv history, against the oracle given the same history
    Cc = 2 * cfg.h_qk * cfg.d_k + cfg.h_v * cfg.d_v
    hist = synth.round_bf16(np.random.default_rng(seed + 500).standard_normal((cfg.N, Cc, 3)).astype(np.float32))
    r3 = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"], init_conv=hist)
    init3 = None if inp["init_state"] is None else to_torch({"init_state": inp["init_state"]}, True)["init_state"]
    out3, fs3, fc3 = gdn.prefill_carry(*args, init3, torch.from_numpy(hist).to("cuda", torch.bfloat16))
    torch.cuda.synchronize()
    parity(out3.float().cpu().numpy(), r3["y"], "bf16", f"{what} carry out")
    parity(fs3.cpu().numpy(), r3["final_state"], "bf16", f"{what} carry final_state")
    np.testing.assert_array_equal(fc3.float().cpu().numpy(),
                                  ref.conv_cache_after_prefill(inp, inp["cu_seqlens"], init_conv=hist))


@pytest.mark.parametrize("seed", range(6))
def test_random_backward(seed):
    """The backward on random small workloads (head dims 16 to 128, 1 to 4
    value heads per q/k head, bf16 or fp32 streams, with or without an initial
    state and a final-state gradient): the per-token gradients and the
    initial state's at the fp32 bar element by element, the parameter
    gradients (sums over every token and head) normwise."""
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    rng = np.random.default_rng(seed + 200)
    n = int(rng.integers(1, 4))
    lengths = tuple(int(rng.choice(EDGE_LENGTHS)) if rng.random() < 0.5 else int(rng.integers(0, 150))
                    for _ in range(n))
    if sum(lengths) == 0:
        lengths = lengths[:-1] + (40,)
    d = int(rng.choice([16, 32, 128]))
    h_qk = int(rng.choice([1, 2]))
    rep = int(rng.choice([1, 2, 4]))
    dtype = str(rng.choice(["bf16", "fp32"]))
    cfg = synth.scaled(synth.VARLEN_32K, lengths=lengths, h_qk=h_qk, h_v=h_qk * rep, d_k=d, d_v=d, dtype=dtype,
                       init_std=float(rng.choice([0.0, 0.02])), seed=2000 + seed)
    bf16 = dtype == "bf16"
    inp = synth.make_prefill(cfg)
    dy = rng.standard_normal((cfg.T, cfg.h_v, cfg.d_v)).astype(np.float32)
    if bf16:
        dy = synth.round_bf16(dy)
    dfinal = rng.standard_normal((cfg.N, cfg.h_v, d, d)).astype(np.float32) if rng.random() < 0.5 else None
    t = to_torch(inp, bf16)
    g = gdn.prefill_backward(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                             t["dt_bias"], t["norm_w"], t["cu_seqlens"],
                             torch.from_numpy(dy).to("cuda", torch.bfloat16 if bf16 else torch.float32),
                             t.get("init_state"), None if dfinal is None else torch.from_numpy(dfinal).cuda())
    torch.cuda.synchronize()
    r = ref.prefill_backward(inp, inp["cu_seqlens"], dy, inp["init_state"], dfinal)
    what = f"seed {seed} (lengths {lengths}, {h_qk}/{h_qk * rep} heads, d {d}, {dtype})"
    for name, key in (("q", "x_q"), ("k", "x_k"), ("v", "x_v"), ("a", "a"), ("b", "b"), ("z", "z"),
                      ("conv_w", "conv_w"), ("A_log", "A_log"), ("dt_bias", "dt_bias"), ("norm_w", "norm_w"),
                      ("init_state", "init_state")):
        check = parity_sum if name in ("conv_w", "A_log", "dt_bias", "norm_w") else parity
        check(g[name].cpu().numpy(), r[key], "fp32", f"{what} d{name}")


@pytest.mark.slow
@pytest.mark.parametrize("seed", range(6))
def test_random_medium_workload(seed):
    """Packed batches of 1 to 40 sequences of 0 to 2000 tokens at the graded
    head counts (16/32 heads, d = 128, nonzero initial states): many chunk-prep
    waves and several state-pass rounds, through the plain prefill and the
    segment-parallel one with a random segment length, every chain against the
    oracle."""
    import os

    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    rng = np.random.default_rng(seed + 5000)
    n = int(rng.integers(1, 41))
    lengths = tuple(int(x) for x in rng.integers(0, 2000, size=n))
    if sum(lengths) == 0:
        lengths = (100,)
    cfg = synth.scaled(synth.VARLEN_32K, lengths=lengths, init_std=0.02, seed=6000 + seed)
    inp = synth.make_prefill(cfg)
    t = to_torch(inp, True)
    args = (t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"], t["dt_bias"],
            t["norm_w"], t["cu_seqlens"], t["init_state"])
    out, fs = gdn.prefill(*args)
    seg = int(rng.integers(1, 17))
    out2, fs2 = gdn.prefill_segmented(*args, seg_chunks=seg)
    torch.cuda.synchronize()
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"], threads=os.cpu_count())
    what = f"seed {seed} ({n} sequences, {cfg.T} tokens)"
    parity(out.float().cpu().numpy(), r["y"], "bf16", f"{what} out")
    parity(fs.cpu().numpy(), r["final_state"], "bf16", f"{what} final_state")
    parity(out2.float().cpu().numpy(), r["y"], "bf16", f"{what} segmented({seg}) out")
    parity(fs2.cpu().numpy(), r["final_state"], "bf16", f"{what} segmented({seg}) final_state")


@pytest.mark.parametrize("seed", range(8))
def test_random_decode(seed):
    """The decode step on random batches (1 to 300 sequences), q/k and value
    head counts (1 to 16 value heads per q/k head), head dims (16 to 128, d_k
    and d_v drawn apart) and stream dtypes: output and state against the
    oracle, the conv cache exactly."""
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    rng = np.random.default_rng(seed + 7000)
    h_qk = int(rng.choice([1, 2, 4, 16]))
    rep = int(rng.choice([1, 2, 3, 8, 16]))
    dtype = str(rng.choice(["bf16", "fp32"]))
    cfg = synth.scaled(synth.DECODE_256, batch=int(rng.integers(1, 301)), h_qk=h_qk, h_v=h_qk * rep,
                       d_k=int(rng.choice([16, 32, 64, 128])), d_v=int(rng.choice([16, 32, 64, 128])), dtype=dtype,
                       seed=8000 + seed)
    bf16 = dtype == "bf16"
    inp = synth.make_decode(cfg)
    t = to_torch(inp, bf16)
    out = gdn.decode_step(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                          t["dt_bias"], t["norm_w"], t["conv_state"], t["state"])
    torch.cuda.synchronize()
    r = ref.decode_step(inp, inp["conv_state"], inp["state"])
    what = f"seed {seed} (B {cfg.batch}, {h_qk}/{h_qk * rep} heads, d {cfg.d_k}/{cfg.d_v}, {dtype})"
    parity(out.float().cpu().numpy(), r["y"], dtype, f"{what} out")
    parity(t["state"].cpu().numpy(), r["state"], dtype, f"{what} state")
    np.testing.assert_array_equal(t["conv_state"].float().cpu().numpy(), r["conv_state"])
