"""The library's calls enqueue work and never synchronise the host, so they can
be captured in a CUDA graph and replayed (with a caller-owned workspace), and
calls on different streams with their own workspaces run side by side.  Each
case checks the results against the oracle."""
import numpy as np
import pytest

from gateddeltanet_layer_gb300 import synth
from oracle import oracle as ref
from tests.helpers import parity, parity_sum, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _gdn():
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    return gdn


def _prefill_args(t):
    return (t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"], t["dt_bias"],
            t["norm_w"], t["cu_seqlens"], t.get("init_state"))


@pytest.mark.parametrize("lengths,h_qk,h_v", [((150, 70), 2, 4), ((65, 1, 128, 30, 64, 100), 4, 8)],
                         ids=["few_chains", "many_chains"])
def test_prefill_replayed_from_a_cuda_graph(lengths, h_qk, h_v):
    """Capture one prefill call, then replay it twice with new input values
    copied into the captured tensors: each replay equals the oracle on the
    values it saw."""
    gdn = _gdn()
    cfg = synth.scaled(synth.VARLEN_32K, lengths=lengths, h_qk=h_qk, h_v=h_v, init_std=0.02, seed=71)
    inp = synth.make_prefill(cfg)
    t = to_torch(inp, True)
    ws = torch.zeros(gdn.prefill_workspace_bytes(cfg.T, cfg.N, h_qk, h_v, 128, 128, True), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((cfg.T, h_v, 128), dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((cfg.N, h_v, 128, 128), dtype=torch.float32, device="cuda")
    gdn.prefill(*_prefill_args(t), out=out, final_state=fs, workspace=ws)  # first call outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.prefill(*_prefill_args(t), out=out, final_state=fs, workspace=ws)
    for seed in (72, 73):
        new = synth.make_prefill(synth.scaled(cfg, seed=seed))
        tn = to_torch(new, True)
        for key in ("x_q", "x_k", "x_v", "a", "b", "z", "init_state", "conv_w", "A_log", "dt_bias", "norm_w"):
            t[key].copy_(tn[key])  # new values in the captured tensors (the parameters too)
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.workspace_status(ws) == 0
        r = ref.prefill(new, new["cu_seqlens"], new["init_state"])
        parity(out.float().cpu().numpy(), r["y"], "bf16", f"graph replay {seed} out")
        parity(fs.cpu().numpy(), r["final_state"], "bf16", f"graph replay {seed} final_state")


def test_decode_steps_replayed_from_a_cuda_graph():
    """A serving loop: four decode steps captured in one graph (the state and
    conv cache updated in place from step to step), replayed: every step's
    output and the final state and cache equal four oracle decode steps."""
    gdn = _gdn()
    steps = 4
    dcfg = synth.scaled(synth.DECODE_256, batch=5, h_qk=2, h_v=4)
    base = synth.make_decode(dcfg)
    per_step = [synth.make_decode(synth.scaled(dcfg, seed=100 + i)) for i in range(steps)]
    t0 = to_torch(base, True)
    conv_state, state = t0["conv_state"], t0["state"]
    ins = [to_torch(s_, True) for s_ in per_step]
    outs = [torch.empty((dcfg.batch, dcfg.h_v, dcfg.d_v), dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    keys = ("x_q", "x_k", "x_v", "a", "b", "z")

    def loop():
        for i in range(steps):
            d = ins[i]
            gdn.decode_step(d["x_q"], d["x_k"], d["x_v"], d["a"], d["b"], d["z"], t0["conv_w"], t0["A_log"],
                            t0["dt_bias"], t0["norm_w"], conv_state, state, out=outs[i])

    # warm the library up on scratch copies, then capture on the real state
    cs_keep, st_keep = conv_state.clone(), state.clone()
    loop()
    torch.cuda.synchronize()
    conv_state.copy_(cs_keep)
    state.copy_(st_keep)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        loop()
    conv_state.copy_(cs_keep)  # capture does not run the work; start from the initial state
    state.copy_(st_keep)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    cs_ref, st_ref = base["conv_state"], base["state"]
    for i in range(steps):
        step_inp = dict(base)
        for k in keys:
            step_inp[k] = per_step[i][k]
        r = ref.decode_step(step_inp, cs_ref, st_ref)
        parity(outs[i].float().cpu().numpy(), r["y"], "bf16", f"graph decode step {i}")
        cs_ref, st_ref = r["conv_state"], r["state"]
    parity(state.cpu().numpy(), st_ref, "bf16", "graph decode final state")
    np.testing.assert_array_equal(conv_state.float().cpu().numpy(), cs_ref)


def test_two_prefills_on_two_streams():
    """Two different workloads on two streams at once, each with its own
    workspace: both equal the oracle."""
    gdn = _gdn()
    cfgs = [synth.scaled(synth.VARLEN_32K, lengths=(300, 90), h_qk=2, h_v=4, init_std=0.02, seed=81),
            synth.scaled(synth.VARLEN_32K, lengths=(64, 1, 200, 7, 130), h_qk=4, h_v=8, init_std=0.02, seed=82)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    results = []
    for cfg, st in zip(cfgs, streams):
        inp = synth.make_prefill(cfg)
        t = to_torch(inp, True)
        torch.cuda.synchronize()
        ws = torch.zeros(gdn.prefill_workspace_bytes(cfg.T, cfg.N, cfg.h_qk, cfg.h_v, 128, 128, True),
                         dtype=torch.uint8, device="cuda")
        with torch.cuda.stream(st):
            out, fs = gdn.prefill(*_prefill_args(t), workspace=ws, stream=st)
        results.append((inp, out, fs, ws, st))
    torch.cuda.synchronize()
    for inp, out, fs, ws, st in results:
        assert gdn.workspace_status(ws, st) == 0
        r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"])
        parity(out.float().cpu().numpy(), r["y"], "bf16", "two streams out")
        parity(fs.cpu().numpy(), r["final_state"], "bf16", "two streams final_state")


@pytest.mark.parametrize("path", ["segmented", "carry", "fp32", "backward"])
def test_other_paths_replayed_from_a_cuda_graph(path):
    """The segment-parallel prefill, the carried-conv prefill, the fp32 prefill
    and the backward, each captured once with a caller-owned workspace and
    replayed on new values copied into the captured tensors: each replay
    equals the oracle on the values it saw."""
    gdn = _gdn()
    fp32 = path == "fp32"
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(200, 1, 97), h_qk=2, h_v=4, init_std=0.02,
                       dtype="fp32" if fp32 else "bf16", seed=91)
    sdt = torch.float32 if fp32 else torch.bfloat16
    inp = synth.make_prefill(cfg)
    t = to_torch(inp, not fp32)
    Cc = 2 * cfg.h_qk * cfg.d_k + cfg.h_v * cfg.d_v
    hist = torch.zeros((cfg.N, Cc, 3), dtype=sdt, device="cuda")
    dy = torch.zeros((cfg.T, cfg.h_v, cfg.d_v), dtype=sdt, device="cuda")
    if path == "segmented":
        nbytes = gdn.prefill_segmented_workspace_bytes(cfg.T, cfg.N, cfg.h_qk, cfg.h_v, 128, 128, 2)
    elif path == "backward":
        nbytes = gdn.prefill_backward_workspace_bytes(cfg.T, cfg.N, cfg.h_qk, cfg.h_v, 128, 128, not fp32)
    else:
        nbytes = gdn.prefill_workspace_bytes(cfg.T, cfg.N, cfg.h_qk, cfg.h_v, 128, 128, not fp32)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((cfg.T, cfg.h_v, 128), dtype=sdt, device="cuda")
    fs = torch.empty((cfg.N, cfg.h_v, 128, 128), dtype=torch.float32, device="cuda")
    fc = torch.empty((cfg.N, Cc, 3), dtype=sdt, device="cuda")
    res = {}

    def call():
        args = _prefill_args(t)
        if path == "segmented":
            gdn.prefill_segmented(*args, seg_chunks=2, out=out, final_state=fs, workspace=ws)
        elif path == "carry":
            gdn.prefill_carry(*args, hist, out=out, final_state=fs, final_conv=fc, workspace=ws)
        elif path == "fp32":
            gdn.prefill(*args, out=out, final_state=fs, workspace=ws)
        else:
            res["g"] = gdn.prefill_backward(*args[:-1], dy, args[-1], workspace=ws)

    call()  # first call outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for seed in (92, 93):
        new = synth.make_prefill(synth.scaled(cfg, seed=seed))
        tn = to_torch(new, not fp32)
        for key in ("x_q", "x_k", "x_v", "a", "b", "z", "init_state", "conv_w", "A_log", "dt_bias", "norm_w"):
            t[key].copy_(tn[key])
        rng = np.random.default_rng(seed)
        h_new = synth.round_bf16(rng.standard_normal((cfg.N, Cc, 3)).astype(np.float32))
        dy_new = rng.standard_normal((cfg.T, cfg.h_v, 128)).astype(np.float32)
        if not fp32:
            dy_new = synth.round_bf16(dy_new)
        hist.copy_(torch.from_numpy(h_new))
        dy.copy_(torch.from_numpy(dy_new))
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.workspace_status(ws) == 0
        what = f"{path} graph replay {seed}"
        if path == "backward":
            r = ref.prefill_backward(new, new["cu_seqlens"], dy_new, new["init_state"])
            g = res["g"]
            for name, key in (("q", "x_q"), ("k", "x_k"), ("v", "x_v"), ("a", "a"), ("b", "b"), ("z", "z"),
                              ("init_state", "init_state")):
                parity(g[name].cpu().numpy(), r[key], "fp32", f"{what} d{name}")
            for name in ("conv_w", "A_log", "dt_bias", "norm_w"):
                parity_sum(g[name].cpu().numpy(), r[name], "fp32", f"{what} d{name}")
            continue
        r = ref.prefill(new, new["cu_seqlens"], new["init_state"], init_conv=h_new if path == "carry" else None)
        dt = "fp32" if fp32 else "bf16"
        parity(out.float().cpu().numpy(), r["y"], dt, f"{what} out")
        parity(fs.cpu().numpy(), r["final_state"], dt, f"{what} final_state")
        if path == "carry":
            np.testing.assert_array_equal(fc.float().cpu().numpy(),
                                          ref.conv_cache_after_prefill(new, new["cu_seqlens"], init_conv=h_new))
