"""GPU parity of gdn_prefill against the fp64 oracle.

Every case compares every (sequence, value head) chain: all of `out` and all
of `final_state`.  The full-size workloads run the whole GPU call exactly as
the benchmark launches it and run the oracle sequence by sequence on every
host core.
"""
import os

import numpy as np
import pytest

from gateddeltanet_layer_gb300 import synth
from oracle import oracle as ref
from tests.helpers import Parity, parity, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _gdn():
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    return gdn


def run_gpu(inp, bf16, *, workspace=None, in_place=False):
    gdn = _gdn()
    t = to_torch(inp, bf16)
    init = t.get("init_state")
    fs = init if (in_place and init is not None) else None
    out, fs = gdn.prefill(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                          t["dt_bias"], t["norm_w"], t["cu_seqlens"], init, final_state=fs,
                          workspace=workspace)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fs.cpu().numpy()


def check(inp, cfg_dtype, **kw):
    bf16 = cfg_dtype == "bf16"
    y, fs = run_gpu(inp, bf16, **kw)
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"])
    parity(y, r["y"], cfg_dtype, "out")
    parity(fs, r["final_state"], cfg_dtype, "final_state")
    return y, fs, r


def test_tiny_fp32_config():
    """T=64, H=2/2, d=16, fp32: every output and the final state within 1e-4."""
    check(synth.make_prefill(synth.TINY), "fp32")


@pytest.mark.parametrize("case", ["ragged_single", "varlen_edges", "long_memory", "gqa4", "gqa8", "gqa12", "gqa16",
                                  "fp32_d128", "gqa1", "gqa3", "chunk_edges", "fast_decay", "bf16_dk128_dv64",
                                  "fp32_dk64_dv128"])
def test_small_cases(case):
    if case == "ragged_single":      # several chunks plus a ragged tail
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(200,), h_qk=2, h_v=4)
    elif case == "varlen_edges":     # empty, 1-token, exact-chunk and straddling sequences
        cfg = synth.scaled(synth.VARLEN_32K, lengths=(64, 1, 0, 130, 63, 65), h_qk=1, h_v=2, seed=3)
    elif case == "long_memory":      # slow decay: dt_bias = -6 keeps alpha near 1
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(300,), h_qk=1, h_v=2, a_log_range=(1.0, 1.5),
                           init_std=0.02, seed=5)
    elif case == "gqa4":             # 4 value heads per q/k head
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(97, 31), h_qk=1, h_v=4, seed=7)
    elif case == "gqa3":             # value heads in a pair and a single one after it
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(130, 45), h_qk=2, h_v=6, init_std=0.02, seed=11)
    elif case == "gqa1":             # one value head per q/k head
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(150,), h_qk=2, h_v=2, init_std=0.02, seed=10)
    elif case == "chunk_edges":      # exactly one chunk, one chunk + 1, two chunks - 1, one token
        cfg = synth.scaled(synth.VARLEN_32K, lengths=(64, 65, 127, 1, 128), h_qk=1, h_v=2, seed=11)
    elif case == "fast_decay":       # gates near their strongest: A_log up to log 16 and large dt_bias
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(200,), h_qk=1, h_v=2, init_std=0.02, seed=12)
    elif case == "gqa8":             # the most value heads one chunk-prep CTA takes
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(70,), h_qk=1, h_v=8, seed=8)
    elif case == "gqa12":            # a group of 8 value heads and one of 4, each redoing the q/k part
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(70, 130), h_qk=1, h_v=12, init_std=0.02, seed=13)
    elif case == "gqa16":            # two groups of 8 value heads per q/k head
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(70,), h_qk=1, h_v=16, seed=9)
    elif case == "bf16_dk128_dv64":  # the token-sequential kernel's d_k = 128 form with two 32-column slices
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(90, 41), h_qk=1, h_v=2, d_k=128, d_v=64, init_std=0.02, seed=14)
    elif case == "fp32_dk64_dv128":  # its general form with four slices
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(77,), h_qk=2, h_v=4, d_k=64, d_v=128, dtype="fp32",
                           init_std=0.02, seed=15)
    else:                            # fp32 streams at d = 128 (token-sequential fp32 kernel)
        cfg = synth.scaled(synth.SINGLE_4K, lengths=(130, 7), h_qk=1, h_v=2, dtype="fp32", init_std=0.02)
    inp = synth.make_prefill(cfg)
    if case == "long_memory":
        inp["dt_bias"][:] = -6.0
    if case == "fast_decay":
        inp["dt_bias"][:] = 4.0
        inp["A_log"][:] = np.log(16.0)
    check(inp, cfg.dtype)


@pytest.mark.parametrize("lengths,h_qk,h_v", [
    ((150, 1, 64), 2, 8),                  # 24 chains: one CTA per SM, a ring of operand sets
    ((65, 1, 128, 30, 64), 4, 8),          # 40 chains: two CTAs per SM, one set per kind
    ((65, 1, 128, 30, 64, 100, 7, 64, 129, 3), 16, 32),  # 320 chains: more CTAs than fit at once
    ((200, 64, 1, 90), 2, 32),             # 128 chains, 16 value heads per q/k head (two prep groups)
], ids=["chains24", "chains40", "chains320", "chains128_gqa16"])
def test_state_pass_chain_counts(lengths, h_qk, h_v):
    """Few and many (sequence, value head) chains (the state pass runs a ring
    of operand sets at one CTA per SM for few chains, two CTAs per SM
    otherwise), every chain against the oracle."""
    cfg = synth.scaled(synth.VARLEN_32K, lengths=lengths, h_qk=h_qk, h_v=h_v, init_std=0.02, seed=21)
    check(synth.make_prefill(cfg), "bf16")


def _sequence(inp, cu, n):
    """The inputs of sequence n alone (tokens [cu[n], cu[n+1])), as a one-sequence workload."""
    s0, s1 = int(cu[n]), int(cu[n + 1])
    one = dict(inp)
    for key in ("x_q", "x_k", "x_v", "z", "a", "b"):
        one[key] = inp[key][s0:s1]
    one["cu_seqlens"] = np.array([0, s1 - s0], dtype=np.int32)
    one["init_state"] = None if inp["init_state"] is None else inp["init_state"][n:n + 1]
    return one


def check_every_chain(cfg):
    """The whole GPU call, exactly as the benchmark launches it, against the
    oracle on every (sequence, value head) chain: all of `out` and all of
    `final_state`, element by element, one sequence at a time on every host core."""
    inp = synth.make_prefill(cfg)
    y, fs = run_gpu(inp, True)
    cu = inp["cu_seqlens"]
    py, pf = Parity("bf16", f"{cfg.name} out"), Parity("bf16", f"{cfg.name} final_state")
    for n in range(cfg.N):
        one = _sequence(inp, cu, n)
        r = ref.prefill(one, one["cu_seqlens"], one["init_state"], threads=os.cpu_count())
        py.add(y[cu[n]:cu[n + 1]], r["y"])
        pf.add(fs[n:n + 1], r["final_state"])
    assert py.count == y.size and pf.count == fs.size
    print(py.summary())
    print(pf.summary())
    py.check()
    pf.check()


@pytest.mark.slow
def test_full_single_4k():
    check_every_chain(synth.SINGLE_4K)


@pytest.mark.slow
def test_full_varlen_32k():
    check_every_chain(synth.VARLEN_32K)


@pytest.mark.slow
def test_full_long_128k():
    check_every_chain(synth.LONG_128K)


def test_deterministic_and_workspace_equivalent():
    """Bitwise-identical results run to run, with and without a caller workspace."""
    gdn = _gdn()
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(150, 77), h_qk=2, h_v=4, seed=11)
    inp = synth.make_prefill(cfg)
    y1, f1 = run_gpu(inp, True)
    y2, f2 = run_gpu(inp, True)
    nbytes = gdn.prefill_workspace_bytes(cfg.T, cfg.N, cfg.h_qk, cfg.h_v, 128, 128, True)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    y3, f3 = run_gpu(inp, True, workspace=ws)
    assert np.array_equal(y1, y2) and np.array_equal(f1, f2)
    assert np.array_equal(y1, y3) and np.array_equal(f1, f3)
    assert gdn.workspace_status(ws) == 0


def test_in_place_state_update():
    """final_state may be the init_state buffer."""
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(100, 64), h_qk=1, h_v=2, seed=12)
    inp = synth.make_prefill(cfg)
    y_a, f_a = run_gpu(inp, True)
    y_b, f_b = run_gpu(inp, True, in_place=True)
    assert np.array_equal(y_a, y_b) and np.array_equal(f_a, f_b)


def test_bad_cu_seqlens_sets_device_status():
    """Decreasing cu_seqlens is caught on the device and reported through the workspace."""
    gdn = _gdn()
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(64, 64), h_qk=1, h_v=2, seed=13)
    inp = synth.make_prefill(cfg)
    inp["cu_seqlens"] = np.array([0, 100, 64], dtype=np.int32)  # sequence 1 has negative length
    nbytes = gdn.prefill_workspace_bytes(cfg.T, cfg.N, 1, 2, 128, 128, True)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    run_gpu(inp, True, workspace=ws)
    assert gdn.workspace_status(ws) == 5
    assert gdn.workspace_status(ws) == 0  # reading clears it


@pytest.mark.parametrize("path", ["segmented", "carry", "fp32", "backward"])
def test_bad_cu_seqlens_sets_device_status_on_every_path(path):
    """The same decreasing cu_seqlens through the segment-parallel prefill,
    the carried-conv prefill (the chunk table and the conv-cache pass), the
    fp32 token-sequential prefill and the backward: each reports status 5
    through its workspace."""
    gdn = _gdn()
    fp32 = path == "fp32"
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(64, 64), h_qk=1, h_v=2, dtype="fp32" if fp32 else "bf16", seed=13)
    inp = synth.make_prefill(cfg)
    inp["cu_seqlens"] = np.array([0, 100, 64], dtype=np.int32)  # sequence 1 has negative length
    t = to_torch(inp, not fp32)
    args = (t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"], t["dt_bias"],
            t["norm_w"], t["cu_seqlens"])
    if path == "segmented":
        nbytes = gdn.prefill_segmented_workspace_bytes(cfg.T, cfg.N, 1, 2, 128, 128, 1)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        gdn.prefill_segmented(*args, seg_chunks=1, workspace=ws)
    elif path == "carry":
        ws = torch.zeros(gdn.prefill_workspace_bytes(cfg.T, cfg.N, 1, 2, 128, 128, True), dtype=torch.uint8,
                         device="cuda")
        _, _, fc = gdn.prefill_carry(*args, workspace=ws)
    elif path == "fp32":
        ws = torch.zeros(gdn.prefill_workspace_bytes(cfg.T, cfg.N, 1, 2, 128, 128, False), dtype=torch.uint8,
                         device="cuda")
        gdn.prefill(*args, workspace=ws)
    else:
        ws = torch.zeros(gdn.prefill_backward_workspace_bytes(cfg.T, cfg.N, 1, 2, 128, 128), dtype=torch.uint8,
                         device="cuda")
        dy = torch.randn((cfg.T, 2, 128), generator=torch.Generator().manual_seed(3)).to("cuda", torch.bfloat16)
        gdn.prefill_backward(*args, dy, workspace=ws)
    torch.cuda.synchronize()
    assert gdn.workspace_status(ws) == 5
    assert gdn.workspace_status(ws) == 0  # reading clears it
    if path == "carry":  # the invalid sequence's conv history is zeros; the valid one's is its last 3 inputs
        fcn = fc.float().cpu().numpy()
        assert not fcn[1].any()
        Cq = cfg.h_qk * cfg.d_k
        np.testing.assert_array_equal(fcn[0, :Cq], inp["x_q"][97:100].reshape(3, Cq).T)


def test_invalid_arguments_raise():
    gdn = _gdn()
    t = to_torch(synth.make_prefill(synth.scaled(synth.SINGLE_4K, lengths=(8,), h_qk=2, h_v=3)), True)
    with pytest.raises(gdn.GdnError) as e:   # h_v not a multiple of h_qk
        gdn.prefill(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                    t["dt_bias"], t["norm_w"], t["cu_seqlens"])
    assert e.value.status == 1


def test_kernel_trace_counts_each_launch():
    """With tracing on, each prefill records its three launches (chunk table,
    chunk prep, state pass) with positive device times; tracing off records nothing."""
    gdn = _gdn()
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(130, 64), h_qk=2, h_v=4, seed=14)
    inp = synth.make_prefill(cfg)
    gdn.trace_enable(True)
    gdn.trace_read()
    run_gpu(inp, True)
    run_gpu(inp, True)
    rec = gdn.trace_read()
    gdn.trace_enable(False)
    assert set(rec) == {"chunk_table_kernel", "chunk_prep_kernel", "state_kernel"}
    for name, (n, ms) in rec.items():
        assert n == 2 and ms > 0, (name, n, ms)
    run_gpu(inp, True)
    assert gdn.trace_read() == {}


def test_kernel_trace_of_the_other_paths():
    """The trace of a segment-parallel prefill (chunk table, prep, the two
    state passes, the segment table and scan), of an fp32 prefill (one record
    around its three launches) and of a backward (one record around the
    inputs, forward, norm and reverse kernels, one around the conv / norm
    prologue), each with positive device times."""
    gdn = _gdn()
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(300, 70), h_qk=2, h_v=4, seed=15)
    inp = synth.make_prefill(cfg)
    t = to_torch(inp, True)
    args = (t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"], t["dt_bias"],
            t["norm_w"], t["cu_seqlens"])
    gdn.trace_enable(True)
    try:
        gdn.trace_read()
        gdn.prefill_segmented(*args, seg_chunks=2)
        torch.cuda.synchronize()
        rec = gdn.trace_read()
        assert {k: v[0] for k, v in rec.items()} == {"chunk_table_kernel": 1, "chunk_prep_kernel": 1,
                                                      "state_kernel": 2, "seg_scan_kernels": 2}, rec
        assert all(v[1] > 0 for v in rec.values()), rec
        f = to_torch(synth.make_prefill(synth.scaled(cfg, dtype="fp32")), False)
        gdn.prefill(f["x_q"], f["x_k"], f["x_v"], f["a"], f["b"], f["z"], f["conv_w"], f["A_log"], f["dt_bias"],
                    f["norm_w"], f["cu_seqlens"])
        torch.cuda.synchronize()
        rec = gdn.trace_read()
        assert list(rec) == ["prefill_simt_kernel"] and rec["prefill_simt_kernel"][0] == 1, rec
        dy = torch.randn((cfg.T, cfg.h_v, cfg.d_v), generator=torch.Generator().manual_seed(4)).to("cuda", torch.bfloat16)
        gdn.prefill_backward(*args, dy)
        torch.cuda.synchronize()
        rec = gdn.trace_read()
        assert {k: v[0] for k, v in rec.items()} == {"bwd_state_kernels": 1, "bwd_prologue_kernel": 1}, rec
        assert all(v[1] > 0 for v in rec.values()), rec
    finally:
        gdn.trace_enable(False)


def _segment(inp, cu, bounds):
    """Tokens [bounds[n][0], bounds[n][1]) of every sequence n, as one packed workload."""
    idx = np.concatenate([np.arange(cu[n] + b0, cu[n] + b1) for n, (b0, b1) in enumerate(bounds)]).astype(np.int64)
    seg = {k_: (v_[idx] if k_ in ("x_q", "x_k", "x_v", "z", "a", "b") else v_) for k_, v_ in inp.items()}
    seg["cu_seqlens"] = np.concatenate([[0], np.cumsum([b1 - b0 for b0, b1 in bounds])]).astype(np.int32)
    return seg, idx


def _run_segments(inp, cuts, dtype, in_place=False):
    """gdn_prefill_carry over consecutive segments of every sequence, each call
    started from the previous call's final state and final conv history.
    Returns the outputs of the token indices, the last final state and conv."""
    gdn = _gdn()
    bf16 = dtype == "bf16"
    cu = inp["cu_seqlens"].astype(np.int64)
    state = None if inp["init_state"] is None else to_torch({"init_state": inp["init_state"]}, bf16)["init_state"]
    conv = None
    ys, idxs = [], []
    for s in range(len(cuts[0]) - 1):
        seg, idx = _segment(inp, cu, [(c[s], c[s + 1]) for c in cuts])
        t = to_torch(seg, bf16)
        kw = {"final_conv": conv} if (in_place and conv is not None) else {}
        out, state, conv = gdn.prefill_carry(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"],
                                             t["A_log"], t["dt_bias"], t["norm_w"], t["cu_seqlens"], state, conv,
                                             **kw)
        ys.append(out.float().cpu().numpy())
        idxs.append(idx)
    torch.cuda.synchronize()
    return np.concatenate(ys), np.concatenate(idxs), state.cpu().numpy(), conv.float().cpu().numpy()


def test_split_4096_token_sequence_into_two_calls():
    """One 4096-token sequence (16/32 heads, d = 128) as two gdn_prefill_carry
    calls, split inside a chunk; the second call starts from the first one's
    final state and conv history.  Every chain against the oracle's single run."""
    cfg = synth.SINGLE_4K
    inp = synth.make_prefill(cfg)
    y, idx, fs, conv = _run_segments(inp, [(0, 1500, 4096)], "bf16")
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"])
    parity(y, r["y"][idx], "bf16", "out")
    parity(fs, r["final_state"], "bf16", "final_state")
    np.testing.assert_array_equal(conv, ref.conv_cache_after_prefill(inp, inp["cu_seqlens"]))


@pytest.mark.parametrize("dtype,d,in_place", [("bf16", 128, False), ("bf16", 128, True), ("fp32", 32, False)],
                         ids=["tensor_core", "tensor_core_in_place", "fp32"])
def test_split_packed_sequences_into_short_segments(dtype, d, in_place):
    """Three packed sequences, each cut into four consecutive segments of its
    own lengths (empty, 1- and 2-token segments among them: the conv history of
    a token then reaches back over several calls).  The concatenated outputs,
    the last final state and the last conv history equal the oracle's single
    run (the conv history exactly: it is a byte move)."""
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(150, 64, 9), h_qk=2, h_v=4, d_k=d, d_v=d, dtype=dtype,
                       init_std=0.02, seed=41)
    inp = synth.make_prefill(cfg)
    cuts = [(0, 70, 71, 73, 150), (0, 0, 64, 64, 64), (0, 1, 2, 4, 9)]
    y, idx, fs, conv = _run_segments(inp, cuts, dtype, in_place=in_place)
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"])
    parity(y, r["y"][idx], dtype, "out")
    parity(fs, r["final_state"], dtype, "final_state")
    np.testing.assert_array_equal(conv, ref.conv_cache_after_prefill(inp, inp["cu_seqlens"]))


def run_segmented(inp, seg_chunks, *, in_place=False):
    gdn = _gdn()
    t = to_torch(inp, True)
    init = t.get("init_state")
    fs = init if (in_place and init is not None) else None
    out, fs = gdn.prefill_segmented(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                                    t["dt_bias"], t["norm_w"], t["cu_seqlens"], init, seg_chunks=seg_chunks,
                                    final_state=fs)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fs.cpu().numpy()


@pytest.mark.parametrize("lengths,seg_chunks,in_place", [
    ((1000,), 1, False),                   # every chunk a segment: 14 middle segments, a ragged last one
    ((1000,), 3, False),                   # 6 segments, the last one short
    ((1000,), 8, False),                   # 2 segments: no middle segment, so no transfer matrix
    ((1000,), 16, False),                  # one segment: the plain state pass
    ((300, 0, 1, 640, 65, 128), 2, False),  # packed: empty, 1-token, exact-segment and straddling sequences
    ((300, 0, 1, 640, 65, 128), 2, True),   # the same with the final state written over the initial one
], ids=["seg1", "seg3", "seg8", "seg16", "varlen_seg2", "varlen_seg2_in_place"])
def test_segmented_prefill(lengths, seg_chunks, in_place):
    """gdn_prefill_segmented against the oracle on every chain: each segment's
    start state comes out of the scan over the earlier segments' affine maps
    (B from a zero state, M from the identity), so every output and final
    state checks the transfer matrices and the scan as well."""
    cfg = synth.scaled(synth.SINGLE_4K, lengths=lengths, h_qk=2, h_v=4, init_std=0.02, seed=61)
    inp = synth.make_prefill(cfg)
    y, fs = run_segmented(inp, seg_chunks, in_place=in_place)
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"])
    parity(y, r["y"], "bf16", "out")
    parity(fs, r["final_state"], "bf16", "final_state")


def test_segmented_prefill_slow_decay():
    """Slow decay (alpha near 1): the earlier segments' states reach far, so a
    wrong transfer matrix or scan order shows in the later segments' outputs."""
    cfg = synth.scaled(synth.SINGLE_4K, lengths=(1500,), h_qk=1, h_v=2, init_std=0.02, seed=62)
    inp = synth.make_prefill(cfg)
    inp["dt_bias"][:] = -6.0
    y, fs = run_segmented(inp, 4)
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"])
    parity(y, r["y"], "bf16", "out")
    parity(fs, r["final_state"], "bf16", "final_state")


@pytest.mark.slow
@pytest.mark.parametrize("name,seg_chunks", [("prefill_T4096", 22), ("prefill_T16384_hv4", 16)])
def test_full_size_segmented(name, seg_chunks):
    """The 4096-token workload (16/32 heads) and the few-chain 16384-token one
    (2/4 heads) through gdn_prefill_segmented, with the segment lengths the
    benchmark's segmented lines use, every chain against the oracle."""
    cfg = {**synth.CONFIGS, synth.FEW_CHAINS_16K.name: synth.FEW_CHAINS_16K}[name]
    inp = synth.make_prefill(cfg)
    y, fs = run_segmented(inp, seg_chunks)
    r = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"], threads=os.cpu_count())
    parity(y, r["y"], "bf16", "out")
    parity(fs, r["final_state"], "bf16", "final_state")
