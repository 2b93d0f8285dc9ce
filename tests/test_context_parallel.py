"""Context-parallel prefill on the CPU: the hand-off protocol of
gateddeltanet_layer_gb300.context_parallel over `gloo` ranks, each rank's
compute done by the fp64 oracle through the semantics of gdn_prefill_carry
(the GPU kernels of that entry point are checked against the oracle in
tests/test_gpu_prefill.py).  The ranks' outputs and final states must equal the
oracle's single run over the whole batch."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_prefill_carry(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu, init_state, init_conv):
    """gdn_prefill_carry's results, computed by the oracle (fp32 state, stream dtype conv history)."""
    from oracle import oracle as ref
    inp = {"x_q": q.numpy(), "x_k": k.numpy(), "x_v": v.numpy(), "a": a.numpy(), "b": b.numpy(), "z": z.numpy(),
           "conv_w": conv_w.numpy(), "A_log": A_log.numpy(), "dt_bias": dt_bias.numpy(), "norm_w": norm_w.numpy()}
    cu_np = cu.numpy()
    st = None if init_state is None else init_state.numpy()
    conv = None if init_conv is None else init_conv.numpy()
    r = ref.prefill(inp, cu_np, st, init_conv=conv, threads=1)
    fc = ref.conv_cache_after_prefill(inp, cu_np, init_conv=conv)
    return (torch.from_numpy(r["y"]).to(q.dtype), torch.from_numpy(r["final_state"]).float(),
            torch.from_numpy(fc).to(q.dtype))


def _rank_main(rank, world, port, lengths, slices, out):
    sys.path.insert(0, ROOT)
    from gateddeltanet_layer_gb300 import context_parallel as cp
    from gateddeltanet_layer_gb300 import synth
    from oracle import oracle as ref
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = synth.scaled(synth.TINY, lengths=lengths, h_qk=1, h_v=2, d_k=16, d_v=16, init_std=0.02, seed=51)
        inp = synth.make_prefill(cfg)
        t0, t1 = slices[rank]
        sl = {key: torch.from_numpy(np.ascontiguousarray(inp[key][t0:t1])) for key in ("x_q", "x_k", "x_v", "a", "b",
                                                                                       "z")}
        par = {key: torch.from_numpy(inp[key]) for key in ("conv_w", "A_log", "dt_bias", "norm_w")}
        plan, y, fs, fc = cp.context_parallel_prefill(
            sl["x_q"], sl["x_k"], sl["x_v"], sl["a"], sl["b"], sl["z"], par["conv_w"], par["A_log"], par["dt_bias"],
            par["norm_w"], inp["cu_seqlens"], t0, t1, torch.from_numpy(inp["init_state"]),
            prefill_fn=_oracle_prefill_carry)
        full = ref.prefill(inp, inp["cu_seqlens"], inp["init_state"])
        y_err = float(np.max(np.abs(y.numpy() - full["y"][t0:t1]), initial=0.0))
        s_err = 0.0
        for i, n in enumerate(plan.seqs):
            if plan.ends_here[i]:
                s_err = max(s_err, float(np.max(np.abs(fs[i].numpy() - full["final_state"][n]))))
        out[rank] = (plan.seqs, plan.continues_in, plan.continues_out, y_err, s_err)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,lengths,slices", [
    (2, (37, 64, 9), [(0, 55), (55, 110)]),                   # the split falls inside the second sequence
    (3, (150, 10), [(0, 50), (50, 100), (100, 160)]),         # the first sequence spans all three ranks
    (2, (20, 3), [(0, 21), (21, 23)]),                        # the second rank holds a 2-token tail
], ids=["two_ranks", "three_ranks_one_long_sequence", "short_tail"])
def test_context_parallel_prefill_gloo(world, lengths, slices):
    with mp.Manager() as manager:
        out = manager.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), lengths, slices, out), nprocs=world,
                           start_method="spawn")
        got = dict(out)
    assert set(got) == set(range(world))
    for rank in range(world):
        seqs, cin, cout, y_err, s_err = got[rank]
        # the carried state crosses a boundary in fp32 (the library's state type)
        assert y_err < 1e-5 and s_err < 1e-6, (rank, y_err, s_err)
    assert got[0][1] is False and got[world - 1][2] is False
    for rank in range(1, world):
        assert got[rank][1] == got[rank - 1][2]  # a hand-off has a sender and a receiver


def test_plan_rank_edges():
    from gateddeltanet_layer_gb300.context_parallel import plan_rank
    cu = [0, 10, 10, 25, 40]
    p = plan_rank(cu, 0, 10)
    assert p.seqs == (0,) and p.local_cu == (0, 10) and not p.continues_in and not p.continues_out
    p = plan_rank(cu, 10, 30)                    # the empty sequence 1 starts at 10: it belongs here
    assert p.seqs == (1, 2, 3) and p.local_cu == (0, 0, 15, 20) and p.continues_out
    assert p.ends_here == (True, True, False)
    p = plan_rank(cu, 30, 40)
    assert p.seqs == (3,) and p.continues_in and not p.continues_out and p.local_cu == (0, 10)
    p = plan_rank([0, 5, 5], 5, 5)               # an empty sequence at the very end, on the last (empty) slice
    assert p.seqs == (1,) and p.local_cu == (0, 0)
    with pytest.raises(ValueError):
        plan_rank(cu, 0, 41)
