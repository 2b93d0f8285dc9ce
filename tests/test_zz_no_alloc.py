"""gdn_prefill_noalloc, the prefill for callers that cannot allocate device
memory (an engine whose memory planner owns all of HBM, a serving loop that
forbids allocation after warm-up, code inside another allocator's callback).

It takes its workspace from a fixed array in the library's device memory, so
two calls in a row share that array: the second call must not see anything
the first one left there.  Each call's output and final state are checked
against gdn_prefill (which uses a caller workspace) on the same inputs, within
the parity tolerances of the other tests.  This file is collected last so that
a failure here stops a `-x` run only after every other test has run.
"""
import pytest

from gateddeltanet_layer_gb300 import synth
from tests.helpers import parity, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _inputs(cfg):
    t = to_torch(synth.make_prefill(cfg), cfg.dtype == "bf16")
    return (t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"], t["dt_bias"],
            t["norm_w"], t["cu_seqlens"], t.get("init_state"))


def test_noalloc_matches_prefill_on_two_calls_in_a_row():
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    cases = [synth.scaled(synth.VARLEN_32K, lengths=(150, 0, 77, 64), h_qk=2, h_v=4, seed=31),
             synth.scaled(synth.SINGLE_4K, lengths=(333,), h_qk=1, h_v=2, seed=32)]
    args = [_inputs(cfg) for cfg in cases]
    refs = [gdn.prefill(*a) for a in args]          # the existing entry point, caller workspace
    torch.cuda.synchronize()
    got = []
    for a, (ro, rf) in zip(args, refs):             # two gdn_prefill_noalloc calls back to back
        out, fs = torch.empty_like(ro), torch.empty_like(rf)
        gdn.prefill_noalloc(*a, out=out, final_state=fs)
        got.append((out, fs))
    torch.cuda.synchronize()
    for cfg, (ro, rf), (out, fs) in zip(cases, refs, got):
        parity(out.float().cpu().numpy(), ro.float().cpu().numpy(), cfg.dtype, f"noalloc out {cfg.lengths}")
        parity(fs.cpu().numpy(), rf.cpu().numpy(), cfg.dtype, f"noalloc final_state {cfg.lengths}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    # find a sequence count whose workspace exceeds the fixed scratch, if the
    # workspace grows with the problem at all
    n = next((n for n in (1 << e for e in range(8, 21))
              if gdn.prefill_workspace_bytes(0, n, 16, 32, 128, 128) > gdn.NOALLOC_SCRATCH_BYTES), None)
    if n is None:
        pytest.skip("the prefill workspace does not grow with the problem size")
    empty = lambda *s, dt=torch.bfloat16: torch.empty(s, dtype=dt, device="cuda")  # noqa: E731
    cu = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
    f32 = torch.float32
    with pytest.raises(gdn.GdnError) as e:
        gdn.prefill_noalloc(empty(0, 16, 128), empty(0, 16, 128), empty(0, 32, 128), empty(0, 32), empty(0, 32),
                            empty(0, 32, 128), empty(2 * 16 * 128 + 32 * 128, 4, dt=f32), empty(32, dt=f32),
                            empty(32, dt=f32), empty(128, dt=f32), cu, out=empty(0, 32, 128))
    assert e.value.status == 3
