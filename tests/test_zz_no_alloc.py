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
import ctypes

import pytest

from gateddeltanet_layer_gb300 import synth
from tests.helpers import parity, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _inputs(cfg):
    t = to_torch(synth.make_prefill(cfg), cfg.dtype == "bf16")
    return (t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"], t["dt_bias"],
            t["norm_w"], t["cu_seqlens"], t.get("init_state"))


# Driver attribute of a memory pool: the most memory of the pool in use at once
# since the watermark was last reset to zero (CU_MEMPOOL_ATTR_USED_MEM_HIGH).
_USED_MEM_HIGH = 8


def _default_pool():
    """The device's default stream-ordered memory pool (where cudaMallocAsync
    takes memory), through the driver library, which every GPU process has."""
    cu = ctypes.CDLL("libcuda.so.1")
    dev = ctypes.c_int(0)
    assert cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
    pool = ctypes.c_void_p()
    assert cu.cuDeviceGetDefaultMemPool(ctypes.byref(pool), dev) == 0
    return cu, pool


def _pool_used_high(cu, pool) -> int:
    v = ctypes.c_uint64(0)
    assert cu.cuMemPoolGetAttribute(pool, _USED_MEM_HIGH, ctypes.byref(v)) == 0
    return v.value


def test_noalloc_matches_prefill_on_two_calls_in_a_row():
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    cases = [synth.scaled(synth.VARLEN_32K, lengths=(150, 0, 77, 64), h_qk=2, h_v=4, seed=31),
             synth.scaled(synth.SINGLE_4K, lengths=(333,), h_qk=1, h_v=2, seed=32)]
    args = [_inputs(cfg) for cfg in cases]
    refs = [gdn.prefill(*a) for a in args]          # the existing entry point, caller workspace
    torch.cuda.synchronize()
    outs = [(torch.empty_like(ro), torch.empty_like(rf)) for ro, rf in refs]
    # gdn_prefill takes its own workspace from the default pool; with every such
    # call complete, no pool memory is in use: reset the watermark to zero, so
    # any pool allocation made by the calls below would raise it again
    cu, pool = _default_pool()
    torch.cuda.synchronize()
    assert cu.cuMemPoolSetAttribute(pool, _USED_MEM_HIGH, ctypes.byref(ctypes.c_uint64(0))) == 0
    assert _pool_used_high(cu, pool) == 0
    got = []
    for a, (out, fs) in zip(args, outs):            # two gdn_prefill_noalloc calls back to back
        gdn.prefill_noalloc(*a, out=out, final_state=fs)
        got.append((out, fs))
    torch.cuda.synchronize()
    assert _pool_used_high(cu, pool) == 0, "gdn_prefill_noalloc took memory from the stream-ordered pool"
    # the control: gdn_prefill without a workspace does take pool memory, so the watermark sees it
    gdn.prefill(*args[0])
    torch.cuda.synchronize()
    assert _pool_used_high(cu, pool) > 0
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
