"""Failure detection without a GPU fault: every wait of the library's kernels
is bounded; a wait on a barrier that nothing signals gives up after its limit,
reports GDN_ERR_TIMEOUT through a device status word, and leaves the CUDA
context usable (the next prefill still matches the oracle)."""
import ctypes
import time

import pytest

from gateddeltanet_layer_gb300 import synth
from oracle import oracle as ref
from tests.helpers import parity, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports():
    import gateddeltanet_layer_gb300 as gdn
    lib = gdn.library()
    fn = lib.gdn_selftest_wait_timeout
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert fn(flag.data_ptr(), 20000, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert gdn.STATUS[int(flag.item())] == "GDN_ERR_TIMEOUT"
    assert waited >= 0.019
    # the context is intact: a prefill right after still computes the layer
    cfg = synth.scaled(synth.VARLEN_32K, lengths=(90, 40), h_qk=1, h_v=2, seed=41)
    inp = synth.make_prefill(cfg)
    t = to_torch(inp, True)
    out, fs = gdn.prefill(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                          t["dt_bias"], t["norm_w"], t["cu_seqlens"])
    torch.cuda.synchronize()
    r = ref.prefill(inp, inp["cu_seqlens"])
    parity(out.float().cpu().numpy(), r["y"], "bf16", "out after a timed-out wait")
