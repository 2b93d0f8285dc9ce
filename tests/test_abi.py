"""The C-ABI library builds for sm_103a, loads, exports every entry point that
include/gdn.h declares, and rejects invalid arguments on the host before
touching the GPU (so these run without one)."""
import ctypes
import os
import re

import pytest

import gateddeltanet_layer_gb300 as gdn
from gateddeltanet_layer_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.library()


def declared_functions():
    """Every gdn_* function declared by a header under include/."""
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            src = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
            names |= set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("gdn_prefill", "gdn_decode_step", "gdn_prefill_workspace_bytes", "gdn_status_string",
                 "gdn_workspace_status"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in gdn.STATUS.items():
        assert lib.gdn_status_string(code).decode().startswith(name)
    assert lib.gdn_status_string(99) == b"GDN_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    assert gdn.prefill_workspace_bytes(4096, 1, 16, 32, 128, 128) >= 256
    assert gdn.prefill_workspace_bytes(64, 1, 2, 2, 16, 16, bf16=False) >= 256
    assert gdn.prefill_workspace_bytes(64, 1, 2, 3, 16, 16) == 0        # h_v % h_qk != 0
    assert gdn.prefill_workspace_bytes(64, 1, 2, 2, 24, 16) == 0        # unsupported head dim
    assert lib.gdn_prefill_workspace_bytes(None) == 0


def _call_prefill(lib, dims, ptr=1 << 20, ws=None, ws_bytes=0, cu=1 << 20):
    p = ctypes.c_void_p(ptr)
    return lib.gdn_prefill(None if dims is None else ctypes.byref(dims), p, p, p, p, p, p, p, p, p, p,
                           ctypes.c_void_p(cu), None, p, None, ws, ws_bytes, None)


def test_prefill_rejects_bad_arguments_without_a_gpu(lib):
    D = gdn.Dims
    assert _call_prefill(lib, None) == 1
    assert _call_prefill(lib, D(64, 1, 2, 3, 128, 128, 0)) == 1          # h_v % h_qk
    assert _call_prefill(lib, D(-1, 1, 2, 2, 128, 128, 0)) == 1          # negative T
    assert _call_prefill(lib, D(64, 0, 2, 2, 128, 128, 0)) == 1          # no sequences
    assert _call_prefill(lib, D(64, 1, 2, 2, 128, 128, 7)) == 1          # bad dtype
    assert _call_prefill(lib, D(64, 1, 2, 2, 96 + 8, 128, 0)) == 2       # unsupported d_k
    assert _call_prefill(lib, D(64, 1, 2, 2, 128, 128, 0), ptr=(1 << 20) + 2) == 1  # misaligned
    assert _call_prefill(lib, D(64, 1, 2, 2, 128, 128, 0), cu=0) == 1    # NULL cu_seqlens
    ws = ctypes.c_void_p(1 << 24)
    assert _call_prefill(lib, D(64, 1, 2, 2, 128, 128, 0), ws=ws, ws_bytes=8) == 3  # short workspace


def test_decode_rejects_bad_arguments_without_a_gpu(lib):
    D = gdn.Dims
    p = ctypes.c_void_p(1 << 20)
    args = [p] * 14
    assert lib.gdn_decode_step(ctypes.byref(D(4, 1, 2, 3, 128, 128, 0)), *args) == 1
    assert lib.gdn_decode_step(ctypes.byref(D(4, 1, 2, 2, 100, 128, 0)), *args) == 2
    bad = list(args)
    bad[11] = None  # state
    assert lib.gdn_decode_step(ctypes.byref(D(4, 1, 2, 2, 128, 128, 0)), *bad) == 1


def test_library_fails_loudly_when_missing(monkeypatch, tmp_path):
    """No fallback: a missing libgdn.so raises instead of computing anything."""
    monkeypatch.setattr(gdn, "LIB_PATH", str(tmp_path / "libgdn.so"))
    monkeypatch.setattr(gdn, "_lib", None)
    with pytest.raises(ImportError):
        gdn.library()


def test_trace_read_without_launches(lib):
    """The kernel trace reads back empty (and names its kernel kinds) without a GPU."""
    assert gdn.trace_read() == {}
    names = [lib.gdn_trace_kernel_name(k).decode() for k in range(gdn.TRACE_KINDS)]
    assert names == ["chunk_table_kernel", "chunk_prep_kernel", "state_kernel", "prefill_simt_kernel",
                     "decode_kernel", "bwd_state_kernels", "bwd_prologue_kernel", "seg_scan_kernels"]
    assert lib.gdn_trace_kernel_name(gdn.TRACE_KINDS) == b""
    assert lib.gdn_trace_read(0, None, None) == 1


def test_hand_off_calls_reject_bad_arguments_without_a_gpu(lib):
    D = gdn.Dims
    p = ctypes.c_void_p(1 << 20)
    d = ctypes.byref(D(64, 2, 2, 2, 128, 128, 0))
    assert lib.gdn_conv_cache_from_prefill(None, p, p, p, p, p, None) == 1
    assert lib.gdn_conv_cache_from_prefill(d, p, p, p, None, p, None) == 1       # no cu_seqlens
    assert lib.gdn_conv_cache_from_prefill(d, p, p, p, p, None, None) == 1       # no cache
    assert lib.gdn_conv_cache_from_prefill(ctypes.byref(D(64, 0, 2, 2, 128, 128, 0)), p, p, p, p, p, None) == 1
    args = [p] * 12
    dd = ctypes.byref(D(4, 1, 2, 2, 128, 128, 0))
    assert lib.gdn_decode_step_slots(dd, *args, p, 0, p, None, None) == 1        # slots without a pool size
    assert lib.gdn_decode_step_slots(ctypes.byref(D(4, 1, 2, 3, 128, 128, 0)), *args, p, 4, p, None, None) == 1


def test_timeout_selftest_rejects_bad_arguments_without_a_gpu(lib):
    fn = lib.gdn_selftest_wait_timeout
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert fn(None, 1000, None) == 1
    assert fn(ctypes.c_void_p(1 << 20), 0, None) == 1
    assert fn(ctypes.c_void_p(1 << 20), 2000000, None) == 1


def test_backward_and_carry_reject_bad_arguments_without_a_gpu(lib):
    """Host-side validation of gdn_prefill_backward and gdn_prefill_carry (and
    the binding's argument lists) without a launch."""
    D = gdn.Dims
    d = D(64, 1, 2, 2, 16, 16, gdn.GDN_FP32)
    null = [None] * 26
    assert lib.gdn_prefill_backward(ctypes.byref(d), *null, 0, None) == 1       # required pointers missing
    bad = D(64, 1, 2, 3, 16, 16, gdn.GDN_FP32)                                  # h_v % h_qk != 0
    assert lib.gdn_prefill_backward(ctypes.byref(bad), *null, 0, None) == 1
    assert lib.gdn_prefill_backward_workspace_bytes(ctypes.byref(d)) > 256
    assert lib.gdn_prefill_backward_workspace_bytes(ctypes.byref(bad)) == 0
    assert lib.gdn_prefill_carry(ctypes.byref(d), *([None] * 17), 0, None) == 1
    unsup = D(64, 1, 2, 2, 24, 16, gdn.GDN_FP32)                                # head dim not a multiple of 16
    assert lib.gdn_prefill_carry(ctypes.byref(unsup), *([None] * 17), 0, None) == 2


def test_segmented_prefill_rejects_bad_arguments_without_a_gpu(lib):
    """gdn_prefill_segmented: only the chunked tensor-core shapes, seg_chunks >= 1,
    required pointers; its workspace holds the plain prefill's and the segment
    buffers (three fp32 states per segment and value head)."""
    D = gdn.Dims
    tc = D(4096, 1, 4, 8, 128, 128, gdn.GDN_BF16)
    fp32 = D(4096, 1, 4, 8, 128, 128, gdn.GDN_FP32)
    null = [None] * 14
    assert lib.gdn_prefill_segmented(ctypes.byref(tc), *null, 8, None, 0, None) == 1      # pointers missing
    assert lib.gdn_prefill_segmented(ctypes.byref(tc), *null, 0, None, 0, None) == 1      # seg_chunks < 1
    assert lib.gdn_prefill_segmented(ctypes.byref(fp32), *null, 8, None, 0, None) == 2    # not a tensor-core shape
    assert lib.gdn_prefill_segmented_workspace_bytes(ctypes.byref(fp32), 8) == 0
    assert lib.gdn_prefill_segmented_workspace_bytes(ctypes.byref(tc), 0) == 0
    plain = lib.gdn_prefill_workspace_bytes(ctypes.byref(tc))
    segs = (4096 // 64 + 1) // 8 + 1 + 1                      # upper bound on the segments
    extra = lib.gdn_prefill_segmented_workspace_bytes(ctypes.byref(tc), 8) - plain
    assert 3 * segs * 8 * 128 * 128 * 4 <= extra < 3 * segs * 8 * 128 * 128 * 4 + 8192
