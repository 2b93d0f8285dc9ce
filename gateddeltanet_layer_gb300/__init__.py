"""GatedDeltaNet layer on GB300: thin Python binding of the C-ABI library.

Every step of the layer runs in the CUDA kernels of ``libgdn.so``; this module
only marshals torch tensors (device memory) and the current CUDA stream into
the C entry points of ``include/gdn.h`` under the same names.  There is no
Python or CPU implementation of the layer here: if ``libgdn.so`` is missing or
fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["prefill", "prefill_carry", "prefill_segmented", "prefill_segmented_workspace_bytes", "prefill_backward",
           "prefill_backward_workspace_bytes", "decode_step", "decode_step_slots", "conv_cache_from_prefill",
           "prefill_workspace_bytes", "workspace_status", "library", "GdnError", "STATUS", "prefill_noalloc", "NOALLOC_SCRATCH_BYTES",
           "trace_enable", "trace_read"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_BF16, GDN_FP32 = 0, 1
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_WORKSPACE",
          4: "GDN_ERR_CUDA", 5: "GDN_ERR_DEVICE_CHECK", 6: "GDN_ERR_TIMEOUT"}


class GdnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_seqs", ctypes.c_int32), ("h_qk", ctypes.c_int32),
                ("h_v", ctypes.c_int32), ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("io_dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p


def library() -> ctypes.CDLL:
    """Load libgdn.so (built by ``gateddeltanet_layer_gb300.build.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is not built: run `python -m gateddeltanet_layer_gb300.build` "
                                  "(nvcc, sm_103a); there is no fallback implementation")
            lib = ctypes.CDLL(LIB_PATH)
            dp = ctypes.POINTER(Dims)
            lib.gdn_prefill_workspace_bytes.argtypes = [dp]
            lib.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
            lib.gdn_prefill.argtypes = [dp] + [_vp] * 15 + [ctypes.c_size_t, _vp]
            lib.gdn_prefill.restype = ctypes.c_int
            lib.gdn_prefill_carry.argtypes = [dp] + [_vp] * 17 + [ctypes.c_size_t, _vp]
            lib.gdn_prefill_carry.restype = ctypes.c_int
            lib.gdn_prefill_segmented_workspace_bytes.argtypes = [dp, ctypes.c_int]
            lib.gdn_prefill_segmented_workspace_bytes.restype = ctypes.c_size_t
            lib.gdn_prefill_segmented.argtypes = [dp] + [_vp] * 14 + [ctypes.c_int, _vp, ctypes.c_size_t, _vp]
            lib.gdn_prefill_segmented.restype = ctypes.c_int
            lib.gdn_prefill_backward_workspace_bytes.argtypes = [dp]
            lib.gdn_prefill_backward_workspace_bytes.restype = ctypes.c_size_t
            lib.gdn_prefill_backward.argtypes = [dp] + [_vp] * 26 + [ctypes.c_size_t, _vp]
            lib.gdn_prefill_backward.restype = ctypes.c_int
            lib.gdn_decode_step.argtypes = [dp] + [_vp] * 14
            lib.gdn_decode_step.restype = ctypes.c_int
            lib.gdn_workspace_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int)]
            lib.gdn_workspace_status.restype = ctypes.c_int
            lib.gdn_status_string.argtypes = [ctypes.c_int]
            lib.gdn_status_string.restype = ctypes.c_char_p
            lib.gdn_decode_step_slots.argtypes = [dp] + [_vp] * 13 + [ctypes.c_int] + [_vp] * 3
            lib.gdn_decode_step_slots.restype = ctypes.c_int
            lib.gdn_conv_cache_from_prefill.argtypes = [dp] + [_vp] * 6
            lib.gdn_conv_cache_from_prefill.restype = ctypes.c_int
            lib.gdn_trace_enable.argtypes = [ctypes.c_int]
            lib.gdn_trace_enable.restype = ctypes.c_int
            lib.gdn_trace_read.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_double)]
            lib.gdn_trace_read.restype = ctypes.c_int
            lib.gdn_trace_kernel_name.argtypes = [ctypes.c_int]
            lib.gdn_trace_kernel_name.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _check(status: int, what: str):
    if status != 0:
        msg = library().gdn_status_string(status).decode()
        raise GdnError(status, f"{what}: {msg}")


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    torch = _torch()
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _io_dtype(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_FP32
    raise TypeError(f"unsupported stream dtype {t.dtype} (bf16 or fp32)")


def _req(t, name, dtype=None, cuda=True):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def dims_of(q, v, num_seqs: int) -> Dims:
    T, h_qk, d_k = q.shape
    _, h_v, d_v = v.shape
    return Dims(T, num_seqs, h_qk, h_v, d_k, d_v, _io_dtype(q))


def prefill_workspace_bytes(T: int, N: int, h_qk: int, h_v: int, d_k: int, d_v: int, bf16: bool = True) -> int:
    d = Dims(T, N, h_qk, h_v, d_k, d_v, GDN_BF16 if bf16 else GDN_FP32)
    return int(library().gdn_prefill_workspace_bytes(ctypes.byref(d)))


def prefill(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state=None, *,
            out=None, final_state=None, return_final_state=True, workspace=None, stream=None):
    """``gdn_prefill``: the layer over packed sequences.

    q, k [T, h_qk, d_k]; v, z [T, h_v, d_v]; a, b [T, h_v] (bf16 or fp32, one
    dtype); conv_w [Cc, 4], A_log, dt_bias [h_v], norm_w [d_v] fp32;
    cu_seqlens int32 [N+1]; init_state fp32 [N, h_v, d_k, d_v] or None.
    Returns (out [T, h_v, d_v], final_state or None).
    """
    return _prefill(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state, 0, out,
                    final_state, return_final_state, workspace, stream)


def prefill_segmented_workspace_bytes(T: int, N: int, h_qk: int, h_v: int, d_k: int, d_v: int,
                                      seg_chunks: int) -> int:
    d = Dims(T, N, h_qk, h_v, d_k, d_v, GDN_BF16)
    return int(library().gdn_prefill_segmented_workspace_bytes(ctypes.byref(d), int(seg_chunks)))


def prefill_segmented(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state=None, *,
                      seg_chunks: int, out=None, final_state=None, return_final_state=True, workspace=None,
                      stream=None):
    """``gdn_prefill_segmented``: ``prefill``'s results with every sequence cut
    into segments of ``seg_chunks`` chunks of 64 tokens, run in parallel and
    joined by a scan over the segments' affine state maps (more chains in
    flight for few long sequences).  bf16 streams with d_k = d_v = 128 only.
    Returns (out, final_state or None)."""
    return _prefill(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state, int(seg_chunks), out,
                    final_state, return_final_state, workspace, stream)


def _prefill(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state, seg, out, final_state,
             return_final_state, workspace, stream):
    torch = _torch()
    lib = library()
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("z", z)):
        _req(t, name, dt)
    for name, t in (("conv_w", conv_w), ("A_log", A_log), ("dt_bias", dt_bias), ("norm_w", norm_w)):
        _req(t, name, torch.float32)
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    N = cu_seqlens.numel() - 1
    d = dims_of(q, v, N)
    T, h_v, d_v = v.shape
    if init_state is not None:
        _req(init_state, "init_state", torch.float32)
    if out is None:
        out = torch.empty((T, h_v, d_v), dtype=dt, device=q.device)
    _req(out, "out", dt)
    if final_state is None and return_final_state:
        final_state = torch.empty((N, h_v, d.d_k, d_v), dtype=torch.float32, device=q.device)
    if final_state is not None:
        _req(final_state, "final_state", torch.float32)
    ws_bytes = 0
    if workspace is not None:
        _req(workspace, "workspace", torch.uint8)
        ws_bytes = workspace.numel()
    args = (ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z), _ptr(conv_w), _ptr(A_log),
            _ptr(dt_bias), _ptr(norm_w), _ptr(cu_seqlens), _ptr(init_state), _ptr(out), _ptr(final_state))
    tail = (_ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    if seg:
        _check(lib.gdn_prefill_segmented(*args, seg, *tail), "gdn_prefill_segmented")
    else:
        _check(lib.gdn_prefill(*args, *tail), "gdn_prefill")
    return out, final_state


def prefill_carry(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state=None, init_conv=None,
                  *, out=None, final_state=None, final_conv=None, workspace=None, stream=None):
    """``gdn_prefill_carry``: ``prefill`` that continues each sequence from a
    carried conv history ``init_conv`` ([N, Cc, 3], stream dtype, the raw inputs
    of the three tokens before the sequence, oldest first; None = zeros) as well
    as ``init_state``, and returns the conv history it leaves.  Consecutive
    segments of a sequence, each started from the previous one's final state
    and final conv history, give the result of one call over the whole
    sequence.  Returns (out, final_state, final_conv)."""
    torch = _torch()
    lib = library()
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("z", z)):
        _req(t, name, dt)
    for name, t in (("conv_w", conv_w), ("A_log", A_log), ("dt_bias", dt_bias), ("norm_w", norm_w)):
        _req(t, name, torch.float32)
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    N = cu_seqlens.numel() - 1
    d = dims_of(q, v, N)
    T, h_v, d_v = v.shape
    Cc = 2 * d.h_qk * d.d_k + h_v * d_v
    if init_state is not None:
        _req(init_state, "init_state", torch.float32)
    if init_conv is not None:
        _req(init_conv, "init_conv", dt)
        if tuple(init_conv.shape) != (N, Cc, 3):
            raise ValueError(f"init_conv must be [{N}, {Cc}, 3]")
    if out is None:
        out = torch.empty((T, h_v, d_v), dtype=dt, device=q.device)
    _req(out, "out", dt)
    if final_state is None:
        final_state = torch.empty((N, h_v, d.d_k, d_v), dtype=torch.float32, device=q.device)
    _req(final_state, "final_state", torch.float32)
    if final_conv is None:
        final_conv = torch.empty((N, Cc, 3), dtype=dt, device=q.device)
    _req(final_conv, "final_conv", dt)
    ws_bytes = 0
    if workspace is not None:
        _req(workspace, "workspace", torch.uint8)
        ws_bytes = workspace.numel()
    st = lib.gdn_prefill_carry(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z),
                               _ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w), _ptr(cu_seqlens),
                               _ptr(init_state), _ptr(init_conv), _ptr(out), _ptr(final_state), _ptr(final_conv),
                               _ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    _check(st, "gdn_prefill_carry")
    return out, final_state, final_conv


def prefill_backward_workspace_bytes(T: int, N: int, h_qk: int, h_v: int, d_k: int, d_v: int,
                                     bf16: bool = True) -> int:
    d = Dims(T, N, h_qk, h_v, d_k, d_v, GDN_BF16 if bf16 else GDN_FP32)
    return int(library().gdn_prefill_backward_workspace_bytes(ctypes.byref(d)))


def prefill_backward(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, dy, init_state=None,
                     dfinal_state=None, *, want_dinit_state=True, workspace=None, stream=None):
    """``gdn_prefill_backward``: gradients of sum(dy * y) + sum(dfinal_state *
    final_state) of the prefill with these inputs.  Returns a dict of fp32
    tensors named after the inputs: q, k, v, a, b, z, conv_w, A_log, dt_bias,
    norm_w and init_state (None unless want_dinit_state)."""
    torch = _torch()
    lib = library()
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("z", z), ("dy", dy)):
        _req(t, name, dt)
    for name, t in (("conv_w", conv_w), ("A_log", A_log), ("dt_bias", dt_bias), ("norm_w", norm_w)):
        _req(t, name, torch.float32)
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    for name, t in (("init_state", init_state), ("dfinal_state", dfinal_state)):
        if t is not None:
            _req(t, name, torch.float32)
    N = cu_seqlens.numel() - 1
    d = dims_of(q, v, N)
    f32 = dict(dtype=torch.float32, device=q.device)
    g = {"q": torch.empty(q.shape, **f32), "k": torch.empty(k.shape, **f32), "v": torch.empty(v.shape, **f32),
         "a": torch.empty(a.shape, **f32), "b": torch.empty(b.shape, **f32), "z": torch.empty(z.shape, **f32),
         "conv_w": torch.empty(conv_w.shape, **f32), "A_log": torch.empty(A_log.shape, **f32),
         "dt_bias": torch.empty(dt_bias.shape, **f32), "norm_w": torch.empty(norm_w.shape, **f32),
         "init_state": torch.empty((N, d.h_v, d.d_k, d.d_v), **f32) if want_dinit_state else None}
    ws_bytes = 0
    if workspace is not None:
        _req(workspace, "workspace", torch.uint8)
        ws_bytes = workspace.numel()
    st = lib.gdn_prefill_backward(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z),
                                  _ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w), _ptr(cu_seqlens),
                                  _ptr(init_state), _ptr(dy), _ptr(dfinal_state), _ptr(g["q"]), _ptr(g["k"]),
                                  _ptr(g["v"]), _ptr(g["a"]), _ptr(g["b"]), _ptr(g["z"]), _ptr(g["conv_w"]),
                                  _ptr(g["A_log"]), _ptr(g["dt_bias"]), _ptr(g["norm_w"]), _ptr(g["init_state"]),
                                  _ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    _check(st, "gdn_prefill_backward")
    return g


def decode_step(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, conv_state, state, *, out=None,
                stream=None):
    """``gdn_decode_step``: one token per sequence; updates ``state`` (fp32
    [B, h_v, d_k, d_v]) and ``conv_state`` ([B, Cc, 3], stream dtype) in place.
    Returns out [B, h_v, d_v]."""
    torch = _torch()
    lib = library()
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("z", z), ("conv_state", conv_state)):
        _req(t, name, dt)
    for name, t in (("conv_w", conv_w), ("A_log", A_log), ("dt_bias", dt_bias), ("norm_w", norm_w),
                    ("state", state)):
        _req(t, name, torch.float32)
    d = dims_of(q, v, 1)
    B, h_v, d_v = v.shape
    if out is None:
        out = torch.empty((B, h_v, d_v), dtype=dt, device=q.device)
    _req(out, "out", dt)
    st = lib.gdn_decode_step(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z),
                             _ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w), _ptr(conv_state),
                             _ptr(state), _ptr(out), _stream_handle(stream, q.device))
    _check(st, "gdn_decode_step")
    return out


def decode_step_slots(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, conv_state, state, slots, *, out=None,
                      status=None, stream=None):
    """``gdn_decode_step_slots``: one token per sequence against pools of conv
    caches ([P, Cc, 3]) and states (fp32 [P, h_v, d_k, d_v]); sequence b uses
    pool entry ``slots[b]`` (int32, device).  An entry outside [0, P) writes
    zeros for that sequence and sets ``status`` (int32 [1] device tensor, if
    given) to 5.  Returns out [B, h_v, d_v]."""
    torch = _torch()
    lib = library()
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("z", z), ("conv_state", conv_state)):
        _req(t, name, dt)
    for name, t in (("conv_w", conv_w), ("A_log", A_log), ("dt_bias", dt_bias), ("norm_w", norm_w),
                    ("state", state)):
        _req(t, name, torch.float32)
    _req(slots, "slots", torch.int32)
    if status is not None:
        _req(status, "status", torch.int32)
    d = dims_of(q, v, 1)
    B, h_v, d_v = v.shape
    if slots.numel() != B:
        raise ValueError("slots must hold one entry per sequence")
    if out is None:
        out = torch.empty((B, h_v, d_v), dtype=dt, device=q.device)
    _req(out, "out", dt)
    st = lib.gdn_decode_step_slots(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z),
                                   _ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w), _ptr(conv_state),
                                   _ptr(state), _ptr(slots), int(state.shape[0]), _ptr(out), _ptr(status),
                                   _stream_handle(stream, q.device))
    _check(st, "gdn_decode_step_slots")
    return out


def conv_cache_from_prefill(q, k, v, cu_seqlens, *, out=None, stream=None):
    """``gdn_conv_cache_from_prefill``: the decode conv cache [N, Cc, 3] (stream
    dtype) that the sequences of a prefill call leave: their last three raw
    q, k, v inputs per channel, oldest first, zeros before a sequence start."""
    torch = _torch()
    lib = library()
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v)):
        _req(t, name, dt)
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    N = cu_seqlens.numel() - 1
    d = dims_of(q, v, N)
    T, h_qk, d_k = q.shape
    _, h_v, d_v = v.shape
    Cc = 2 * h_qk * d_k + h_v * d_v
    if out is None:
        out = torch.empty((N, Cc, 3), dtype=dt, device=q.device)
    _req(out, "out", dt)
    _check(lib.gdn_conv_cache_from_prefill(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(out),
                                           _stream_handle(stream, q.device)), "gdn_conv_cache_from_prefill")
    return out


def workspace_status(workspace, stream=None) -> int:
    """Read and clear the device status word of a prefill workspace (synchronises the stream)."""
    lib = library()
    res = ctypes.c_int(0)
    _check(lib.gdn_workspace_status(_ptr(workspace), _stream_handle(stream, workspace.device),
                                    ctypes.byref(res)), "gdn_workspace_status")
    return res.value


# Number of kernel kinds the trace distinguishes (GDN_K_COUNT in include/gdn_trace.h).
TRACE_KINDS = 8


def trace_enable(on: bool = True) -> None:
    """Start (or stop) recording CUDA events around every kernel the library launches."""
    _check(library().gdn_trace_enable(1 if on else 0), "gdn_trace_enable")


def trace_read() -> dict:
    """Per kernel name: (launches, total device ms) recorded since the last read; clears the record."""
    lib = library()
    n = (ctypes.c_int * TRACE_KINDS)()
    ms = (ctypes.c_double * TRACE_KINDS)()
    _check(lib.gdn_trace_read(TRACE_KINDS, n, ms), "gdn_trace_read")
    return {lib.gdn_trace_kernel_name(k).decode(): (n[k], ms[k]) for k in range(TRACE_KINDS) if n[k]}


# Size of the library's fixed scratch array used by gdn_prefill_noalloc
# (GDN_NOALLOC_SCRATCH_BYTES in include/gdn.h).
NOALLOC_SCRATCH_BYTES = 8 << 20


def prefill_noalloc(q, k, v, a, b, z, conv_w, A_log, dt_bias, norm_w, cu_seqlens, init_state=None, *,
                    out=None, final_state=None, stream=None):
    """``gdn_prefill_noalloc``: the prefill for callers that cannot allocate
    device memory (an engine whose memory planner owns all of HBM, a serving
    loop that forbids allocation after warm-up, code running inside another
    allocator's callback).  The library takes its workspace from a fixed
    device array of NOALLOC_SCRATCH_BYTES instead of allocating one.  ``out``
    and ``final_state`` must be passed in (this wrapper does not create them
    either).  Calls that overlap on the GPU share that array and race: order
    them on one stream.  Returns (out, final_state)."""
    torch = _torch()
    lib = library()
    fn = lib.gdn_prefill_noalloc
    fn.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 15
    fn.restype = ctypes.c_int
    if out is None:
        raise ValueError("prefill_noalloc allocates nothing: pass `out`")
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("z", z), ("out", out)):
        _req(t, name, dt)
    for name, t in (("conv_w", conv_w), ("A_log", A_log), ("dt_bias", dt_bias), ("norm_w", norm_w)):
        _req(t, name, torch.float32)
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    for name, t in (("init_state", init_state), ("final_state", final_state)):
        if t is not None:
            _req(t, name, torch.float32)
    d = dims_of(q, v, cu_seqlens.numel() - 1)
    st = fn(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z), _ptr(conv_w), _ptr(A_log),
            _ptr(dt_bias), _ptr(norm_w), _ptr(cu_seqlens), _ptr(init_state), _ptr(out), _ptr(final_state),
            _stream_handle(stream, q.device))
    _check(st, "gdn_prefill_noalloc")
    return out, final_state
