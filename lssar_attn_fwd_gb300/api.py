"""ctypes binding of liblssar_attn_fwd.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
only checks tensor metadata, takes raw device pointers and the current CUDA
stream from PyTorch and calls the C ABI declared in
``include/lssar_attn_fwd.h``.  There is no fallback: if the library is not
built, or a call fails, an exception is raised.
"""

import ctypes
import os

from .inputs import MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX, MODE_SOFTMAX_RW  # noqa: F401

_LIB = None

_EXPORTS = (
    "lssar_attn_fwd",
    "lssar_attn_fwd_simt",
    "lssar_attn_fwd_profiled",
    "lssar_attn_fwd_noalloc",
    "lssar_attn_fwd_heads_p",
    "lssar_attn_decode",
    "lssar_attn_fwd_train",
    "lssar_attn_bwd",
    "lssar_attn_bwd_simt",
    "lssar_attn_fwd_train_heads_p",
    "lssar_attn_bwd_heads_p",
    "lssar_selftest_stall",
    "lssar_schedule_plan",
    "lssar_decode_plan",
    "lssar_status_string",
    "lssar_device_error_word",
    "lssar_abi_version",
)


class LssarError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"lssar status {status}: {message}")
        self.status = status


def lib_path(debug=False):
    name = "liblssar_attn_fwd_debug.so" if debug else "liblssar_attn_fwd.so"
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", name)


_DEBUG_LIB = None


def load_debug_library():
    """Loads the debug-check build of the library (built with
    ``build(debug=True)``): the same C ABI, with device-side bounds checks
    that record codes 101-105 in its own device error word.  The functions of
    this module keep calling the default library; call the debug one through
    the returned handle (the argument declarations are the same)."""
    global _DEBUG_LIB
    if _DEBUG_LIB is None:
        _DEBUG_LIB = _open(lib_path(debug=True))
    return _DEBUG_LIB


def load_library():
    """Loads the shared library (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        _LIB = _open(lib_path())
    return _LIB


def _open(path):
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m lssar_attn_fwd_gb300.build` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    fwd_args = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 6 + [ctypes.c_void_p]
    for name in ("lssar_attn_fwd", "lssar_attn_fwd_simt", "lssar_attn_fwd_noalloc", "lssar_attn_decode"):
        fn = getattr(lib, name)
        fn.argtypes = fwd_args
        fn.restype = ctypes.c_int
    lib.lssar_attn_fwd_heads_p.argtypes = ([ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 +
                                           [ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_void_p])
    lib.lssar_attn_fwd_heads_p.restype = ctypes.c_int
    lib.lssar_attn_fwd_train.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_void_p]
    lib.lssar_attn_fwd_train.restype = ctypes.c_int
    lib.lssar_attn_fwd_train_heads_p.argtypes = ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 +
                                                 [ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_void_p])
    lib.lssar_attn_fwd_train_heads_p.restype = ctypes.c_int
    lib.lssar_attn_bwd_heads_p.argtypes = ([ctypes.c_void_p] * 8 + [ctypes.c_int] * 4 +
                                           [ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_void_p])
    lib.lssar_attn_bwd_heads_p.restype = ctypes.c_int
    for name in ("lssar_attn_bwd", "lssar_attn_bwd_simt"):
        fn = getattr(lib, name)
        fn.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int] * 6 + [ctypes.c_void_p]
        fn.restype = ctypes.c_int
    lib.lssar_attn_fwd_profiled.argtypes = fwd_args + [ctypes.c_void_p] * 3
    lib.lssar_attn_fwd_profiled.restype = ctypes.c_int
    lib.lssar_schedule_plan.argtypes = [ctypes.c_int] * 3 + [ctypes.POINTER(ctypes.c_int)] * 2
    lib.lssar_schedule_plan.restype = ctypes.c_int
    lib.lssar_decode_plan.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_int)] * 4
    lib.lssar_decode_plan.restype = ctypes.c_int
    lib.lssar_selftest_stall.argtypes = [ctypes.c_void_p]
    lib.lssar_selftest_stall.restype = ctypes.c_int
    lib.lssar_status_string.argtypes = [ctypes.c_int]
    lib.lssar_status_string.restype = ctypes.c_char_p
    lib.lssar_device_error_word.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.lssar_device_error_word.restype = ctypes.c_int
    lib.lssar_abi_version.argtypes = []
    lib.lssar_abi_version.restype = ctypes.c_int
    return lib


def status_string(status):
    return load_library().lssar_status_string(int(status)).decode()


def call_raw(name, q_ptr, k_ptr, v_ptr, out_ptr, B, H, L, d, p, mode, stream_handle):
    """Calls a forward entry point with raw integer pointers; returns the status."""
    fn = getattr(load_library(), name)
    return fn(ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
              ctypes.c_void_p(out_ptr), int(B), int(H), int(L), int(d), int(p), int(mode),
              ctypes.c_void_p(stream_handle))


def _check(status):
    if status != 0:
        raise LssarError(status, status_string(status))


def _forward(name, q, k, v, p, mode, out, stream):
    import torch

    for t in (q, k, v):
        if not isinstance(t, torch.Tensor):
            raise TypeError("q, k, v must be torch tensors")
        if t.device.type != "cuda" or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bfloat16 CUDA tensors")
        if t.dim() != 4 or t.shape != q.shape:
            raise ValueError("q, k, v must share one [B, H, L, d] shape")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    B, H, L, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    elif (out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous()
          or out.device != q.device):
        raise ValueError("out must be a contiguous bfloat16 tensor shaped like q on q's device")
    with torch.cuda.device(q.device):
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        _check(call_raw(name, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                        B, H, L, d, p, mode, handle))
    return out


def lssar_attn_fwd(q, k, v, p=3, mode=MODE_LSSAR, out=None, stream=None):
    """Causal LSSAR / LSSA / softmax attention forward on the tensor-core kernel.

    q, k, v: contiguous bf16 CUDA tensors [B, H, L, d] (d = 64 or 128).
    p: re-weighting exponent (modes 2-4).  mode: 0 softmax, 1 LSSA, 2 LSSAR,
    3 re-weighting on a softmax normaliser, 4 sigmoid + L1 + re-weighting.
    Runs asynchronously on ``stream`` (default: the current stream).
    """
    return _forward("lssar_attn_fwd", q, k, v, p, mode, out, stream)


def lssar_attn_fwd_simt(q, k, v, p=3, mode=MODE_LSSAR, out=None, stream=None):
    """Same operation on the plain CUDA-core kernel (cross-check only)."""
    return _forward("lssar_attn_fwd_simt", q, k, v, p, mode, out, stream)


def call_train(q_ptr, k_ptr, v_ptr, out_ptr, stats_ptr, B, H, L, d, p, mode, stream_handle):
    """Raw call of lssar_attn_fwd_train; returns the status."""
    return load_library().lssar_attn_fwd_train(
        *(ctypes.c_void_p(x) for x in (q_ptr, k_ptr, v_ptr, out_ptr, stats_ptr)),
        int(B), int(H), int(L), int(d), int(p), int(mode), ctypes.c_void_p(stream_handle))


def call_bwd(name, ptrs, B, H, L, d, p, mode, stream_handle):
    """Raw call of a backward entry point; ptrs = (q, k, v, dout, stats, dq,
    dk, dv) integer device pointers.  Returns the status."""
    return getattr(load_library(), name)(
        *(ctypes.c_void_p(x) for x in ptrs), int(B), int(H), int(L), int(d), int(p), int(mode),
        ctypes.c_void_p(stream_handle))


def _check_like(q, *ts):
    import torch
    for t in ts:
        if (not isinstance(t, torch.Tensor) or t.shape != q.shape or t.dtype != torch.bfloat16
                or not t.is_contiguous() or t.device != q.device):
            raise ValueError("tensors must be contiguous bfloat16 CUDA tensors shaped like q")


def lssar_attn_fwd_train(q, k, v, p=3, mode=MODE_LSSAR, out=None, stats=None, stream=None):
    """Training forward: returns (out, stats), stats [B, H, L, 4] float32 row
    statistics {m, kappa, beta, W} for :func:`lssar_attn_bwd_simt`."""
    import torch
    if q.device.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _check_like(q, q, k, v)
    B, H, L, d = q.shape
    out = torch.empty_like(q) if out is None else out
    _check_like(q, out)
    if stats is None:
        stats = torch.empty((B, H, L, 4), dtype=torch.float32, device=q.device)
    elif stats.shape != (B, H, L, 4) or stats.dtype != torch.float32 or not stats.is_contiguous():
        raise ValueError("stats must be a contiguous float32 [B, H, L, 4] tensor")
    with torch.cuda.device(q.device):
        s = torch.cuda.current_stream(q.device) if stream is None else stream
        _check(call_train(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), stats.data_ptr(),
                          B, H, L, d, p, mode, s.cuda_stream))
    return out, stats


def _backward(name, q, k, v, dout, stats, p, mode, stream):
    import torch
    if q.device.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _check_like(q, q, k, v, dout)
    B, H, L, d = q.shape
    if stats.shape != (B, H, L, 4) or stats.dtype != torch.float32 or not stats.is_contiguous():
        raise ValueError("stats must be the float32 [B, H, L, 4] tensor of lssar_attn_fwd_train")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    with torch.cuda.device(q.device):
        s = torch.cuda.current_stream(q.device) if stream is None else stream
        ptrs = tuple(t.data_ptr() for t in (q, k, v, dout, stats, dq, dk, dv))
        _check(call_bwd(name, ptrs, B, H, L, d, p, mode, s.cuda_stream))
    return dq, dk, dv


def lssar_attn_bwd(q, k, v, dout, stats, p=3, mode=MODE_LSSAR, stream=None):
    """Gradients (dq, dk, dv) of sum(dout * out) on the tensor-core backward,
    from the row statistics of :func:`lssar_attn_fwd_train` (same q, k, v, p,
    mode).  Runs asynchronously on ``stream`` (default: the current stream)."""
    return _backward("lssar_attn_bwd", q, k, v, dout, stats, p, mode, stream)


def lssar_attn_bwd_simt(q, k, v, dout, stats, p=3, mode=MODE_LSSAR, stream=None):
    """Gradients (dq, dk, dv) of sum(dout * out) on the plain CUDA-core
    backward (cross-check path), from the row statistics of
    :func:`lssar_attn_fwd_train`."""
    return _backward("lssar_attn_bwd_simt", q, k, v, dout, stats, p, mode, stream)


def call_heads_p(q_ptr, k_ptr, v_ptr, out_ptr, B, H, L, d, p_per_head, mode, stream_handle):
    """Raw call of lssar_attn_fwd_heads_p; returns the status."""
    arr = (ctypes.c_int * max(1, len(p_per_head)))(*[int(x) for x in p_per_head])
    ptr = arr if len(p_per_head) else None
    return load_library().lssar_attn_fwd_heads_p(
        ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
        ctypes.c_void_p(out_ptr), int(B), int(H), int(L), int(d), ptr, int(mode),
        ctypes.c_void_p(stream_handle))


def lssar_attn_fwd_heads_p(q, k, v, p_per_head, mode=MODE_LSSAR, out=None, stream=None):
    """Re-weighting modes with one exponent per head (p_per_head: H ints)."""
    import torch
    B, H, L, d = q.shape
    if len(p_per_head) != H:
        raise ValueError("p_per_head must hold one exponent per head")
    if out is None:
        out = torch.empty_like(q)
    with torch.cuda.device(q.device):
        s = torch.cuda.current_stream(q.device) if stream is None else stream
        _check(call_heads_p(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            B, H, L, d, p_per_head, mode, s.cuda_stream))
    return out


def _int_array(values):
    arr = (ctypes.c_int * max(1, len(values)))(*[int(x) for x in values])
    return arr if len(values) else None


def call_train_heads_p(q_ptr, k_ptr, v_ptr, out_ptr, stats_ptr, B, H, L, d, p_per_head, mode, stream_handle):
    """Raw call of lssar_attn_fwd_train_heads_p; returns the status."""
    return load_library().lssar_attn_fwd_train_heads_p(
        *(ctypes.c_void_p(x) for x in (q_ptr, k_ptr, v_ptr, out_ptr, stats_ptr)),
        int(B), int(H), int(L), int(d), _int_array(p_per_head), int(mode), ctypes.c_void_p(stream_handle))


def call_bwd_heads_p(ptrs, B, H, L, d, p_per_head, mode, stream_handle):
    """Raw call of lssar_attn_bwd_heads_p; ptrs as for :func:`call_bwd`."""
    return load_library().lssar_attn_bwd_heads_p(
        *(ctypes.c_void_p(x) for x in ptrs), int(B), int(H), int(L), int(d), _int_array(p_per_head),
        int(mode), ctypes.c_void_p(stream_handle))


def lssar_attn_fwd_train_heads_p(q, k, v, p_per_head, mode=MODE_LSSAR, stream=None):
    """Training forward with one re-weighting exponent per head: returns
    (out, stats) for :func:`lssar_attn_bwd_heads_p` (same p_per_head)."""
    import torch
    if q.device.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _check_like(q, q, k, v)
    B, H, L, d = q.shape
    if len(p_per_head) != H:
        raise ValueError("p_per_head must hold one exponent per head")
    out = torch.empty_like(q)
    stats = torch.empty((B, H, L, 4), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        s = torch.cuda.current_stream(q.device) if stream is None else stream
        _check(call_train_heads_p(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), stats.data_ptr(),
                                  B, H, L, d, p_per_head, mode, s.cuda_stream))
    return out, stats


def lssar_attn_bwd_heads_p(q, k, v, dout, stats, p_per_head, mode=MODE_LSSAR, stream=None):
    """Tensor-core backward with one re-weighting exponent per head, from the
    statistics of :func:`lssar_attn_fwd_train_heads_p`."""
    import torch
    if q.device.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    _check_like(q, q, k, v, dout)
    B, H, L, d = q.shape
    if len(p_per_head) != H:
        raise ValueError("p_per_head must hold one exponent per head")
    if stats.shape != (B, H, L, 4) or stats.dtype != torch.float32 or not stats.is_contiguous():
        raise ValueError("stats must be the float32 [B, H, L, 4] tensor of lssar_attn_fwd_train_heads_p")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    with torch.cuda.device(q.device):
        s = torch.cuda.current_stream(q.device) if stream is None else stream
        ptrs = tuple(t.data_ptr() for t in (q, k, v, dout, stats, dq, dk, dv))
        _check(call_bwd_heads_p(ptrs, B, H, L, d, p_per_head, mode, s.cuda_stream))
    return dq, dk, dv


def lssar_attn_decode(q, k_cache, v_cache, p=3, mode=MODE_LSSAR, out=None, stream=None):
    """One new query row per head (position L) against a K/V cache.

    q: [B, H, d] bf16; k_cache, v_cache: [B, H, L, d] bf16 (contiguous, CUDA).
    Returns out [B, H, d] bf16, equal to row L of the full causal forward.
    """
    import torch
    for t in (q, k_cache, v_cache):
        if t.device.type != "cuda" or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k_cache, v_cache must be contiguous bfloat16 CUDA tensors")
    B, H, L, d = k_cache.shape
    if v_cache.shape != k_cache.shape or tuple(q.shape) != (B, H, d):
        raise ValueError("shapes must be q [B, H, d] and caches [B, H, L, d]")
    if out is None:
        out = torch.empty_like(q)
    with torch.cuda.device(q.device):
        s = torch.cuda.current_stream(q.device) if stream is None else stream
        _check(call_raw("lssar_attn_decode", q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                        out.data_ptr(), B, H, L, d, p, mode, s.cuda_stream))
    return out


def lssar_attn_fwd_profiled(q, k, v, p, mode, out, stream, ev_start, ev_main, ev_end):
    """The tensor-core forward recording caller-owned torch.cuda.Events around
    the prologue and the attention kernel (each event must have been recorded
    once before, so that its CUDA handle exists; None skips that event)."""
    B, H, L, d = q.shape
    handle = lambda e: ctypes.c_void_p(None if e is None else e.cuda_event)  # noqa: E731
    status = load_library().lssar_attn_fwd_profiled(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), B, H, L, d, int(p), int(mode),
        ctypes.c_void_p(stream.cuda_stream), handle(ev_start), handle(ev_main), handle(ev_end))
    _check(status)
    return out


def decode_plan(B, H, L, d):
    """Launch plan of lssar_attn_decode for these sizes on the current device:
    dict(path=0 cluster | 1 cooperative | 2 three launches, launches,
    chunks, chunk_rows)."""
    vals = [ctypes.c_int(0) for _ in range(4)]
    _check(load_library().lssar_decode_plan(B, H, L, d, *(ctypes.byref(v) for v in vals)))
    return dict(zip(("path", "launches", "chunks", "chunk_rows"), (v.value for v in vals)))


def selftest_stall():
    """Test only: launches a decode step whose copies are withheld, so that its
    bounded waits give up (about 2 s); read the code with device_error_word()."""
    import torch
    _check(load_library().lssar_selftest_stall(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))


def device_error_word():
    """Reads and clears the device error word (synchronises the device)."""
    w = ctypes.c_uint(0)
    _check(load_library().lssar_device_error_word(ctypes.byref(w)))
    return w.value
