"""Exact sequential fp64 sums on one GB300 (sm_103a).

A thin ctypes binding over the C-ABI library ``libseqsum.so`` (declared in
``include/seqsum.h``).  The binding only marshals arguments: every step of the
sum runs in the library's CUDA kernels.  There is no CPU fallback -- if the
library cannot be loaded, every call raises.

PyTorch is used for device memory and streams only: the tensors passed in
must be CUDA tensors, and the work is enqueued on the current torch stream
unless a stream is given.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = ["seqsum_f64", "seqsum_f64_static", "seqsum_f64_batched", "seqsum_f64_batched_sized", "get_stats",
           "debug_set_plan", "debug_set_fault", "debug_counters", "release_workspace", "version", "lib", "lib_path",
           "seqsum_f64_strided", "SeqsumPlan",
           "SeqsumError"]

_lock = threading.Lock()
_lib = None


class SeqsumError(RuntimeError):
    pass


class _Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "tiles", "tiles_complex", "ranges_from_x", "lanes_raw", "lanes_raw2", "lanes_tie", "walk_batches",
        "walk_segments", "runs_rejected", "terms_dadd", "raw_rounds", "cy_walk_wait", "cy_walk_serial",
        "cy_walk_raw", "cy_tma_wait", "cy_plan", "cy_pfx_wait", "cy_run", "scan_windows", "scan_polls", "pfx_late", "ctas_alone", "tiles_redone",
        "t_stream_ns", "t_walk_tail_ns", "t_total_ns", "t_scan_ns", "t_units_ns")] + [
        ("device_status", ctypes.c_int32), ("device_error_bits", ctypes.c_int32),
        ("check_site", ctypes.c_int32), ("check_pad", ctypes.c_int32), ("check_value", ctypes.c_int64),
        ("timeout_site", ctypes.c_int32), ("timeout_pad", ctypes.c_int32), ("timeout_a", ctypes.c_int64),
        ("timeout_b", ctypes.c_int64)]


def lib():
    """Load libseqsum.so (building it first if needed).  Raises if it cannot."""
    global _lib
    with _lock:
        if _lib is None:
            checks = os.environ.get("SEQSUM_CHECKS", "") == "1"
            profile = os.environ.get("SEQSUM_PROFILE", "") == "1"
            path = _build.CHECK_LIB if checks else (_build.PROFILE_LIB if profile else _build.LIB)
            if not os.path.exists(path):
                path = _build.build(checks=checks, profile=profile)
            L = ctypes.CDLL(path)
            vp, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            L.seqsum_f64.argtypes = [vp, i64, d, vp, vp]
            L.seqsum_f64.restype = ctypes.c_int
            L.seqsum_f64_static.argtypes = [vp, i64, d, vp, vp]
            L.seqsum_f64_static.restype = ctypes.c_int
            L.seqsum_f64_batched.argtypes = [vp, vp, i32, vp, vp, vp]
            L.seqsum_f64_batched.restype = ctypes.c_int
            L.seqsum_f64_batched_sized.argtypes = [vp, i64, vp, i32, vp, vp, vp]
            L.seqsum_f64_batched_sized.restype = ctypes.c_int
            L.seqsum_f64_strided.argtypes = [vp, i64, i32, vp, vp, vp, vp]
            L.seqsum_f64_strided.restype = ctypes.c_int
            L.seqsum_plan_create.argtypes = [ctypes.POINTER(vp)]
            L.seqsum_plan_create.restype = ctypes.c_int
            L.seqsum_plan_destroy.argtypes = [vp]
            L.seqsum_plan_destroy.restype = None
            L.seqsum_f64_planned.argtypes = [vp, vp, i64, d, vp, vp]
            L.seqsum_f64_planned.restype = ctypes.c_int
            L.seqsum_get_stats.argtypes = [ctypes.POINTER(_Stats)]
            L.seqsum_get_stats.restype = ctypes.c_int
            L.seqsum_strerror.argtypes = [ctypes.c_int]
            L.seqsum_strerror.restype = ctypes.c_char_p
            L.seqsum_last_cuda_error.argtypes = []
            L.seqsum_last_cuda_error.restype = ctypes.c_int
            L.seqsum_release_workspace.argtypes = []
            L.seqsum_release_workspace.restype = None
            L.seqsum_debug_set_plan.argtypes = [ctypes.c_int]
            L.seqsum_debug_set_plan.restype = ctypes.c_int
            L.seqsum_debug_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int]
            L.seqsum_debug_read.restype = ctypes.c_int
            L.seqsum_debug_counters.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int]
            L.seqsum_debug_counters.restype = ctypes.c_int
            L.seqsum_debug_set_fault.argtypes = [ctypes.c_int, i64, i64]
            L.seqsum_debug_set_fault.restype = ctypes.c_int
            L.seqsum_version.argtypes = []
            L.seqsum_version.restype = ctypes.c_char_p
            L._path = path
            _lib = L
        return _lib


def lib_path() -> str:
    """The file of the loaded library (the plain, self-checking or profiling build)."""
    return lib()._path


def _check(rc: int):
    if rc != 0:
        L = lib()
        raise SeqsumError(f"seqsum: {L.seqsum_strerror(rc).decode()} (code {rc}, "
                          f"cuda error {L.seqsum_last_cuda_error()})")


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev_f64(t, name):
    import torch
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float64 and t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous CUDA float64 tensor")
    return t


def seqsum_f64(x, s0: float = 0.0, out=None, stream=None):
    """out[0] = s0 + x[0] + ... + x[n-1], added in index order, exactly as the
    CPU loop rounds each add.  Returns `out` (a 1-element CUDA float64 tensor);
    the value is ready once `stream` reaches it."""
    import torch
    x = _dev_f64(x, "x").reshape(-1)
    if out is None:
        out = torch.empty(1, dtype=torch.float64, device=x.device)
    _dev_f64(out, "out")
    with torch.cuda.device(x.device):
        _check(lib().seqsum_f64(ctypes.c_void_p(x.data_ptr()), x.numel(), float(s0),
                                ctypes.c_void_p(out.data_ptr()), _stream_handle(stream)))
    return out


class SeqsumPlan:
    """A plan kept from one frame to the next (seqsum_plan_create /
    seqsum_f64_planned / seqsum_plan_destroy).  ``plan(x, s0)`` returns the
    same bits as seqsum_f64(x, s0); after the first frame it reads x once and
    forms again only the tiles whose binades the new prefix moved."""

    def __init__(self):
        h = ctypes.c_void_p()
        _check(lib().seqsum_plan_create(ctypes.byref(h)))
        self._h = h

    def __call__(self, x, s0: float = 0.0, out=None, stream=None):
        import torch
        if self._h is None:
            raise SeqsumError("seqsum: the plan was closed")
        x = _dev_f64(x, "x").reshape(-1)
        if out is None:
            out = torch.empty(1, dtype=torch.float64, device=x.device)
        _dev_f64(out, "out")
        with torch.cuda.device(x.device):
            _check(lib().seqsum_f64_planned(self._h, ctypes.c_void_p(x.data_ptr()), x.numel(), float(s0),
                                            ctypes.c_void_p(out.data_ptr()), _stream_handle(stream)))
        return out

    def close(self):
        if self._h is not None and _lib is not None:
            _lib.seqsum_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


STATIC_MAX_TERMS = 1 << 21


def seqsum_f64_static(x, s0: float = 0.0, out=None, stream=None):
    """As seqsum_f64 for at most STATIC_MAX_TERMS terms, on the library's
    fixed-size device scratch: the call allocates nothing.  Calls that
    overlap in time race (they share the scratch)."""
    import torch
    x = _dev_f64(x, "x").reshape(-1)
    if out is None:
        out = torch.empty(1, dtype=torch.float64, device=x.device)
    _dev_f64(out, "out")
    with torch.cuda.device(x.device):
        _check(lib().seqsum_f64_static(ctypes.c_void_p(x.data_ptr()), x.numel(), float(s0),
                                       ctypes.c_void_p(out.data_ptr()), _stream_handle(stream)))
    return out


def seqsum_f64_strided(x, stride: int, s0s=None, outs=None, means=None, stream=None):
    """stride interleaved sums: outs[k] = s0s[k] + x[k] + x[k + stride] + ...
    in index order; means (a float32 tensor, or True to allocate one) gets
    float(outs[k] / n).  Returns outs, or (outs, means) when means is given."""
    import torch
    x = _dev_f64(x, "x").reshape(-1)
    stride = int(stride)
    if stride < 1 or x.numel() % stride:
        raise ValueError("x must hold a whole number of interleaved rows of `stride` terms")
    n = x.numel() // stride
    if s0s is None:
        s0s = torch.zeros(stride, dtype=torch.float64, device=x.device)
    _dev_f64(s0s, "s0s")
    if outs is None:
        outs = torch.empty(stride, dtype=torch.float64, device=x.device)
    _dev_f64(outs, "outs")
    m = None
    if means is True:
        m = torch.empty(stride, dtype=torch.float32, device=x.device)
    elif means is not None:
        m = means
        if not (m.is_cuda and m.dtype == torch.float32 and m.is_contiguous() and m.numel() >= stride):
            raise TypeError("means must be a contiguous CUDA float32 tensor of stride entries")
    with torch.cuda.device(x.device):
        _check(lib().seqsum_f64_strided(ctypes.c_void_p(x.data_ptr()), n, stride, ctypes.c_void_p(s0s.data_ptr()),
                                        ctypes.c_void_p(outs.data_ptr()),
                                        ctypes.c_void_p(m.data_ptr() if m is not None else 0),
                                        _stream_handle(stream)))
    return (outs, m) if m is not None else outs


def seqsum_f64_batched(x, offsets, s0s, outs=None, stream=None):
    """outs[k] = s0s[k] + x[offsets[k]] + ... + x[offsets[k+1]-1] for every k.
    Reads offsets[0] and offsets[-1] back once to size the workspace."""
    import torch
    x = _dev_f64(x, "x").reshape(-1)
    if not (offsets.is_cuda and offsets.dtype == torch.int64 and offsets.is_contiguous()):
        raise TypeError("offsets must be a contiguous CUDA int64 tensor")
    nsums = offsets.numel() - 1
    _dev_f64(s0s, "s0s")
    if outs is None:
        outs = torch.empty(max(nsums, 0), dtype=torch.float64, device=x.device)
    _dev_f64(outs, "outs")
    with torch.cuda.device(x.device):
        _check(lib().seqsum_f64_batched(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(offsets.data_ptr()),
                                        nsums, ctypes.c_void_p(s0s.data_ptr()),
                                        ctypes.c_void_p(outs.data_ptr()), _stream_handle(stream)))
    return outs


def seqsum_f64_batched_sized(x, offsets, s0s, outs=None, stream=None, x_len=None):
    """As seqsum_f64_batched, without any host wait: x_len (default x.numel())
    bounds every offset."""
    import torch
    x = _dev_f64(x, "x").reshape(-1)
    if not (offsets.is_cuda and offsets.dtype == torch.int64 and offsets.is_contiguous()):
        raise TypeError("offsets must be a contiguous CUDA int64 tensor")
    nsums = offsets.numel() - 1
    _dev_f64(s0s, "s0s")
    if outs is None:
        outs = torch.empty(max(nsums, 0), dtype=torch.float64, device=x.device)
    _dev_f64(outs, "outs")
    n = x.numel() if x_len is None else int(x_len)
    with torch.cuda.device(x.device):
        _check(lib().seqsum_f64_batched_sized(ctypes.c_void_p(x.data_ptr()), n,
                                              ctypes.c_void_p(offsets.data_ptr()), nsums,
                                              ctypes.c_void_p(s0s.data_ptr()),
                                              ctypes.c_void_p(outs.data_ptr()), _stream_handle(stream)))
    return outs


def get_stats() -> dict:
    """Device counters of the calls since the last get_stats() (waits)."""
    st = _Stats()
    _check(lib().seqsum_get_stats(ctypes.byref(st)))
    return {name: getattr(st, name) for name, _ in _Stats._fields_}


def debug_set_plan(mode: int) -> int:
    """Force the plan of later calls (tests only); returns the old mode."""
    return lib().seqsum_debug_set_plan(int(mode))


def debug_read(n: int = 64) -> list:
    """Diagnostic words recorded by a self-checking build (tests only)."""
    buf = (ctypes.c_ulonglong * n)()
    _check(lib().seqsum_debug_read(buf, n))
    return list(buf)


def debug_set_fault(mode: int, arg: int = 0, wait_ns: int = 0) -> None:
    """Test hook for the bounded device waits: mode 1 withholds the header of
    tile `arg` in later calls; wait_ns > 0 shortens every wait (0: 2 s)."""
    _check(lib().seqsum_debug_set_fault(int(mode), int(arg), int(wait_ns)))


_COUNTER_NAMES = ["ticket", "role", "exit", "sum_ticket", "err", "epoch", "ntiles", "skip", "check_site",
                  "check_lo", "check_hi", "timeout_site", "timeout_a", "timeout_b", "walk_sm", "scan_sm",
                  "redo_reserved", "scan_finished"]


def debug_counters() -> dict:
    """The device counters of the most recent call, read without waiting for
    it (diagnostics of a call that does not finish)."""
    n = len(_COUNTER_NAMES)
    buf = (ctypes.c_ulonglong * n)()
    _check(lib().seqsum_debug_counters(buf, n))
    return dict(zip(_COUNTER_NAMES, list(buf)))


def release_workspace():
    lib().seqsum_release_workspace()


def version() -> str:
    return lib().seqsum_version().decode()
