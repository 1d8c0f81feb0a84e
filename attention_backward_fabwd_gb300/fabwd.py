"""ctypes binding of libfabwd (include/fabwd.h): argument marshalling only.

Every function here has the name and argument order of the C entry point it wraps.  Pointers
are plain integers (device or host addresses); `stream` is a cudaStream_t as an integer (0 is
the legacy default stream).  The library must have been built (build.build()); loading fails
loudly otherwise, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

from . import build as _build

FABWD_OK, FABWD_ERR_NULLPTR, FABWD_ERR_INVALID, FABWD_ERR_UNSUPPORTED = 0, 1, 2, 3
FABWD_ERR_WORKSPACE, FABWD_ERR_CUDA, FABWD_ERR_TIMEOUT, FABWD_ERR_DEVICE = 4, 5, 6, 7
FABWD_BF16, FABWD_FP16 = 0, 1
FABWD_BSND, FABWD_TND, FABWD_BNSD = 0, 1, 2
FABWD_MASK_NONE, FABWD_MASK_CAUSAL, FABWD_MASK_BAND = 0, 1, 2
FABWD_DEV_TIMEOUT, FABWD_DEV_BAD_SEQLENS, FABWD_DEV_INTERNAL = 0x1, 0x2, 0x4
FABWD_DQ_AUTO, FABWD_DQ_ATOMIC, FABWD_DQ_SEPARATE = 0, 1, 2

HEADER = os.path.join(_build.ROOT, "include", "fabwd.h")


class fabwd_params(ctypes.Structure):
    """Mirror of the C struct fabwd_params (field order and types as in include/fabwd.h)."""

    _fields_ = [
        ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("B", ctypes.c_int64), ("S1", ctypes.c_int64), ("S2", ctypes.c_int64),
        ("N1", ctypes.c_int64), ("N2", ctypes.c_int64), ("D", ctypes.c_int64), ("Dv", ctypes.c_int64),
        ("T1", ctypes.c_int64), ("T2", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("dout", ctypes.c_void_p), ("attn_out", ctypes.c_void_p), ("softmax_lse", ctypes.c_void_p),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_kv", ctypes.c_void_p),
        ("softmax_scale", ctypes.c_double),
        ("mask_mode", ctypes.c_int32), ("dq_mode", ctypes.c_int32),
        ("win_left", ctypes.c_int64), ("win_right", ctypes.c_int64),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("seqused_q", ctypes.c_void_p), ("seqused_kv", ctypes.c_void_p), ("sinks", ctypes.c_void_p),
    ]


class FabwdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libfabwd.so (built in-tree).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libfabwd is not built ({_build.LIB} missing): run build.build() first")
        L = ctypes.CDLL(_build.LIB)
        P = ctypes.POINTER(fabwd_params)
        sz = ctypes.c_size_t
        L.fabwd_workspace_size.argtypes = [P, ctypes.POINTER(sz)]
        L.fabwd_workspace_layout.argtypes = [P, ctypes.POINTER(sz), ctypes.POINTER(sz), ctypes.POINTER(sz),
                                             ctypes.POINTER(ctypes.c_int64)]
        L.fabwd_resolve_dq_mode.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
        L.fabwd_preprocess.argtypes = [P, ctypes.c_void_p, sz, ctypes.c_void_p]
        L.fabwd_forward.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, sz, ctypes.c_void_p]
        L.fabwd_preprocess_stats.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, sz,
                                             ctypes.c_void_p]
        L.fabwd_run.argtypes = [P, ctypes.c_void_p, sz, ctypes.c_void_p]
        L.fabwd_run_main.argtypes = [P, ctypes.c_void_p, sz, ctypes.c_void_p]
        L.fabwd_run_dq.argtypes = [P, ctypes.c_void_p, sz, ctypes.c_void_p]
        L.fabwd_run_static_workspace.argtypes = [P, ctypes.c_void_p]
        L.fabwd_static_workspace_capacity.argtypes = []
        L.fabwd_static_workspace_capacity.restype = ctypes.c_size_t
        L.fabwd_static_workspace_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
        L.fabwd_read_device_status.argtypes = [ctypes.c_void_p, sz, ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
        L.fabwd_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.fabwd_set_wait_limit_ns.restype = ctypes.c_uint64
        L.fabwd_debug_inject_timeout.argtypes = [ctypes.c_int]
        L.fabwd_kernel_binary_version.argtypes = [ctypes.POINTER(ctypes.c_int32)]
        L.fabwd_status_string.argtypes = [ctypes.c_int]
        L.fabwd_status_string.restype = ctypes.c_char_p
        for f in ("fabwd_workspace_size", "fabwd_workspace_layout", "fabwd_preprocess", "fabwd_run",
                  "fabwd_run_main", "fabwd_run_dq", "fabwd_read_device_status", "fabwd_run_static_workspace",
                  "fabwd_resolve_dq_mode", "fabwd_preprocess_stats", "fabwd_forward",
                  "fabwd_static_workspace_status", "fabwd_kernel_binary_version"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def declared_functions() -> list:
    """Names of the functions include/fabwd.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:fabwd_status|const char\*|uint64_t|size_t|int)\s+(fabwd_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return lib().fabwd_status_string(int(status)).decode()


def fabwd_workspace_size(p: fabwd_params) -> int:
    n = ctypes.c_size_t(0)
    s = lib().fabwd_workspace_size(ctypes.byref(p), ctypes.byref(n))
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_workspace_size")
    return n.value


def fabwd_workspace_layout(p: fabwd_params):
    a, b, c = ctypes.c_size_t(0), ctypes.c_size_t(0), ctypes.c_size_t(0)
    r = ctypes.c_int64(0)
    s = lib().fabwd_workspace_layout(ctypes.byref(p), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), ctypes.byref(r))
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_workspace_layout")
    return {"sfmg": a.value, "lse2": b.value, "dq_accum": c.value, "row_stride": r.value}


def fabwd_resolve_dq_mode(p: fabwd_params) -> int:
    m = ctypes.c_int32(0)
    s = lib().fabwd_resolve_dq_mode(ctypes.byref(p), ctypes.byref(m))
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_resolve_dq_mode")
    return m.value


def fabwd_preprocess(p: fabwd_params, workspace: int, workspace_bytes: int, stream: int) -> None:
    s = lib().fabwd_preprocess(ctypes.byref(p), workspace, workspace_bytes, stream)
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_preprocess")


def fabwd_forward(p: fabwd_params, attn_out: int, softmax_lse: int, workspace: int, workspace_bytes: int,
                  stream: int) -> None:
    s = lib().fabwd_forward(ctypes.byref(p), attn_out, softmax_lse, workspace, workspace_bytes, stream)
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_forward")


def fabwd_preprocess_stats(p: fabwd_params, softmax_max: int, softmax_sum: int, stat_stride: int, workspace: int,
                           workspace_bytes: int, stream: int) -> None:
    s = lib().fabwd_preprocess_stats(ctypes.byref(p), softmax_max, softmax_sum, stat_stride, workspace,
                                     workspace_bytes, stream)
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_preprocess_stats")


def fabwd_run(p: fabwd_params, workspace: int, workspace_bytes: int, stream: int) -> None:
    s = lib().fabwd_run(ctypes.byref(p), workspace, workspace_bytes, stream)
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_run")


def fabwd_run_main(p: fabwd_params, workspace: int, workspace_bytes: int, stream: int) -> None:
    s = lib().fabwd_run_main(ctypes.byref(p), workspace, workspace_bytes, stream)
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_run_main")


def fabwd_run_dq(p: fabwd_params, workspace: int, workspace_bytes: int, stream: int) -> None:
    s = lib().fabwd_run_dq(ctypes.byref(p), workspace, workspace_bytes, stream)
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_run_dq")


def fabwd_run_static_workspace(p: fabwd_params, stream: int) -> None:
    """Preprocess + main + convert with the library's fixed scratch array (no allocation)."""
    s = lib().fabwd_run_static_workspace(ctypes.byref(p), stream)
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_run_static_workspace")


def fabwd_static_workspace_capacity() -> int:
    return lib().fabwd_static_workspace_capacity()


def fabwd_static_workspace_status(stream: int):
    """Returns (status code, device status bits) of the last fabwd_run_static_workspace call on the
    current device; synchronises the stream."""
    v = ctypes.c_uint32(0)
    s = lib().fabwd_static_workspace_status(stream, ctypes.byref(v))
    return s, v.value


def fabwd_read_device_status(workspace: int, workspace_bytes: int, stream: int):
    """Returns (status code, device status bits); synchronises the stream."""
    v = ctypes.c_uint32(0)
    s = lib().fabwd_read_device_status(workspace, workspace_bytes, stream, ctypes.byref(v))
    return s, v.value


def fabwd_set_wait_limit_ns(ns: int) -> int:
    return lib().fabwd_set_wait_limit_ns(int(ns))


def fabwd_debug_inject_timeout(on: bool) -> int:
    return lib().fabwd_debug_inject_timeout(1 if on else 0)


def fabwd_kernel_binary_version() -> int:
    v = ctypes.c_int32(0)
    s = lib().fabwd_kernel_binary_version(ctypes.byref(v))
    if s != FABWD_OK:
        raise FabwdError(s, "fabwd_kernel_binary_version")
    return v.value


def fabwd_version() -> int:
    return lib().fabwd_version()


def call_status(name: str, p: fabwd_params, *args) -> int:
    """Raw status of a C entry point (for tests of the error paths)."""
    f = getattr(lib(), name)
    if name in ("fabwd_workspace_size",):
        n = ctypes.c_size_t(0)
        return f(ctypes.byref(p) if p is not None else None, ctypes.byref(n))
    return f(ctypes.byref(p) if p is not None else None, *args)
