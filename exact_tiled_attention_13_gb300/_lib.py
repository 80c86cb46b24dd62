"""ctypes binding of libattn's C ABI (include/attn.h). Argument marshalling only."""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

ATTN_MASK_NONE = 0
ATTN_MASK_CAUSAL = 1
ATTN_BIAS_DENSE = 2
ATTN_BIAS_KEY = 4
ATTN_BIAS_SHARED = 8
ATTN_OUT_BF16 = 0
ATTN_OUT_F32 = 1

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_NO_DEVICE = -3
ATTN_ERR_UNSUPPORTED_DEVICE = -4
ATTN_ERR_LAUNCH = -5
ATTN_ERR_DEVICE_TIMEOUT = -6
ATTN_ERR_CUDA = -7
ATTN_ERR_SCRATCH_LIMIT = -8
ATTN_STATIC_SCRATCH_BYTES = 33554432
ATTN_ABI_VERSION = 107

ATTN_FAULT_NONE = 0
ATTN_FAULT_SKIP_FIRST_K = 1

# Every symbol include/attn.h declares, with its ctypes signature.
_P = ctypes.c_void_p
SIGNATURES = {
    "attn_fwd": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _P, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, ctypes.c_float, _P, ctypes.c_int, _P,
                                _P]),
    "attn_fwd_ex": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, _P,
                                   ctypes.c_int, _P, _P]),
    "attn_fwd_splitkv": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_int, _P, ctypes.c_ulonglong, _P,
                                        ctypes.c_int, _P, _P]),
    "attn_fwd_splitkv_plan": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                             ctypes.POINTER(ctypes.c_ulonglong)]),
    "attn_fwd_splitkv_static": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_float, ctypes.c_int, _P,
                                               ctypes.c_int, _P, _P]),
    "attn_fwd_host": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, _P,
                                     ctypes.c_int, _P, _P, ctypes.c_ulonglong, ctypes.c_int, _P]),
    "attn_fwd_host_staging_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_ulonglong)]),
    "attn_bwd_host": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_float, _P, _P, _P, _P, ctypes.c_ulonglong,
                                     ctypes.c_int, _P]),
    "attn_bwd_host_staging_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_ulonglong)]),
    "attn_bwd": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_float, _P, _P, _P, _P, ctypes.c_ulonglong,
                                _P]),
    "attn_bwd_workspace_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_ulonglong)]),
    "attn_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_device_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint)]),
    "attn_set_wait_timeout_ns": (ctypes.c_ulonglong, [ctypes.c_ulonglong]),
    "attn_set_fault_injection": (ctypes.c_int, [ctypes.c_int]),
    "attn_version": (ctypes.c_int, []),
}

_lock = threading.Lock()
_lib = None
_path = None


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


def load():
    """Load libattn, building it in-tree first if the current sources have no library.

    There is no fallback: if the library cannot be built or loaded this raises.
    """
    global _lib, _path
    with _lock:
        if _lib is not None:
            return _lib
        path = os.environ.get("ATTN_LIBRARY") or _build.build()
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib, _path = lib, path
        return lib


def library_path() -> str:
    load()
    return _path


def strerror(code: int) -> str:
    return load().attn_strerror(int(code)).decode()


def attn_fwd_raw(Q, K, V, mode, C, BH, N, d, d_v, scale, O, out_dtype, LSE, stream) -> int:
    """The C entry point with plain integers as pointers; returns its code unchanged."""
    return load().attn_fwd(Q, K, V, int(mode), C, int(BH), int(N), int(d), int(d_v), float(scale), O,
                           int(out_dtype), LSE, stream)


def attn_fwd_ex_raw(Q, K, V, mode, C, ckey, BH, Nq, Nk, d, d_v, scale, O, out_dtype, LSE,
                    stream) -> int:
    """attn_fwd_ex with plain integers as pointers; returns its code unchanged."""
    return load().attn_fwd_ex(Q, K, V, int(mode), C, ckey, int(BH), int(Nq), int(Nk), int(d),
                              int(d_v), float(scale), O, int(out_dtype), LSE, stream)


def attn_fwd_splitkv_raw(Q, K, V, mode, C, ckey, BH, Nq, Nk, d, d_v, scale, n_splits, workspace,
                         workspace_bytes, O, out_dtype, LSE, stream) -> int:
    """attn_fwd_splitkv with plain integers as pointers; returns its code unchanged."""
    return load().attn_fwd_splitkv(Q, K, V, int(mode), C, ckey, int(BH), int(Nq), int(Nk), int(d),
                                   int(d_v), float(scale), int(n_splits), workspace,
                                   int(workspace_bytes), O, int(out_dtype), LSE, stream)


def attn_fwd_splitkv_static_raw(Q, K, V, mode, C, ckey, BH, Nq, Nk, d, d_v, scale, n_splits, O,
                                out_dtype, LSE, stream) -> int:
    """attn_fwd_splitkv_static (partials in the library's fixed array) with plain integers
    as pointers; returns its code unchanged."""
    return load().attn_fwd_splitkv_static(Q, K, V, int(mode), C, ckey, int(BH), int(Nq), int(Nk),
                                          int(d), int(d_v), float(scale), int(n_splits), O,
                                          int(out_dtype), LSE, stream)


def attn_fwd_splitkv_plan(mode, BH, Nq, Nk, d, d_v, n_splits=0):
    """(code, key ranges, workspace bytes) of attn_fwd_splitkv for these arguments."""
    splits = ctypes.c_int(0)
    nbytes = ctypes.c_ulonglong(0)
    code = load().attn_fwd_splitkv_plan(int(mode), int(BH), int(Nq), int(Nk), int(d), int(d_v),
                                        int(n_splits), ctypes.byref(splits), ctypes.byref(nbytes))
    return code, splits.value, nbytes.value


def attn_fwd_host_raw(Q, K, V, mode, C, ckey, BH, Nq, Nk, d, d_v, scale, O, out_dtype, LSE, staging,
                      staging_bytes, heads_per_chunk, stream) -> int:
    """attn_fwd_host (host tensors streamed through a device staging buffer) with plain
    integers as pointers; returns its code unchanged."""
    return load().attn_fwd_host(Q, K, V, int(mode), C, ckey, int(BH), int(Nq), int(Nk), int(d),
                                int(d_v), float(scale), O, int(out_dtype), LSE, staging,
                                int(staging_bytes), int(heads_per_chunk), stream)


def attn_fwd_host_staging_bytes(mode, BH, Nq, Nk, d, d_v, out_dtype, heads_per_chunk=0):
    """(code, bytes) of the staging buffer attn_fwd_host needs."""
    nbytes = ctypes.c_ulonglong(0)
    code = load().attn_fwd_host_staging_bytes(int(mode), int(BH), int(Nq), int(Nk), int(d), int(d_v),
                                              int(out_dtype), int(heads_per_chunk), ctypes.byref(nbytes))
    return code, nbytes.value


def attn_bwd_raw(Q, K, V, O, o_dtype, dO, LSE, mode, C, ckey, BH, Nq, Nk, d, d_v, scale, dQ, dK,
                 dV, workspace, workspace_bytes, stream) -> int:
    """attn_bwd with plain integers as pointers; returns its code unchanged."""
    return load().attn_bwd(Q, K, V, O, int(o_dtype), dO, LSE, int(mode), C, ckey, int(BH), int(Nq),
                           int(Nk), int(d), int(d_v), float(scale), dQ, dK, dV, workspace,
                           int(workspace_bytes), stream)


def attn_bwd_host_raw(Q, K, V, O, o_dtype, dO, LSE, mode, C, ckey, BH, Nq, Nk, d, d_v, scale, dQ,
                      dK, dV, staging, staging_bytes, heads_per_chunk, stream) -> int:
    """attn_bwd_host (host tensors streamed through a device staging buffer) with plain
    integers as pointers; returns its code unchanged."""
    return load().attn_bwd_host(Q, K, V, O, int(o_dtype), dO, LSE, int(mode), C, ckey, int(BH),
                                int(Nq), int(Nk), int(d), int(d_v), float(scale), dQ, dK, dV, staging,
                                int(staging_bytes), int(heads_per_chunk), stream)


def attn_bwd_host_staging_bytes(mode, BH, Nq, Nk, d, d_v, o_dtype, heads_per_chunk=0):
    """(code, bytes) of the staging buffer attn_bwd_host needs."""
    nbytes = ctypes.c_ulonglong(0)
    code = load().attn_bwd_host_staging_bytes(int(mode), int(BH), int(Nq), int(Nk), int(d), int(d_v),
                                              int(o_dtype), int(heads_per_chunk), ctypes.byref(nbytes))
    return code, nbytes.value


def attn_bwd_workspace_bytes(BH, Nq):
    """(code, bytes) of the workspace attn_bwd needs."""
    nbytes = ctypes.c_ulonglong(0)
    code = load().attn_bwd_workspace_bytes(int(BH), int(Nq), ctypes.byref(nbytes))
    return code, nbytes.value


def attn_device_status(stream=None):
    """(code, raw watchdog word) after synchronising `stream` (a raw cudaStream_t or None)."""
    word = ctypes.c_uint(0)
    code = load().attn_device_status(stream, ctypes.byref(word))
    return code, word.value


def attn_set_wait_timeout_ns(ns: int) -> int:
    return load().attn_set_wait_timeout_ns(int(ns))


def attn_set_fault_injection(fault: int) -> int:
    """Test hook of the watchdog (see include/attn.h); returns the library's code."""
    return load().attn_set_fault_injection(int(fault))


def attn_version() -> int:
    return load().attn_version()
