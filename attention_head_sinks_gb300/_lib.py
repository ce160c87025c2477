"""ctypes loader for ``libsa.so`` (the C ABI in ``include/sa.h``).

The library is built in-tree by :mod:`attention_head_sinks_gb300.build`.  There
is no fallback: if the library is missing, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsa.so")

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_CUDA, SA_ERR_WORKSPACE = range(5)
# sa_sink_mode values of include/sa.h
SINK_NONE, SINK_KEY0_BIAS, SINK_NULL_LOGIT = 0, 1, 2
STATUS_NAMES = {0: "SA_OK", 1: "SA_ERR_INVALID_ARG", 2: "SA_ERR_UNSUPPORTED",
                3: "SA_ERR_CUDA", 4: "SA_ERR_WORKSPACE"}

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F32 = ctypes.c_float
_SZ = ctypes.c_size_t

# name -> (restype, argtypes); every symbol include/sa.h declares.
SIGNATURES = {
    "sa_varlen_window_fwd": (ctypes.c_int, [
        _P, _P, _P, _P, _I32, _I64, _I32, _I32, _I32, _I32, _I32, _P, _I32,
        _F32, _P, _P, _P]),
    "sa_sparse_index_fwd": (ctypes.c_int, [
        _P, _P, _I64, _I32, _I32, _P, _I32, _I32, _I32, _P, _I32, _F32, _P, _P,
        _P, _SZ, _P]),
    "sa_sparse_index_fwd_fp8": (ctypes.c_int, [
        _P, _P, _P, _I64, _I32, _I32, _P, _I32, _I32, _I32, _P, _I32, _F32, _P,
        _P, _P, _SZ, _P]),
    "sa_sparse_index_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "sa_sparse_index_fwd_noalloc": (ctypes.c_int, [
        _P, _P, _I64, _I32, _I32, _P, _I32, _I32, _I32, _P, _I32, _F32, _P, _P,
        _P]),
    "sa_block_sparse_fwd": (ctypes.c_int, [
        _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I32, _I32, _P, _I32, _P,
        _I32, _F32, _P, _P, _P, _SZ, _P]),
    "sa_block_sparse_fwd_index_heads": (ctypes.c_int, [
        _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I32, _I32, _I32, _P, _I32,
        _P, _I32, _F32, _P, _P, _P]),
    "sa_block_select": (ctypes.c_int, [
        _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P]),
    "sa_merge_attn_states": (ctypes.c_int, [
        _P, _P, _P, _P, _I64, _I32, _I32, _P, _I32, _P, _P, _P]),
    "sa_last_error": (ctypes.c_char_p, []),
    "sa_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "sa_check_wait_expiry": (ctypes.c_int, [_P]),
    "sa_version": (ctypes.c_uint32, []),
}

_lock = threading.Lock()
_lib = None


class SAError(RuntimeError):
    """A non-OK ``sa_status`` from the C ABI."""

    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


def lib() -> ctypes.CDLL:
    """Load ``libsa.so`` once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libsa.so is not built (%s); run "
                    "`python -c \"import __graft_entry__ as g; g.build()\"`" % LIB_PATH)
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
            _lib = l
    return _lib


def check(status: int) -> None:
    if status != SA_OK:
        msg = lib().sa_last_error()
        raise SAError(status, msg.decode() if msg else "")
