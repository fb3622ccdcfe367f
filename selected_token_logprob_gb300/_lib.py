"""ctypes loader of libfused_logp.so (the C ABI of include/fused_logp.h).

There is no fallback: if the library is missing or does not load, every call
raises.  Build it with ``python -m selected_token_logprob_gb300.build``.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

FLP_OK, FLP_EINVAL, FLP_EUNSUPPORTED, FLP_ECUDA = 0, 1, 2, 3
STATUS_NAMES = {0: "FLP_OK", 1: "FLP_EINVAL", 2: "FLP_EUNSUPPORTED", 3: "FLP_ECUDA"}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64

# name -> (restype, argtypes), mirroring include/fused_logp.h
SIGNATURES = {
    "flp_last_error": (ctypes.c_char_p, []),
    "flp_version": (ctypes.c_char_p, []),
    "flp_tile_width": (_I64, [_I64]),
    "fused_logp_forward": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _P]),
    "fused_logp_backward": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _P, _I64, _P]),
    "logp_shard_partials": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "logp_merge_partials": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P]),
    "fused_logp_forward_ex": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I64, _P, _I64, _P,
                                             ctypes.c_float, _P, _P, _P, _P]),
    "fused_logp_backward_ex": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I64, _P, _I64, _P,
                                              ctypes.c_float, _P, _P, _P, _P, _I64, _P]),
    "logp_shard_partials_ex": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I64, _I64, _I64,
                                              ctypes.c_float, _P, _P, _P, _P, _P]),
    "logp_merge_partials_ex": (ctypes.c_int, [_P, _P, _P, _P, _I64, _P, _I64, _I64,
                                              ctypes.c_float, _P, _P, _P, _P]),
    "logp_shard_backward": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _P,
                                           _I64, _P]),
    "logp_shard_backward_ex": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I64, _I64, _I64, _P, _I64, _P,
                                              ctypes.c_float, _P, _P, _P, _P, _I64, _P]),
    "logp_merge_gathered_partials_ex": (ctypes.c_int, [_P, _I64, _I64, ctypes.POINTER(_I64),
                                                       ctypes.POINTER(_I64), _P, _I64, _P, _I64, _I64,
                                                       ctypes.c_float, _P, _P, _P, _P]),
    "logp_grpo_loss_workspace_size": (ctypes.c_int, [_I64, _I64, ctypes.POINTER(_I64)]),
    "logp_grpo_loss": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, ctypes.c_int,
                                      ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_float, _P, _I64, _P, _P, _P, _P]),
    "fused_linear_logp_merge_gathered": (ctypes.c_int, [_P, _I64, ctypes.c_int, _P, _P, _I64, _I64, _P, _I64, _P,
                                                        ctypes.c_float, _P, _P, _P, _P]),
    "flp_sum_blocks": (ctypes.c_int, [_P, _I64, ctypes.c_int, _I64, _I64, _P, _I64, _P]),
    "logp_grpo_loss_counts": (ctypes.c_int, [_P, _P, _I64, _I64, ctypes.c_int, ctypes.c_float, _P, _I64, _P]),
    "logp_grpo_loss_counted": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, ctypes.c_int,
                                              ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                              ctypes.c_float, _P, _I64, _P, _P, _P, _P]),
    "fused_linear_logp_workspace_size": (ctypes.c_int, [_I64, _I64, ctypes.POINTER(_I64)]),
    "fused_linear_logp_forward": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _I64, _P,
                                                 ctypes.c_float, _P, _I64, _P, _P, _P, _P]),
    "fused_linear_logp_forward_noalloc": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _I64,
                                                         _P, ctypes.c_float, _P, _P, _P, _P]),
    "fused_linear_logp_shard_partials": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _I64, _I64, _I64, _P,
                                                        ctypes.c_float, _P, _I64, _P]),
    "fused_linear_logp_merge": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _P, ctypes.c_float, _P, _P, _P,
                                               _P]),
    "fused_linear_logp_shard_backward": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _I64, _I64, _I64, _P,
                                                        _I64, _P, ctypes.c_float, _P, _P, _P, _P, _I64, _P, _I64,
                                                        ctypes.c_int, _P, _I64, ctypes.c_int, _P]),
    "fused_linear_logp_backward_workspace_size": (ctypes.c_int, [_I64, _I64, ctypes.POINTER(_I64)]),
    "fused_linear_logp_backward": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _I64, _P,
                                                  ctypes.c_float, _P, _P, _P, _P, _I64, _P, _I64, _P, _I64,
                                                  ctypes.c_int, _P]),
    "flp_device_error": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_int)]),
    "flp_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int, _I64, ctypes.POINTER(ctypes.c_int)]),
    "flp_selftest_ex2_bias": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                             ctypes.POINTER(ctypes.c_double)]),
}


class FusedLogpError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """The loaded library; raises if it is not built (no silent fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and _build.stale():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m selected_token_logprob_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(fn: str, status: int) -> None:
    if status != FLP_OK:
        msg = load().flp_last_error()
        raise FusedLogpError(fn, status, msg.decode() if msg else "")
