"""ctypes view of the C ABI declared in include/gclip.h.

Argument marshalling only: every step of the clip runs in libgclip.so.  If the
library has not been built, loading raises; there is no other code path.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

# return codes
GCLIP_OK = 0
GCLIP_ERR_INVALID_ARG = 1
GCLIP_ERR_OOM = 2
GCLIP_ERR_CUDA = 3
GCLIP_ERR_UNSUPPORTED = 4
GCLIP_ERR_TOO_LARGE = 5
# device status
GCLIP_STATUS_OK = 0
GCLIP_STATUS_TIMEOUT = 1
# dtypes
GCLIP_F32 = 0
GCLIP_F16 = 1
GCLIP_BF16 = 2
# decisions
GCLIP_DECISION_PASS = 0
GCLIP_DECISION_CLIP = 1
GCLIP_DECISION_SKIP = 2
# variants
GCLIP_VARIANT_SPLIT = 0
GCLIP_VARIANT_PERSISTENT = 1
GCLIP_VARIANT_SPLIT_TMA = 2
GCLIP_VARIANT_PERSISTENT_TMA = 3
GCLIP_VARIANT_SPLIT_WAVE = 4
GCLIP_VARIANT_THREE_KERNEL = 5

GCLIP_CHUNK_BYTES = 32768
GCLIP_MAX_TENSORS = 1 << 24
GCLIP_NOALLOC_MAX_CHUNKS = 65536
GCLIP_NOALLOC_SCRATCH_BYTES = GCLIP_NOALLOC_MAX_CHUNKS * 16 + 256


class clip_tensor_desc_t(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("numel", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class clip_result_t(ctypes.Structure):
    _fields_ = [("norm", ctypes.c_float), ("nonfinite", ctypes.c_int32),
                ("decision", ctypes.c_int32), ("status", ctypes.c_int32),
                ("coef_hi", ctypes.c_float), ("coef_lo", ctypes.c_float),
                ("sumsq_hi", ctypes.c_float), ("sumsq_lo", ctypes.c_float),
                ("calls", ctypes.c_uint32), ("reserved", ctypes.c_int32)]


class clip_adamw_state_t(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p)]


class clip_adamw_params_t(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("zero_grads", ctypes.c_int32)]


class clip_chunk_t(ctypes.Structure):
    _fields_ = [("addr", ctypes.c_uint64), ("numel", ctypes.c_uint32),
                ("meta", ctypes.c_uint32)]


_P = ctypes.c_void_p
_SIGNATURES = {
    "clip_create": (ctypes.c_int, [ctypes.POINTER(clip_tensor_desc_t), ctypes.c_int32,
                                   ctypes.POINTER(_P)]),
    "clip_grad_norm": (ctypes.c_int, [_P, ctypes.c_float, ctypes.c_float, _P, _P, _P]),
    "clip_grad_norm_profiled": (ctypes.c_int, [_P, ctypes.c_float, ctypes.c_float, _P, _P, _P,
                                               ctypes.POINTER(_P)]),
    "clip_destroy": (ctypes.c_int, [_P]),
    "clip_set_variant": (ctypes.c_int, [_P, ctypes.c_int32]),
    "clip_get_variant": (ctypes.c_int32, [_P]),
    "clip_result_device": (_P, [_P]),
    "clip_read_result": (ctypes.c_int, [_P, ctypes.POINTER(clip_result_t), _P]),
    "clip_reset": (ctypes.c_int, [_P, _P]),
    "clip_last_status": (ctypes.c_int, [_P, _P, _P]),
    "clip_num_chunks": (ctypes.c_int64, [_P]),
    "clip_persistent_grid": (ctypes.c_int32, [_P]),
    "clip_tma_grid": (ctypes.c_int32, [_P]),
    "clip_plan": (ctypes.c_int, [ctypes.POINTER(clip_tensor_desc_t), ctypes.c_int32,
                                 ctypes.POINTER(clip_chunk_t), ctypes.c_int64,
                                 ctypes.POINTER(ctypes.c_int64)]),
    "clip_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "clip_debug_barrier": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int64]),
    "clip_set_l2_keep": (ctypes.c_int, [_P, ctypes.c_int64]),
    "clip_attach_adamw": (ctypes.c_int, [_P, ctypes.POINTER(clip_adamw_state_t), ctypes.c_int32]),
    "clip_attach_f32_out": (ctypes.c_int, [_P, ctypes.POINTER(_P), ctypes.c_int32]),
    "clip_grad_norm_per_tensor": (ctypes.c_int, [_P, ctypes.c_float, ctypes.c_float, _P, _P, _P]),
    "clip_read_per_tensor": (ctypes.c_int, [_P, ctypes.POINTER(clip_result_t), ctypes.c_int32, _P]),
    "clip_grad_norm_to_f32": (ctypes.c_int, [_P, ctypes.c_float, ctypes.c_float, _P, _P, _P]),
    "clip_attach_addend": (ctypes.c_int, [_P, ctypes.POINTER(_P), ctypes.c_int32]),
    "clip_grad_norm_accumulate": (ctypes.c_int, [_P, ctypes.c_float, ctypes.c_float, _P, _P, _P]),
    "clip_grad_norm_adamw": (ctypes.c_int, [_P, ctypes.c_float, ctypes.c_float,
                                            ctypes.POINTER(clip_adamw_params_t), ctypes.c_int64,
                                            _P, _P, _P]),
    "clip_adamw_step": (ctypes.c_int, [_P, ctypes.POINTER(clip_adamw_params_t), ctypes.c_int64, _P]),
    "clip_grad_norm_flat_noalloc": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int32,
                                                   ctypes.c_float, ctypes.c_float, _P, _P, _P]),
}

_LIB = None


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libgclip.so (built by ``global_l2_norm_gb300.build()``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"libgclip.so is not built ({path}); run global_l2_norm_gb300.build() "
            "(needs nvcc).  There is no fallback implementation.")
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = L
    return L


class GclipError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = load().clip_status_string(code).decode()
        super().__init__(f"{fn} failed: {msg} (code {code})")
        self.code = code


def check(fn: str, code: int) -> None:
    if code != GCLIP_OK:
        raise GclipError(fn, code)
