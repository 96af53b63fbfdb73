"""ctypes declarations of the lamb1b C ABI (include/lamb1b.h, include/lamb1b_gen.h).

Argument marshalling only: every step of the optimizer runs in liblamb1b.so.
Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

_P = ctypes.c_void_p

LAMB1B_OK = 0
ERR_ARG, ERR_ALIGN, ERR_WORKSPACE, ERR_STATE, ERR_CUDA, ERR_NONFINITE, ERR_DEVICE, ERR_TIMEOUT = \
    -1, -2, -3, -4, -5, -6, -7, -8
GRAD_F32, GRAD_BF16, GRAD_PHILOX = 0, 1, 2

EXPORTED = ("lamb1b_workspace_bytes", "lamb1b_init", "lamb1b_warmup_step",
            "lamb1b_freeze_variance", "lamb1b_compress_step", "lamb1b_compress_step_host",
            "lamb1b_state_view",
            "lamb1b_set_counters", "lamb1b_check_status", "lamb1b_set_trace_events",
            "lamb1b_set_fault_injection", "lamb1b_sync_momentum", "lamb1b_destroy",
            "lamb1b_error_string", "lamb1b_gen_grads", "lamb1b_gen_params",
            "lamb1b_gen_selfcheck", "lamb1b_tensor_sumsq_noalloc")


class Layer(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_int64), ("numel", ctypes.c_int64)]


class HParams(ctypes.Structure):
    _fields_ = [("W", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("coeff_min", ctypes.c_float), ("coeff_max", ctypes.c_float),
                ("coeff_ema", ctypes.c_float),
                ("factor_min", ctypes.c_float), ("factor_max", ctypes.c_float),
                ("factor_threshold", ctypes.c_float), ("check_finite", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("error_storage", ctypes.c_int32)]


class GradsDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("pad0", ctypes.c_int32), ("ptr", _P),
                ("ld", ctypes.c_int64), ("seed", ctypes.c_uint64),
                ("layer_std", _P), ("layer_heavy", _P),
                ("heavy_scale", ctypes.c_float), ("pad1", ctypes.c_int32)]


class State(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("m", "v", "v_fresh", "e_w", "e_s", "signs_w", "signs_s",
                                  "scale_w", "scale_s", "c_bar", "r_prev", "c_cur", "R_last",
                                  "Sx", "Su")] + [
        ("N", ctypes.c_int64), ("Np", ctypes.c_int64), ("K", ctypes.c_int64),
        ("words_ld", ctypes.c_int64), ("L", ctypes.c_int32), ("W", ctypes.c_int32),
        ("C", ctypes.c_int32), ("stage", ctypes.c_int32), ("t", ctypes.c_int64),
        ("n_warmup", ctypes.c_int32), ("pad0", ctypes.c_int32)]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """The loaded library.  Raises when it is missing (no silent fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(
                f"liblamb1b.so is not built ({path}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        _build.build()
    L = ctypes.CDLL(path)
    i32, i64, u64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
    L.lamb1b_workspace_bytes.argtypes = [ctypes.POINTER(Layer), i32, ctypes.POINTER(HParams)]
    L.lamb1b_workspace_bytes.restype = ctypes.c_size_t
    L.lamb1b_init.argtypes = [ctypes.POINTER(_P), ctypes.POINTER(Layer), i32,
                              ctypes.POINTER(HParams), _P, _P, ctypes.c_size_t, _P]
    L.lamb1b_warmup_step.argtypes = [_P, ctypes.POINTER(GradsDesc), _P]
    L.lamb1b_freeze_variance.argtypes = [_P, _P]
    L.lamb1b_compress_step.argtypes = [_P, ctypes.POINTER(GradsDesc), _P]
    L.lamb1b_compress_step_host.argtypes = [_P, ctypes.POINTER(GradsDesc), _P, _P, _P, _P, _P]
    L.lamb1b_state_view.argtypes = [_P, ctypes.POINTER(State)]
    L.lamb1b_set_counters.argtypes = [_P, i64, i32, i32]
    L.lamb1b_check_status.argtypes = [_P, _P]
    L.lamb1b_set_trace_events.argtypes = [_P, ctypes.POINTER(_P), i32]
    L.lamb1b_set_fault_injection.argtypes = [_P, i32, ctypes.c_uint32]
    L.lamb1b_sync_momentum.argtypes = [_P, _P]
    L.lamb1b_destroy.argtypes = [_P]
    L.lamb1b_error_string.argtypes = [ctypes.c_int]
    L.lamb1b_error_string.restype = ctypes.c_char_p
    L.lamb1b_gen_grads.argtypes = [_P, i64, i32, i32, u64, i64, _P, _P, i32, _P, _P, f32, _P]
    L.lamb1b_gen_params.argtypes = [_P, i64, i64, f32, u64, _P]
    L.lamb1b_gen_selfcheck.argtypes = [_P, u64, _P]
    L.lamb1b_tensor_sumsq_noalloc.argtypes = [_P, ctypes.POINTER(Layer), i32, _P, _P]
    for f in EXPORTED:
        if f not in ("lamb1b_workspace_bytes", "lamb1b_error_string"):
            getattr(L, f).restype = ctypes.c_int
    _lib = L
    return L


class Lamb1bError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = load().lamb1b_error_string(code).decode()
        super().__init__(f"{fn}: {msg} ({code})")
        self.code = code


def check(fn: str, code: int) -> int:
    if code != LAMB1B_OK:
        raise Lamb1bError(fn, code)
    return code
