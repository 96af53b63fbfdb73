"""CPU oracle for the 1-bit LAMB hot path (TEST INFRASTRUCTURE).

A ctypes binding to ``lamb1b_oracle.c``: a plain single-threaded C statement
of the warmup (LAMB) step, the variance freeze and the compression step
(error-compensated 1-bit compression of every worker's momentum, the server's
average/recompress/scatter, the reconstructed-gradient layerwise factor and
the frozen-variance update) from the 1-bit LAMB paper (arXiv 2104.06069).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this package.  It shares no code with the GPU library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "liblamb1b_oracle.so")

# binary32 evaluation with no contraction of a*b+c into one rounding
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fno-unsafe-math-optimizations"]


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "lamb1b_oracle.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p


class _OrcT(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64), ("L", ctypes.c_int32), ("W", ctypes.c_int32),
        ("C", ctypes.c_int32), ("variant", ctypes.c_int32),
        ("off", _P), ("numel", _P),
        ("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float), ("wd", ctypes.c_float),
        ("cmin", ctypes.c_float), ("cmax", ctypes.c_float), ("cema", ctypes.c_float),
        ("fmin", ctypes.c_float), ("fmax", ctypes.c_float), ("fthr", ctypes.c_float),
        ("err_bf16", ctypes.c_int32),
        ("x", _P), ("m", _P), ("v", _P), ("v_fresh", _P), ("e_w", _P), ("e_s", _P),
        ("signs_w", _P), ("signs_s", _P), ("scale_w", _P), ("scale_s", _P),
        ("c_bar", _P), ("r_prev", _P), ("c_cur", _P), ("R", _P), ("Sx", _P), ("Su", _P),
        ("t", ctypes.c_int64), ("n_warm", ctypes.c_int32), ("stage", ctypes.c_int32),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        # LAMB1B_ORACLE_LIB: load another build of lamb1b_oracle.c (the
        # mutation test points it at copies with one planted mistake)
        alt = os.environ.get("LAMB1B_ORACLE_LIB")
        L = ctypes.CDLL(alt if alt else build())
        L.orc_cpt_sumsq.argtypes = [_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        L.orc_cpt_sumsq.restype = ctypes.c_float
        L.orc_compress_chunk.argtypes = [_P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64,
                                         _P, _P]
        L.orc_compress_chunk.restype = ctypes.c_float
        L.orc_layer_factor.argtypes = [ctypes.c_float] * 5
        L.orc_bf16_round.argtypes = [ctypes.c_float]
        L.orc_bf16_round.restype = ctypes.c_float
        L.orc_layer_factor.restype = ctypes.c_float
        for f in ("orc_warmup_step", "orc_compress_step"):
            getattr(L, f).argtypes = [ctypes.POINTER(_OrcT), _P, ctypes.c_int64]
            getattr(L, f).restype = ctypes.c_int
        L.orc_freeze.argtypes = [ctypes.POINTER(_OrcT)]
        L.orc_freeze.restype = ctypes.c_int
        L.orc_compress_chunk_step.argtypes = [ctypes.POINTER(_OrcT), _P, ctypes.c_int64,
                                              ctypes.c_int64, _P]
        L.orc_compress_chunk_step.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_P)


# ---------------------------------------------------------------------------
# stand-alone pieces (used by the pin tests)
# ---------------------------------------------------------------------------

def cpt_sumsq(a: np.ndarray, lo: int, hi: int, a0: int = 0) -> np.float32:
    """Canonical pairwise-tree sum of squares of elements [lo, hi); element i
    is a[i - a0]."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return np.float32(lib().orc_cpt_sumsq(_p(a), a0, lo, hi))


def compress_chunk(z: np.ndarray, k: int, C: int):
    """1-bit compression of the n = len(z) values of chunk k (chunk size C).
    Returns (scale, words[C//32] uint32, err[n])."""
    z = np.ascontiguousarray(z, dtype=np.float32)
    n = z.shape[0]
    words = np.zeros(C // 32, dtype=np.uint32)
    err = np.zeros(max(n, 1), dtype=np.float32)
    s = lib().orc_compress_chunk(_p(z), k, C, n, _p(words), _p(err))
    return np.float32(s), words, err[:n]


def bf16_round(x: float) -> np.float32:
    return np.float32(lib().orc_bf16_round(float(x)))


def layer_factor(R, r_prev, fmin, fmax, fthr) -> np.float32:
    return np.float32(lib().orc_layer_factor(R, r_prev, fmin, fmax, fthr))


# ---------------------------------------------------------------------------
# full optimizer state
# ---------------------------------------------------------------------------

class Oracle:
    """Optimizer state held in numpy arrays, stepped by the C oracle."""

    STATE_F32 = ("x", "m", "v", "v_fresh", "e_w", "e_s", "scale_w", "scale_s",
                 "c_bar", "r_prev", "c_cur", "R", "Sx", "Su")

    def __init__(self, offsets, numels, W: int, chunk: int, hp: dict, x0: np.ndarray,
                 variant: int = 0, err_bf16: int = 0):
        self.off = np.ascontiguousarray(offsets, dtype=np.int64)
        self.numel = np.ascontiguousarray(numels, dtype=np.int64)
        L = len(self.off)
        N = int(self.numel.sum())
        self.N, self.L, self.W, self.C = N, L, W, chunk
        self.variant = int(variant)
        self.err_bf16 = int(err_bf16)
        self.K = -(-N // chunk)
        self.NW = -(-N // 32)
        self.hp = dict(hp)
        self.x = np.ascontiguousarray(x0, dtype=np.float32).copy()
        assert self.x.shape == (N,)
        self.m = np.zeros(N, np.float32)
        self.v = np.zeros(N, np.float32)
        self.v_fresh = np.zeros(N, np.float32)
        self.e_w = np.zeros((W, N), np.float32)
        self.e_s = np.zeros(N, np.float32)
        self.signs_w = np.zeros((W, self.NW), np.uint32)
        self.signs_s = np.zeros(self.NW, np.uint32)
        self.scale_w = np.zeros((W, self.K), np.float32)
        self.scale_s = np.zeros(self.K, np.float32)
        self.c_bar = np.ones(L, np.float32)
        self.r_prev = np.ones(L, np.float32)
        self.c_cur = np.ones(L, np.float32)
        self.R = np.zeros(L, np.float32)
        self.Sx = np.zeros(L, np.float32)
        self.Su = np.zeros(L, np.float32)
        self.t = 0
        self.n_warm = 0
        self.stage = 0

    # the C struct is rebuilt around the numpy arrays for every call
    def _struct(self) -> _OrcT:
        h = self.hp
        s = _OrcT()
        s.N, s.L, s.W, s.C = self.N, self.L, self.W, self.C
        s.variant = self.variant
        s.err_bf16 = self.err_bf16
        s.off, s.numel = _p(self.off), _p(self.numel)
        s.lr, s.beta1, s.beta2 = h["lr"], h["beta1"], h["beta2"]
        s.eps, s.wd = h["eps"], h["weight_decay"]
        s.cmin, s.cmax, s.cema = h["coeff_min"], h["coeff_max"], h["coeff_ema"]
        s.fmin, s.fmax, s.fthr = h["factor_min"], h["factor_max"], h["factor_threshold"]
        for name in ("x", "m", "v", "v_fresh", "e_w", "e_s", "signs_w", "signs_s",
                     "scale_w", "scale_s", "c_bar", "r_prev", "c_cur", "R", "Sx", "Su"):
            setattr(s, name, _p(getattr(self, name)))
        s.t, s.n_warm, s.stage = self.t, self.n_warm, self.stage
        return s

    def _pull(self, s: _OrcT):
        self.t, self.n_warm, self.stage = int(s.t), int(s.n_warm), int(s.stage)

    def _grads(self, g):
        g = np.ascontiguousarray(g, dtype=np.float32)
        assert g.ndim == 2 and g.shape[0] == self.W and g.shape[1] >= self.N
        return g

    def warmup_step(self, g: np.ndarray):
        g = self._grads(g)
        s = self._struct()
        rc = lib().orc_warmup_step(ctypes.byref(s), _p(g), g.shape[1])
        self._pull(s)
        if rc:
            raise RuntimeError(f"oracle warmup_step: {rc}")

    def freeze(self):
        s = self._struct()
        rc = lib().orc_freeze(ctypes.byref(s))
        self._pull(s)
        if rc:
            raise RuntimeError(f"oracle freeze: {rc}")

    def compress_step(self, g: np.ndarray):
        g = self._grads(g)
        s = self._struct()
        rc = lib().orc_compress_step(ctypes.byref(s), _p(g), g.shape[1])
        self._pull(s)
        if rc:
            raise RuntimeError(f"oracle compress_step: {rc}")

    def compress_chunk_step(self, g: np.ndarray, k: int) -> np.ndarray:
        """Only chunk k of a compression step (no factor, no update, t kept).
        Returns rho for the chunk's elements."""
        g = self._grads(g)
        s = self._struct()
        rho = np.zeros(self.C, np.float32)
        rc = lib().orc_compress_chunk_step(ctypes.byref(s), _p(g), g.shape[1], k, _p(rho))
        if rc:
            raise RuntimeError(f"oracle compress_chunk_step: {rc}")
        n = min(self.C, self.N - k * self.C)
        return rho[:n]

    def snapshot(self) -> dict:
        d = {k: getattr(self, k).copy() for k in self.STATE_F32}
        d["signs_w"] = self.signs_w.copy()
        d["signs_s"] = self.signs_s.copy()
        d["t"], d["n_warm"], d["stage"] = self.t, self.n_warm, self.stage
        return d
