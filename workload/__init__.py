"""Seeded synthetic workloads for the 1-bit LAMB hot path.

This package is the input generator that both sides of every parity check
consume: the CPU oracle and the GPU library.  It holds none of the
optimizer's arithmetic.  It provides

* the per-tensor layer tables of the five workloads (a toy table, BERT-Base,
  BERT-Large, BERT-Large with 32 workers and in-kernel gradients, GPT-2-XL),
  laid out as concatenated parameter tensors in model order;
* the hyper-parameters each workload runs with;
* a ctypes binding to ``gen.c`` (Philox4x32-10 counter generator with an
  exactly specified Box-Muller normal and Student-t transform) that produces
  initial parameters and gradients.

The 1-bit LAMB paper (arXiv 2104.06069, introduction and background on LAMB)
describes BERT pre-training with one scaling coefficient per tensor; the
tables below are the standard BERT and GPT-2 parameter lists, one row per
tensor.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libworkload.so")


# --------------------------------------------------------------------------
# layer tables
# --------------------------------------------------------------------------

def bert_tensors(n_layers: int, hidden: int, ffn: int, vocab: int,
                 max_pos: int = 512, type_vocab: int = 2):
    """BERT pre-training parameter list (MLM decoder weight tied to the
    word embedding, so only its bias appears)."""
    H, F = hidden, ffn
    t = [("emb.word", (vocab, H)), ("emb.pos", (max_pos, H)),
         ("emb.type", (type_vocab, H)), ("emb.ln.g", (H,)), ("emb.ln.b", (H,))]
    for i in range(n_layers):
        p = f"enc{i}."
        for n in ("q", "k", "v", "attn_out"):
            t += [(p + n + ".w", (H, H)), (p + n + ".b", (H,))]
        t += [(p + "attn_ln.g", (H,)), (p + "attn_ln.b", (H,))]
        t += [(p + "ffn_in.w", (F, H)), (p + "ffn_in.b", (F,)),
              (p + "ffn_out.w", (H, F)), (p + "ffn_out.b", (H,))]
        t += [(p + "ffn_ln.g", (H,)), (p + "ffn_ln.b", (H,))]
    t += [("pooler.w", (H, H)), ("pooler.b", (H,)),
          ("mlm.transform.w", (H, H)), ("mlm.transform.b", (H,)),
          ("mlm.ln.g", (H,)), ("mlm.ln.b", (H,)), ("mlm.dec.b", (vocab,)),
          ("nsp.w", (2, H)), ("nsp.b", (2,))]
    return t


def gpt2_tensors(n_layers: int, hidden: int, ffn: int, vocab: int, n_pos: int = 1024):
    """GPT-2 parameter list (Conv1D weights stored [in, out])."""
    H, F = hidden, ffn
    t = [("wte", (vocab, H)), ("wpe", (n_pos, H))]
    for i in range(n_layers):
        p = f"h{i}."
        t += [(p + "ln_1.g", (H,)), (p + "ln_1.b", (H,)),
              (p + "attn.c_attn.w", (H, 3 * H)), (p + "attn.c_attn.b", (3 * H,)),
              (p + "attn.c_proj.w", (H, H)), (p + "attn.c_proj.b", (H,)),
              (p + "ln_2.g", (H,)), (p + "ln_2.b", (H,)),
              (p + "mlp.c_fc.w", (H, F)), (p + "mlp.c_fc.b", (F,)),
              (p + "mlp.c_proj.w", (F, H)), (p + "mlp.c_proj.b", (H,))]
    t += [("ln_f.g", (H,)), ("ln_f.b", (H,))]
    return t


def toy_tensors():
    return [("t0", (64, 64)), ("t1", (256,)), ("t2", (128, 32)), ("t3", (1000,))]


@dataclass
class Workload:
    """One synthetic workload: a tensor table plus optimizer settings."""
    name: str
    tensors: list
    W: int
    chunk: int
    grad: str                 # "f32", "bf16" or "philox" (generated in-kernel)
    grad_std: float
    fan_in_scaled: bool = False
    heavy_every: int = 0      # tensors with l % heavy_every == heavy_every-1 are Student-t
    heavy_scale: float = 1e-3
    warmup_steps: int = 10
    compress_steps: int = 10
    seed: int = 0
    param_std: float = 2e-2
    hp: dict = field(default_factory=lambda: dict(
        lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-6, weight_decay=0.01,
        coeff_min=0.01, coeff_max=10.0, coeff_ema=0.9,
        factor_min=0.5, factor_max=4.0, factor_threshold=0.1))

    # derived -------------------------------------------------------------
    @property
    def numels(self):
        return np.array([int(np.prod(s)) for _, s in self.tensors], dtype=np.int64)

    @property
    def offsets(self):
        n = self.numels
        return np.concatenate([[0], np.cumsum(n)[:-1]]).astype(np.int64)

    @property
    def N(self) -> int:
        return int(self.numels.sum())

    @property
    def L(self) -> int:
        return len(self.tensors)

    @property
    def K(self) -> int:
        return -(-self.N // self.chunk)

    @property
    def layer_std(self) -> np.ndarray:
        """Per-tensor gradient std in binary32: std / sqrt(fan_in) for 2-D
        [out, in] tensors when fan-in scaling is on, else std."""
        out = np.empty(self.L, dtype=np.float32)
        base = np.float32(self.grad_std)
        for l, (_, shape) in enumerate(self.tensors):
            if self.fan_in_scaled and len(shape) == 2:
                out[l] = base / np.sqrt(np.float32(shape[1]))
            else:
                out[l] = base
        return out

    @property
    def layer_heavy(self) -> np.ndarray:
        h = np.zeros(self.L, dtype=np.uint8)
        if self.heavy_every:
            h[self.heavy_every - 1::self.heavy_every] = 1
        return h


def workloads():
    """The five workloads, by name."""
    return {
        "tiny": Workload("tiny", toy_tensors(), W=4, chunk=256, grad="f32",
                         grad_std=1e-2, warmup_steps=5, compress_steps=5, seed=0),
        "base": Workload("base", bert_tensors(12, 768, 3072, 30522), W=8, chunk=2048,
                         grad="f32", grad_std=1e-3, warmup_steps=10, compress_steps=10),
        "large": Workload("large", bert_tensors(24, 1024, 4096, 30522), W=16, chunk=4096,
                          grad="f32", grad_std=1e-3, fan_in_scaled=True,
                          warmup_steps=10, compress_steps=100),
        "large_w32": Workload("large_w32", bert_tensors(24, 1024, 4096, 30522), W=32,
                              chunk=4096, grad="philox", grad_std=1e-3, fan_in_scaled=True,
                              heavy_every=5, heavy_scale=1e-3,
                              warmup_steps=50, compress_steps=50),
        "gpt2xl": Workload("gpt2xl", gpt2_tensors(48, 1600, 6400, 50257), W=8, chunk=8192,
                           grad="bf16", grad_std=1e-3, warmup_steps=10, compress_steps=50),
    }


def custom(name, tensors, W, chunk, grad="f32", grad_std=1e-2, **kw) -> Workload:
    return Workload(name, tensors, W=W, chunk=chunk, grad=grad, grad_std=grad_std, **kw)


# --------------------------------------------------------------------------
# native generator
# --------------------------------------------------------------------------

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile gen.c into _build/libworkload.so (gcc, host only)."""
    src = os.path.join(_HERE, "gen.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.POINTER
        u32, u64, i64, i32, f32 = (ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64,
                                   ctypes.c_int32, ctypes.c_float)
        L.wl_philox4x32_10.argtypes = [P(u32), P(u32), P(u32)]
        L.wl_uniform.argtypes = [u32]
        L.wl_uniform.restype = f32
        L.wl_log.argtypes = [f32]
        L.wl_log.restype = f32
        L.wl_sincos2pi.argtypes = [f32, P(f32), P(f32)]
        L.wl_box_muller.argtypes = [u32, u32, P(f32), P(f32)]
        L.wl_normal4.argtypes = [u64, u32, u32, u32, u32, P(f32)]
        L.wl_student_t3.argtypes = [u64, i64, u32, u32]
        L.wl_student_t3.restype = f32
        L.wl_bf16_rne.argtypes = [f32]
        L.wl_bf16_rne.restype = ctypes.c_uint16
        gen_args = [u64, i64, i32, i64, i32, ctypes.c_void_p, ctypes.c_void_p,
                    ctypes.c_void_p, ctypes.c_void_p, f32, ctypes.c_void_p]
        L.wl_gen_grads_f32.argtypes = gen_args
        L.wl_gen_grads_bf16.argtypes = gen_args
        L.wl_gen_params.argtypes = [u64, i64, i64, f32, ctypes.c_void_p]
        L.wl_gen_grads_range_f32.argtypes = [u64, i64, i32, i64, i64, i32, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             f32, ctypes.c_void_p]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def philox(ctr, key):
    c = (ctypes.c_uint32 * 4)(*[int(v) & 0xFFFFFFFF for v in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(v) & 0xFFFFFFFF for v in key])
    o = (ctypes.c_uint32 * 4)()
    lib().wl_philox4x32_10(c, k, o)
    return list(o)


def normal4(seed, c0, c1, c2, c3):
    z = (ctypes.c_float * 4)()
    lib().wl_normal4(seed, c0, c1, c2, c3, z)
    return np.array(list(z), dtype=np.float32)


def gen_params(wl: Workload, lo: int = 0, hi: int | None = None) -> np.ndarray:
    hi = wl.N if hi is None else hi
    out = np.empty(hi - lo, dtype=np.float32)
    lib().wl_gen_params(wl.seed, lo, hi, wl.param_std, _ptr(out))
    return out


def gen_grads(wl: Workload, t: int, w: int, N: int | None = None,
              bf16_bits: bool = False) -> np.ndarray:
    """Gradients of worker w at global step t for elements [0, N).  Returns
    binary32 values, or raw bf16 bit patterns (uint16) when bf16_bits."""
    N = wl.N if N is None else N
    off, num = wl.offsets, wl.numels
    std, heavy = wl.layer_std, wl.layer_heavy
    if bf16_bits:
        out = np.empty(N, dtype=np.uint16)
        f = lib().wl_gen_grads_bf16
    else:
        out = np.empty(N, dtype=np.float32)
        f = lib().wl_gen_grads_f32
    f(wl.seed, t, w, N, wl.L, _ptr(off), _ptr(num), _ptr(std), _ptr(heavy),
      wl.heavy_scale, _ptr(out))
    return out


def grad_tables(wl: Workload):
    """The per-tensor arrays the gradient generator reads (offsets, sizes,
    std, Student-t flags), for callers that generate many ranges of one
    workload."""
    return (wl.offsets, wl.numels, wl.layer_std, wl.layer_heavy)


def gen_grads_range(wl: Workload, t: int, w: int, lo: int, hi: int, tables=None) -> np.ndarray:
    """Binary32 gradients of worker w at step t for elements [lo, hi) (the
    bf16 workload's values before rounding to bf16).  tables: the workload's
    grad_tables(), if the caller keeps them."""
    out = np.empty(hi - lo, dtype=np.float32)
    off, num, std, heavy = grad_tables(wl) if tables is None else tables
    lib().wl_gen_grads_range_f32(wl.seed, t, w, lo, hi, len(off), _ptr(off), _ptr(num), _ptr(std),
                                 _ptr(heavy), wl.heavy_scale, _ptr(out))
    return out


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Binary32 values rounded to bf16 (nearest even) and widened back."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.view(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to binary32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def grads_for_step(wl: Workload, t: int, ld: int | None = None) -> np.ndarray:
    """All W workers' gradients at step t as a [W, ld] binary32 array (the
    bf16 workload's values are the widened bf16 values).  Columns >= N are 0."""
    ld = wl.N if ld is None else ld
    g = np.zeros((wl.W, ld), dtype=np.float32)
    for w in range(wl.W):
        if wl.grad == "bf16":
            g[w, :wl.N] = bf16_bits_to_f32(gen_grads(wl, t, w, bf16_bits=True))
        else:
            g[w, :wl.N] = gen_grads(wl, t, w)
    return g
