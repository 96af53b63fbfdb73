"""1-bit LAMB data-parallel hot path on one GB300 (sm_103a).

Python binding of the lamb1b C ABI (``include/lamb1b.h``).  PyTorch supplies
device memory and streams; every step of the optimizer runs in the CUDA
kernels of ``liblamb1b.so`` (``csrc/``).  There is no CPU fallback: building
or loading failures raise.

Method: Li et al., "1-bit LAMB: Communication Efficient Large-Scale
Large-Batch Training with LAMB's Convergence Speed" (arXiv 2104.06069):
LAMB warmup, variance freeze, then error-compensated 1-bit compressed
momentum with a compressed allreduce (gather / average / scatter) among W
data-parallel workers, here held side by side in one GPU's memory.
"""
from __future__ import annotations

import ctypes

from . import _abi
from ._abi import GRAD_BF16, GRAD_F32, GRAD_PHILOX, Lamb1bError  # noqa: F401

__all__ = ["OneBitLamb", "PhiloxGrads", "gen_grads", "gen_params", "Lamb1bError",
           "workspace_bytes", "library_path"]


def library_path() -> str:
    return _abi.lib_path()


def _torch():
    import torch
    return torch


def _layers_array(layers):
    arr = (_abi.Layer * len(layers))()
    for i, (o, n) in enumerate(layers):
        arr[i].offset, arr[i].numel = int(o), int(n)
    return arr


def _hparams(W, chunk, hp):
    h = _abi.HParams()
    h.W, h.chunk = int(W), int(chunk)
    for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "coeff_min", "coeff_max",
              "coeff_ema", "factor_min", "factor_max", "factor_threshold"):
        setattr(h, k, float(hp[k]))
    h.check_finite = int(hp.get("check_finite", 0))
    h.variant = {"lamb": 0, "adam": 1}.get(hp.get("variant", 0), hp.get("variant", 0))
    h.error_storage = {"f32": 0, "bf16": 1}.get(hp.get("error_storage", 0),
                                                hp.get("error_storage", 0))
    return h


DEFAULT_HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-6, weight_decay=0.01,
                  coeff_min=0.01, coeff_max=10.0, coeff_ema=0.9,
                  factor_min=0.5, factor_max=4.0, factor_threshold=0.1, check_finite=0)


def workspace_bytes(layers, W, chunk, **hp) -> int:
    h = _hparams(W, chunk, {**DEFAULT_HP, **hp})
    arr = _layers_array(layers)
    return int(_abi.load().lamb1b_workspace_bytes(arr, len(layers), ctypes.byref(h)))


def _stream_handle(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class PhiloxGrads:
    """Gradients drawn inside the kernels from the seeded workload definition
    (``include/lamb1b_gen.h``): layer_std[l] * N(0,1), or heavy_scale *
    Student-t(3) on tensors with layer_heavy[l] != 0."""

    def __init__(self, seed, layer_std, layer_heavy=None, heavy_scale=1e-3, device="cuda"):
        torch = _torch()
        self.seed = int(seed)
        self.layer_std = torch.as_tensor(layer_std, dtype=torch.float32).to(device).contiguous()
        self.layer_heavy = (None if layer_heavy is None else
                            torch.as_tensor(layer_heavy, dtype=torch.uint8).to(device).contiguous())
        self.heavy_scale = float(heavy_scale)


def _grads_desc(grads, N):
    torch = _torch()
    d = _abi.GradsDesc()
    if isinstance(grads, PhiloxGrads):
        d.kind = GRAD_PHILOX
        d.seed = grads.seed
        d.layer_std = grads.layer_std.data_ptr()
        d.layer_heavy = grads.layer_heavy.data_ptr() if grads.layer_heavy is not None else None
        d.heavy_scale = grads.heavy_scale
        return d
    if not isinstance(grads, torch.Tensor) or grads.dim() != 2 or not grads.is_cuda:
        raise TypeError("grads: a [W, ld] CUDA tensor (float32 or bfloat16) or PhiloxGrads")
    if grads.stride(1) != 1:
        raise ValueError("grads: rows must be contiguous")
    if grads.dtype == torch.float32:
        d.kind = GRAD_F32
    elif grads.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        d.kind = GRAD_BF16
    else:
        raise TypeError(f"grads dtype {grads.dtype}")
    d.ptr = grads.data_ptr()
    d.ld = grads.stride(0)
    return d


class OneBitLamb:
    """One optimizer context over a flat float32 parameter tensor.

    ``layers`` is a list of (offset, numel), one per tensor, contiguous from
    0.  ``W`` virtual workers, compression chunk ``chunk``.  Hyper-parameters
    as in ``lamb1b_hparams``.  All calls are asynchronous on ``stream``
    (default: the current torch stream)."""

    def __init__(self, params, layers, W, chunk, stream=None, **hp):
        torch = _torch()
        self._lib = _abi.load()
        if (not isinstance(params, torch.Tensor) or params.dtype != torch.float32
                or not params.is_cuda or not params.is_contiguous() or params.dim() != 1):
            raise TypeError("params: contiguous 1-D float32 CUDA tensor")
        self.params = params
        self.layers = [(int(o), int(n)) for o, n in layers]
        self.W, self.chunk = int(W), int(chunk)
        self.hp = {**DEFAULT_HP, **hp}
        self._h = _hparams(W, chunk, self.hp)
        self._arr = _layers_array(self.layers)
        nbytes = self._lib.lamb1b_workspace_bytes(self._arr, len(self.layers), ctypes.byref(self._h))
        if nbytes == 0:
            raise Lamb1bError("lamb1b_workspace_bytes", _abi.ERR_ARG)
        self.workspace = torch.empty(int(nbytes), dtype=torch.uint8, device=params.device)
        self._ctx = ctypes.c_void_p()
        _abi.check("lamb1b_init", self._lib.lamb1b_init(
            ctypes.byref(self._ctx), self._arr, len(self.layers), ctypes.byref(self._h),
            ctypes.c_void_p(params.data_ptr()), ctypes.c_void_p(self.workspace.data_ptr()),
            int(nbytes), _stream_handle(stream)))
        self.N = params.numel()
        self.K = -(-self.N // self.chunk)

    # -- steps -------------------------------------------------------------
    def warmup_step(self, grads, stream=None):
        d = _grads_desc(grads, self.N)
        _abi.check("lamb1b_warmup_step",
                   self._lib.lamb1b_warmup_step(self._ctx, ctypes.byref(d), _stream_handle(stream)))

    def freeze_variance(self, stream=None):
        _abi.check("lamb1b_freeze_variance",
                   self._lib.lamb1b_freeze_variance(self._ctx, _stream_handle(stream)))

    def compress_step(self, grads, stream=None):
        d = _grads_desc(grads, self.N)
        _abi.check("lamb1b_compress_step",
                   self._lib.lamb1b_compress_step(self._ctx, ctypes.byref(d), _stream_handle(stream)))

    def compress_step_host(self, host_grads, staging, words_out=None, scales_out=None, stream=None,
                           copy_stream=None):
        """One compression step whose gradients are in pinned host memory.

        host_grads: a pinned CPU tensor [W, ld] (float32, or bfloat16 bits as
        bfloat16/int16); staging: a CUDA tensor of the same shape, strides and
        dtype that receives them; words_out / scales_out: None or pinned CPU
        tensors of ceil(N/32) int32 and K float32 that receive the step's
        server message.  The copy runs on copy_stream (default: the step's
        stream); with two staging tensors used in turn and a separate
        copy_stream, a step's copy overlaps the previous step's kernels."""
        torch = _torch()
        if (not isinstance(host_grads, torch.Tensor) or host_grads.is_cuda
                or not host_grads.is_pinned()):
            raise TypeError("host_grads: a pinned CPU tensor [W, ld]")
        if (not isinstance(staging, torch.Tensor) or not staging.is_cuda
                or staging.shape != host_grads.shape or staging.stride() != host_grads.stride()
                or staging.dtype != host_grads.dtype):
            raise ValueError("staging: a CUDA tensor with host_grads' shape, strides and dtype")
        d = _grads_desc(staging, self.N)
        d.ptr = host_grads.data_ptr()
        outs = []
        for t, n, dt in ((words_out, -(-self.N // 32), (torch.int32, torch.uint32)),
                         (scales_out, self.K, (torch.float32,))):
            if t is None:
                outs.append(None)
                continue
            if t.is_cuda or not t.is_pinned() or t.dtype not in dt or t.numel() < n or not t.is_contiguous():
                raise ValueError("words_out / scales_out: pinned contiguous CPU tensors of the message's size")
            outs.append(ctypes.c_void_p(t.data_ptr()))
        _abi.check("lamb1b_compress_step_host",
                   self._lib.lamb1b_compress_step_host(
                       self._ctx, ctypes.byref(d), ctypes.c_void_p(staging.data_ptr()), outs[0], outs[1],
                       _stream_handle(stream),
                       _stream_handle(copy_stream if copy_stream is not None else stream)))

    def check_status(self, stream=None):
        _abi.check("lamb1b_check_status",
                   self._lib.lamb1b_check_status(self._ctx, _stream_handle(stream)))

    def set_counters(self, t, n_warmup, stage):
        _abi.check("lamb1b_set_counters",
                   self._lib.lamb1b_set_counters(self._ctx, int(t), int(n_warmup), int(stage)))

    def set_fault_injection(self, skip_copy=-1, wait_tries=0):
        """Testing hook: the first CTA of later compression steps leaves out
        bulk copy number skip_copy (-1: none); that CTA's copy waits give up
        after wait_tries try_wait calls (0: the default; other CTAs always
        keep the default).  A step that gave up is reported by check_status()
        as a timeout."""
        _abi.check("lamb1b_set_fault_injection",
                   self._lib.lamb1b_set_fault_injection(self._ctx, int(skip_copy), int(wait_tries)))

    def set_trace_events(self, events):
        """events: 4 torch.cuda.Event objects (or None to stop tracing).
        Each later step records them before its first kernel and after each
        of its three kernels, on the step's stream."""
        if events is None:
            _abi.check("lamb1b_set_trace_events",
                       self._lib.lamb1b_set_trace_events(self._ctx, None, 0))
            return
        for e in events:
            if getattr(e, "cuda_event", 0) == 0:
                e.record()          # torch creates the underlying event lazily
        arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
        self._trace_events = (events, arr)
        _abi.check("lamb1b_set_trace_events",
                   self._lib.lamb1b_set_trace_events(self._ctx, arr, 4))

    # -- state ---------------------------------------------------------------
    def state_raw(self) -> _abi.State:
        s = _abi.State()
        _abi.check("lamb1b_state_view", self._lib.lamb1b_state_view(self._ctx, ctypes.byref(s)))
        return s

    def sync_momentum(self, stream=None):
        """Write the dense momentum m from the last compression step's server
        sign words and chunk scales (a no-op before the first one)."""
        _abi.check("lamb1b_sync_momentum",
                   self._lib.lamb1b_sync_momentum(self._ctx, _stream_handle(stream)))

    def state(self, sync=True) -> dict:
        """Views (not copies) of the state inside the workspace, as torch
        tensors, plus the counters.  sync: first bring the dense momentum
        up to date (sync_momentum on the current stream)."""
        torch = _torch()
        if sync:
            self.sync_momentum()
        s = self.state_raw()
        base = self.workspace.data_ptr()

        def view(ptr, n, dtype, shape=None):
            off = ptr - base
            nbytes = n * torch.empty((), dtype=dtype).element_size()
            t = self.workspace[off:off + nbytes].view(dtype)
            return t if shape is None else t.view(*shape)

        Np, K, WL, L, W = s.Np, s.K, s.words_ld, s.L, s.W
        f32, i32 = torch.float32, torch.int32
        et = torch.bfloat16 if self._h.error_storage == 1 else f32   # error buffers
        out = dict(
            m=view(s.m, Np, f32), v=view(s.v, Np, f32), v_fresh=view(s.v_fresh, Np, f32),
            e_s=view(s.e_s, Np, et), e_w=view(s.e_w, W * Np, et, (W, Np)),
            signs_w=view(s.signs_w, W * WL, i32, (W, WL)), signs_s=view(s.signs_s, WL, i32),
            scale_w=view(s.scale_w, W * K, f32, (W, K)), scale_s=view(s.scale_s, K, f32),
            c_bar=view(s.c_bar, L, f32), r_prev=view(s.r_prev, L, f32),
            c_cur=view(s.c_cur, L, f32), R_last=view(s.R_last, L, f32),
            Sx=view(s.Sx, L, f32), Su=view(s.Su, L, f32))
        out.update(N=s.N, Np=Np, K=K, words_ld=WL, t=s.t, n_warmup=s.n_warmup, stage=s.stage)
        return out

    def close(self):
        if getattr(self, "_ctx", None) and self._ctx.value:
            self._lib.lamb1b_destroy(self._ctx)
            self._ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gen_grads(out, t, seed, layers, layer_std, layer_heavy=None, heavy_scale=1e-3, stream=None):
    """Fill out[W, ld] (float32, or bfloat16/int16 for bf16 bit patterns) with
    the seeded workload's gradients of step t (``lamb1b_gen_grads``)."""
    import numpy as np
    torch = _torch()
    L = len(layers)
    off = np.ascontiguousarray([o for o, _ in layers], dtype=np.int64)
    num = np.ascontiguousarray([n for _, n in layers], dtype=np.int64)
    std = np.ascontiguousarray(layer_std, dtype=np.float32)
    heavy = None if layer_heavy is None else np.ascontiguousarray(layer_heavy, dtype=np.uint8)
    bf16 = out.dtype != torch.float32
    rc = _abi.load().lamb1b_gen_grads(
        ctypes.c_void_p(out.data_ptr()), out.stride(0), out.shape[0], int(bf16), int(seed), int(t),
        off.ctypes.data_as(ctypes.c_void_p), num.ctypes.data_as(ctypes.c_void_p), L,
        std.ctypes.data_as(ctypes.c_void_p),
        None if heavy is None else heavy.ctypes.data_as(ctypes.c_void_p),
        float(heavy_scale), _stream_handle(stream))
    _abi.check("lamb1b_gen_grads", rc)


def gen_params(out, lo, hi, std, seed, stream=None):
    rc = _abi.load().lamb1b_gen_params(ctypes.c_void_p(out.data_ptr()), int(lo), int(hi),
                                       float(std), int(seed), _stream_handle(stream))
    _abi.check("lamb1b_gen_params", rc)
