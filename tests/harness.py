"""Shared pieces of the GPU parity tests: run one workload through the C ABI
(via the Python binding) and through the CPU oracle on the same seeded
inputs, and compare state after every step.

Comparison rules (1-bit LAMB hot path):
  sign words and chunk/layer indexing: bit-exact;
  chunk scales and per-tensor scalars: |a - b| <= 1e-5 |b|;
  vectors: per tensor, max |a - b| <= tol * max |b| (1e-4 for parameters).
"""
from __future__ import annotations

import numpy as np
import torch

import communication_compressed_optimizer_gb300 as pkg
import oracle
import workload

SCALAR_TOL = 1e-5
PARAM_TOL = 1e-4
STATE_TOL = 1e-5


def layers_of(wl):
    return list(zip(wl.offsets.tolist(), wl.numels.tolist()))


def grad_ld(wl):
    q = 8 if wl.grad == "bf16" else 4
    return -(-wl.N // q) * q


def device_grads(wl, t, ld):
    """GPU gradients of step t: the same seeded values the oracle gets."""
    if wl.grad == "philox":
        return pkg.PhiloxGrads(wl.seed, wl.layer_std, wl.layer_heavy, wl.heavy_scale)
    if wl.grad == "bf16":
        g = np.zeros((wl.W, ld), np.uint16)
        for w in range(wl.W):
            g[w, :wl.N] = workload.gen_grads(wl, t, w, bf16_bits=True)
        return torch.from_numpy(g.view(np.int16)).cuda()
    return torch.from_numpy(workload.grads_for_step(wl, t, ld)).cuda()


def host_grads(wl, t):
    return workload.grads_for_step(wl, t)


def close_scalar(a, b, tol=SCALAR_TOL):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    ok = (np.abs(a - b) <= tol * np.abs(b)) | both_nan | (a == b)
    return bool(np.all(ok))


def close_vec_per_tensor(a, b, offsets, numels, tol):
    """Per tensor l (contiguous from 0): max|a - b| <= tol max|b| over the
    tensor's elements (a NaN difference passes here; NaN positions are
    compared bit for bit elsewhere).  Returns (ok, worst relative error)."""
    offsets = np.asarray(offsets, np.int64)
    n = int(offsets[-1] + np.asarray(numels, np.int64)[-1])
    x = np.asarray(a[:n], np.float64)
    y = np.asarray(b[:n], np.float64)
    with np.errstate(invalid="ignore"):
        d = np.maximum.reduceat(np.abs(x - y), offsets)
        ref = np.maximum.reduceat(np.abs(y), offsets)
        bad = (d > tol * ref) & (d != 0)
        if np.any(bad):
            l = int(np.argmax(bad))
            return False, float(d[l] / ref[l] if ref[l] else np.inf)
        rel = np.where(ref != 0, d / np.where(ref != 0, ref, 1.0), 0.0)
    rel = rel[~np.isnan(rel)]
    return True, float(rel.max()) if rel.size else 0.0


class Pair:
    """GPU optimizer and CPU oracle over the same workload."""

    def __init__(self, wl, check_finite=0, variant=0, error_storage=0):
        self.wl = wl
        self.x0 = workload.gen_params(wl)
        self.x = torch.from_numpy(self.x0.copy()).cuda()
        hp = dict(wl.hp, check_finite=check_finite, variant=variant, error_storage=error_storage)
        self.gpu = pkg.OneBitLamb(self.x, layers_of(wl), wl.W, wl.chunk, **hp)
        self.orc = oracle.Oracle(wl.offsets, wl.numels, wl.W, wl.chunk, wl.hp, self.x0,
                                 variant=variant, err_bf16=error_storage)
        self.ld = grad_ld(wl)
        self.t = 0

    def warmup(self):
        self.gpu.warmup_step(device_grads(self.wl, self.t, self.ld))
        self.orc.warmup_step(host_grads(self.wl, self.t))
        self.t += 1

    def freeze(self):
        self.gpu.freeze_variance()
        self.orc.freeze()

    def compress(self):
        self.gpu.compress_step(device_grads(self.wl, self.t, self.ld))
        self.orc.compress_step(host_grads(self.wl, self.t))
        self.t += 1

    def gpu_state(self):
        torch.cuda.synchronize()
        s = self.gpu.state()
        N, W = self.wl.N, self.wl.W
        nw = -(-N // 32)
        out = {k: s[k].cpu().numpy() for k in ("m", "v", "v_fresh", "c_bar", "r_prev",
                                                 "c_cur", "R_last", "Sx", "Su", "scale_s")}
        # error buffers widened to binary32 (exact for bfloat16 storage)
        out["e_s"] = s["e_s"].float().cpu().numpy()
        out["e_w"] = s["e_w"].float().cpu().numpy()
        out["scale_w"] = s["scale_w"].cpu().numpy()
        out["signs_w"] = s["signs_w"].cpu().numpy().view(np.uint32)
        out["signs_s"] = s["signs_s"].cpu().numpy().view(np.uint32)
        out["x"] = self.x.cpu().numpy()
        out["nw"] = nw
        out["t"], out["stage"], out["n_warmup"] = s["t"], s["stage"], s["n_warmup"]
        return out

    def compare(self, where=""):
        """Asserts parity of the full state; returns the number of float
        elements that differ in any bit (expected 0)."""
        g = self.gpu_state()
        o = self.orc
        wl = self.wl
        N, nw = wl.N, g["nw"]
        off, num = wl.offsets, wl.numels
        assert g["t"] == o.t and g["stage"] == o.stage and g["n_warmup"] == o.n_warm, where
        # padding stays zero
        for k in ("m", "v", "v_fresh", "e_s"):
            assert not np.any(g[k][N:]), (where, k)
        assert not np.any(g["e_w"][:, N:]), where
        if o.stage == 1:
            np.testing.assert_array_equal(g["signs_w"][:, :nw], o.signs_w, err_msg=where)
            np.testing.assert_array_equal(g["signs_s"][:nw], o.signs_s, err_msg=where)
            assert not np.any(g["signs_w"][:, nw:]) and not np.any(g["signs_s"][nw:]), where
            assert close_scalar(g["scale_w"], o.scale_w), where
            assert close_scalar(g["scale_s"], o.scale_s), where
            assert close_scalar(g["R_last"], o.R), where
            assert close_scalar(g["r_prev"], o.r_prev), where
        else:
            assert close_scalar(g["Sx"], o.Sx), where
            assert close_scalar(g["Su"], o.Su), where
        assert close_scalar(g["c_cur"], o.c_cur), where
        assert close_scalar(g["c_bar"], o.c_bar), where
        ok, worst = close_vec_per_tensor(g["x"], o.x, off, num, PARAM_TOL)
        assert ok, (where, "x", worst)
        for k in ("m", "v", "v_fresh", "e_s"):
            ok, worst = close_vec_per_tensor(g[k][:N], getattr(o, k), off, num, STATE_TOL)
            assert ok, (where, k, worst)
        for w in range(wl.W):
            ok, worst = close_vec_per_tensor(g["e_w"][w, :N], o.e_w[w], off, num, STATE_TOL)
            assert ok, (where, "e_w", w, worst)
        diff = 0
        for k, ov in (("x", o.x), ("m", o.m), ("v", o.v), ("v_fresh", o.v_fresh), ("e_s", o.e_s)):
            diff += int(np.sum(g[k][:N].view(np.uint32) != ov.view(np.uint32)))
        diff += int(np.sum(g["e_w"][:, :N].view(np.uint32) != o.e_w.view(np.uint32)))
        return diff
