"""GPU side of the full-size whole-run parity tests (test helper): runs a
plan's whole step sequence through the C ABI on cuda:0, gathers the sampled
elements, words and chunk scales, and compares them with the oracle's runs
(tests/fullrun.py), which it starts in spawned processes so that they
compute while the GPU runs.  No value on the oracle side comes from the GPU.
"""
import concurrent.futures as cf
import gc
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import communication_compressed_optimizer_gb300 as pkg
import fullrun
from harness import PARAM_TOL, STATE_TOL, close_scalar, layers_of


def _device_grads(wl, g, t):
    if g is not None and not isinstance(g, pkg.PhiloxGrads):
        pkg.gen_grads(g, t, wl.seed, layers_of(wl), wl.layer_std, None, wl.heavy_scale)
    return g


def _gpu_run(wl, runs, pl):
    """The configuration's whole run on the GPU; per-step reads of the
    sampled words, scales and per-tensor scalars, full sampled state at the
    checkpoints.  Returns (per-step records, checkpoints)."""
    N, W, C = wl.N, wl.W, wl.chunk
    lo_hi = [(k0 * C, min((k1 + 1) * C, N)) for k0, k1 in runs]
    elem = np.concatenate([np.arange(lo, hi) for lo, hi in lo_hi])
    words = np.concatenate([np.arange(lo // 32, -(-hi // 32)) for lo, hi in lo_hi])
    chunks = np.concatenate([np.arange(k0, k1 + 1) for k0, k1 in runs])
    it_e = torch.from_numpy(elem).cuda()
    it_w = torch.from_numpy(words).cuda()
    it_k = torch.from_numpy(chunks).cuda()

    x = torch.empty(N, device="cuda")
    pkg.gen_params(x, 0, N, wl.param_std, wl.seed)
    opt = pkg.OneBitLamb(x, layers_of(wl), W, C, **dict(wl.hp, variant=pl.get("variant", 0),
                                                          error_storage=pl.get("error_storage", 0)))
    if wl.grad == "philox":
        g = pkg.PhiloxGrads(wl.seed, wl.layer_std, wl.layer_heavy, wl.heavy_scale)
    else:
        q = 8 if wl.grad == "bf16" else 4
        ld = -(-N // q) * q
        g = torch.empty((W, ld), dtype=torch.int16 if wl.grad == "bf16" else torch.float32,
                        device="cuda")

    def snapshot():
        s = opt.state()                         # dense m brought up to date
        # error buffers widened to binary32 (exact for bfloat16 storage)
        return dict(x=x[it_e].cpu().numpy(), m=s["m"][it_e].cpu().numpy(),
                    v=s["v"][it_e].cpu().numpy(), v_fresh=s["v_fresh"][it_e].cpu().numpy(),
                    e_s=s["e_s"][it_e].float().cpu().numpy(),
                    e_w=s["e_w"][:, it_e].float().cpu().numpy())

    steps, cps = [], {}
    n_warm, n_comp = pl["n_warm"], pl["n_comp"]
    for step in range(n_warm + n_comp):
        if step == n_warm:
            opt.freeze_variance()
            if "freeze" in pl["checkpoints"]:
                cps["freeze"] = snapshot()
        gs = _device_grads(wl, g, step)
        if step < n_warm:
            opt.warmup_step(gs)
        else:
            opt.compress_step(gs)
        s = opt.state(sync=False)
        rec = {k: s[k].cpu().numpy() for k in ("c_cur", "c_bar")}
        if step < n_warm:
            rec.update(Sx=s["Sx"].cpu().numpy(), Su=s["Su"].cpu().numpy())
        else:
            rec.update(R=s["R_last"].cpu().numpy(), r_prev=s["r_prev"].cpu().numpy(),
                       signs_s=s["signs_s"][it_w].cpu().numpy().view(np.uint32),
                       scale_s=s["scale_s"][it_k].cpu().numpy(),
                       signs_w=s["signs_w"][:, it_w].cpu().numpy().view(np.uint32),
                       scale_w=s["scale_w"][:, it_k].cpu().numpy())
        steps.append(rec)
        if step in pl["checkpoints"]:
            cps[step] = snapshot()
    opt.check_status()
    opt.close()
    del g, x
    return steps, cps


def _bits_differ(a, b):
    return int(np.sum(np.ascontiguousarray(a).view(np.uint32)
                      != np.ascontiguousarray(b).view(np.uint32)))


def _close_per_frag(a, b, frags, tol):
    """Vectors compared per tensor fragment: max|a-b| <= tol max|b|."""
    for l, lo, n, _ in frags:
        x = a[..., lo:lo + n].astype(np.float64)
        y = b[..., lo:lo + n].astype(np.float64)
        d = np.max(np.abs(x - y))
        if d != 0 and d > tol * np.max(np.abs(y)):
            return False, l
    return True, None


def run_and_compare(name, wl, runs, pl):
    """The plan's whole run on the GPU and, in spawned processes at the same
    time, the oracle's runs; then every compared value, run by run.  Returns
    the number of tensors covered completely."""
    N, W, C = wl.N, wl.W, wl.chunk
    gc.collect()
    torch.cuda.empty_cache()              # earlier full-size tests' cached blocks
    free, _ = torch.cuda.mem_get_info()
    gbytes = {"f32": 4, "bf16": 2, "philox": 0}[wl.grad]
    need = pkg.workspace_bytes(layers_of(wl), W, C) + 4 * N + gbytes * W * (N + 8)
    if need > 0.9 * free:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory")

    # the oracle's runs start first, in spawned processes (no CUDA state is
    # inherited), and compute while the GPU runs
    n_proc = max(1, min(16, os.cpu_count() or 1))
    parts = fullrun.groups(wl, runs, 2 * n_proc)
    with cf.ProcessPoolExecutor(max_workers=n_proc, mp_context=mp.get_context("spawn")) as ex:
        futs = [ex.submit(fullrun.oracle_runs, wl, runs, pl, p) for p in parts]
        g_steps, g_cps = _gpu_run(wl, runs, pl)
        orc = {}
        for f in futs:
            orc.update(f.result())

    # ---- compare, run by run ----------------------------------------------------
    n_warm = pl["n_warm"]
    diffs = 0
    e0 = w0 = k0c = 0                     # this run's offsets in the gathered arrays
    covered = 0
    for r, (k0, k1) in enumerate(runs):
        lo, hi, frags = fullrun.run_table(wl, k0, k1)
        n, nw, nk = hi - lo, -(-(hi - lo) // 32), k1 - k0 + 1
        whole = [(j, f) for j, f in enumerate(frags) if f[3]]
        covered += len(whole)
        rec = orc[r]
        for step, (gs, os_) in enumerate(zip(g_steps, rec["steps"])):
            where = f"{name} run {r} (chunks {k0}..{k1}) step {step}"
            keys = ("Sx", "Su", "c_cur", "c_bar") if step < n_warm else ("R", "r_prev", "c_cur", "c_bar")
            for j, (l, _, _, _) in whole:
                for k in keys:
                    a, b = gs[k][l], os_[k][j]
                    assert close_scalar(a, b), (where, k, wl.tensors[l][0], a, b)
                    diffs += int(np.float32(a).view(np.uint32) != np.float32(b).view(np.uint32))
            if step >= n_warm:
                np.testing.assert_array_equal(gs["signs_s"][w0:w0 + nw], os_["signs_s"], err_msg=where)
                np.testing.assert_array_equal(gs["signs_w"][:, w0:w0 + nw], os_["signs_w"],
                                              err_msg=where)
                for k in ("scale_s", "scale_w"):
                    a = gs[k][..., k0c:k0c + nk]
                    assert close_scalar(a, os_[k]), (where, k)
                    diffs += _bits_differ(a, os_[k])
        for cp, ost in rec["checkpoints"].items():
            gst = g_cps[cp]
            where = f"{name} run {r} (chunks {k0}..{k1}) checkpoint {cp}"
            for k in ("m", "v", "v_fresh", "e_s", "e_w"):
                a = gst[k][..., e0:e0 + n]
                ok, l = _close_per_frag(a, ost[k], frags, STATE_TOL)
                assert ok, (where, k, l)
                diffs += _bits_differ(a, ost[k])
            for j, (l, lo_, nl, _) in whole:
                a, b = gst["x"][e0 + lo_:e0 + lo_ + nl], ost["x"][lo_:lo_ + nl]
                d = np.max(np.abs(a.astype(np.float64) - b))
                assert d == 0 or d <= PARAM_TOL * np.max(np.abs(b)), (where, "x", wl.tensors[l][0])
                diffs += _bits_differ(a, b)
        e0 += n
        w0 += nw
        k0c += nk
    assert diffs == 0, f"{diffs} compared floats differ in some bit"
    return covered
