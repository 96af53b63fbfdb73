"""GPU parity at the full workload sizes (BERT-Base, BERT-Large W=16,
BERT-Large W=32 with in-kernel gradients, GPT-2-XL with bf16 gradients), in
the launch configuration the benchmark times.

One compression step runs on the GPU from a seeded synthetic mid-training
state (parameters, momentum, frozen and fresh second moments, every worker's
error, the server error, per-tensor c_bar and r_prev).  The oracle runs the
same step on a sample of whole chunks: every chunk that meets a small tensor
(so those tensors are covered completely), the first and last chunks and a
seeded random set.  Compared: every chunk-local output bit for bit / within
tolerance, and for completely covered tensors the max ratio, factor,
coefficient and updated parameters.  For the other tensors the GPU's max
ratio must bound the sampled ratios from above.
"""
import gc

import numpy as np
import pytest
import torch

import communication_compressed_optimizer_gb300 as pkg
import oracle
import workload
from harness import SCALAR_TOL, close_scalar, layers_of

pytestmark = pytest.mark.gpu

SEEDS = dict(m=101, v=102, v_fresh=103, e_s=104, e_w=1000, signs=105, scales=106)
STDS = dict(m=1e-3, v=1e-3, v_fresh=1e-3, e_s=1e-4, e_w=1e-4, signs=1.0, scales=1e-3)
STEP = 10


def host_normal(seed, std, lo, hi):
    out = np.empty(hi - lo, np.float32)
    workload.lib().wl_gen_params(seed, lo, hi, std, workload._ptr(out))
    return out


def c_bar_of(L):
    return (np.float32(0.25) + np.float32(0.05) * (np.arange(L) % 31)).astype(np.float32)


def r_prev_of(L):
    return (np.float32(0.8) + np.float32(0.01) * (np.arange(L) % 41)).astype(np.float32)


def sample_chunks(wl, small, n_random=12):
    C, K = wl.chunk, wl.K
    ks = {0, 1, K - 2, K - 1}
    for o, n in zip(wl.offsets, wl.numels):
        if n <= small:
            ks.update(range(o // C, (o + n - 1) // C + 1))
    rng = np.random.default_rng(7)
    ks.update(rng.integers(0, K, size=n_random).tolist())
    return np.array(sorted(ks), dtype=np.int64)


def fragments(wl, ks):
    """Local layer table of the sampled chunks laid end to end: each original
    tensor's intersection with each run of consecutive sampled chunks."""
    C, N = wl.chunk, wl.N
    frags = []   # (orig layer, local offset, numel, whole)
    local = 0
    runs = []
    start = ks[0]
    for a, b in zip(ks[:-1], ks[1:]):
        if b != a + 1:
            runs.append((start, a))
            start = b
    runs.append((start, ks[-1]))
    ends = wl.offsets + wl.numels
    for k0, k1 in runs:
        lo, hi = k0 * C, min((k1 + 1) * C, N)
        l = int(np.searchsorted(ends, lo, side="right"))
        while l < wl.L and wl.offsets[l] < hi:
            a, b = max(lo, wl.offsets[l]), min(hi, ends[l])
            whole = a == wl.offsets[l] and b == ends[l]
            frags.append((l, local + (a - lo), b - a, whole))
            l += 1
        local += hi - lo
    return frags, local


@pytest.mark.parametrize("name", ["base", "large", "large_w32", "gpt2xl"])
def test_full_size_compression_step_sampled(name):
    wl = workload.workloads()[name]
    N, W, C, K, L = wl.N, wl.W, wl.chunk, wl.K, wl.L
    gc.collect()
    torch.cuda.empty_cache()              # earlier full-size tests' cached blocks
    free, _ = torch.cuda.mem_get_info()
    gbytes = {"f32": 4, "bf16": 2, "philox": 0}[wl.grad]
    need = pkg.workspace_bytes(layers_of(wl), W, C) + 4 * N + gbytes * W * (N + 8)
    if need > 0.9 * free:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory")

    # ---- GPU: synthetic state, one compression step -------------------------
    x = torch.empty(N, device="cuda")
    pkg.gen_params(x, 0, N, wl.param_std, wl.seed)
    opt = pkg.OneBitLamb(x, layers_of(wl), W, C, **wl.hp)
    opt.freeze_variance()
    st = opt.state()
    for k in ("v", "v_fresh", "e_s"):
        pkg.gen_params(st[k], 0, N, STDS[k], SEEDS[k])
    # mid-training momentum: the last step's server message, in the packed
    # form a compression step keeps (random sign words, positive chunk scales)
    nwords = -(-N // 32)
    pkg.gen_params(st["signs_s"].view(torch.float32), 0, nwords, STDS["signs"], SEEDS["signs"])
    pkg.gen_params(st["scale_s"], 0, K, STDS["scales"], SEEDS["scales"])
    st["scale_s"][:K].abs_()
    st["v"][:N].mul_(st["v"][:N])
    st["v_fresh"][:N].mul_(st["v_fresh"][:N])
    for w in range(W):
        pkg.gen_params(st["e_w"][w], 0, N, STDS["e_w"], SEEDS["e_w"] + w)
    st["c_bar"].copy_(torch.from_numpy(c_bar_of(L)))
    st["r_prev"].copy_(torch.from_numpy(r_prev_of(L)))
    opt.set_counters(STEP, 0, 1)
    if wl.grad == "philox":
        g = pkg.PhiloxGrads(wl.seed, wl.layer_std, wl.layer_heavy, wl.heavy_scale)
    else:
        q = 8 if wl.grad == "bf16" else 4
        ld = -(-N // q) * q
        g = torch.empty((W, ld), dtype=torch.int16 if wl.grad == "bf16" else torch.float32,
                        device="cuda")
        pkg.gen_grads(g, STEP, wl.seed, layers_of(wl), wl.layer_std, None, wl.heavy_scale)
    opt.compress_step(g)
    torch.cuda.synchronize()
    del g

    # ---- host: the same step on the sampled chunks ----------------------------
    ks = sample_chunks(wl, small=2 * C)
    frags, NL = fragments(wl, ks)
    idx = np.concatenate([np.arange(k * C, min((k + 1) * C, N)) for k in ks])
    assert len(idx) == NL
    runs_lo = [(k * C, min((k + 1) * C, N)) for k in ks]

    def gather_host(fn):
        return np.concatenate([fn(lo, hi) for lo, hi in runs_lo])

    x0 = gather_host(lambda lo, hi: host_normal(wl.seed, wl.param_std, lo, hi))
    o = oracle.Oracle([f[1] for f in frags], [f[2] for f in frags], W, C, wl.hp, x0)
    def packed_m(lo, hi):
        q0, q1 = lo // 32, -(-hi // 32)
        words = host_normal(SEEDS["signs"], STDS["signs"], q0, q1).view(np.uint32)
        bits = np.unpackbits(words.view(np.uint8), bitorder="little")[lo - q0 * 32:hi - q0 * 32]
        sc = np.abs(host_normal(SEEDS["scales"], STDS["scales"], lo // C, lo // C + 1))[0]
        return np.where(bits == 1, sc, -sc).astype(np.float32)
    o.m[:] = gather_host(packed_m)
    v = gather_host(lambda lo, hi: host_normal(SEEDS["v"], STDS["v"], lo, hi))
    o.v[:] = v * v
    vf = gather_host(lambda lo, hi: host_normal(SEEDS["v_fresh"], STDS["v_fresh"], lo, hi))
    o.v_fresh[:] = vf * vf
    o.e_s[:] = gather_host(lambda lo, hi: host_normal(SEEDS["e_s"], STDS["e_s"], lo, hi))
    for w in range(W):
        o.e_w[w] = gather_host(lambda lo, hi: host_normal(SEEDS["e_w"] + w, STDS["e_w"], lo, hi))
    cb, rp = c_bar_of(L), r_prev_of(L)
    o.c_bar[:] = [cb[f[0]] for f in frags]
    o.r_prev[:] = [rp[f[0]] for f in frags]
    o.stage, o.t = 1, STEP
    gh = np.empty((W, NL), np.float32)
    for w in range(W):
        gw = gather_host(lambda lo, hi: workload.gen_grads_range(wl, STEP, w, lo, hi))
        gh[w] = workload.bf16_round(gw) if wl.grad == "bf16" else gw
    o.compress_step(gh)

    # ---- compare ---------------------------------------------------------------
    s = opt.state()
    it = torch.from_numpy(idx).cuda()
    wi = torch.from_numpy(np.concatenate([np.arange(k * C // 32, k * C // 32 + C // 32)
                                          for k in ks])).cuda()
    kk = torch.from_numpy(ks).cuda()
    nloc = -(-NL // 32)
    words_s = s["signs_s"][wi].cpu().numpy().view(np.uint32)[:nloc]
    np.testing.assert_array_equal(words_s, o.signs_s)
    words_w = s["signs_w"][:, wi].cpu().numpy().view(np.uint32)[:, :nloc]
    np.testing.assert_array_equal(words_w, o.signs_w)
    assert close_scalar(s["scale_w"][:, kk].cpu().numpy(), o.scale_w)
    assert close_scalar(s["scale_s"][kk].cpu().numpy(), o.scale_s)
    for name_, ov in (("m", o.m), ("e_s", o.e_s), ("v_fresh", o.v_fresh)):
        gv = s[name_][it].cpu().numpy()
        np.testing.assert_array_equal(gv.view(np.uint32), ov.view(np.uint32), err_msg=name_)
    np.testing.assert_array_equal(s["e_w"][:, it].cpu().numpy().view(np.uint32),
                                  o.e_w.view(np.uint32))
    R = s["R_last"].cpu().numpy()
    r = s["r_prev"].cpu().numpy()
    c = s["c_cur"].cpu().numpy()
    xg = x[it].cpu().numpy()
    n_whole = 0
    for j, (l, lo, n, whole) in enumerate(frags):
        if whole:
            n_whole += 1
            assert close_scalar(R[l], o.R[j]), (l, R[l], o.R[j])
            assert close_scalar(r[l], o.r_prev[j]), l
            assert close_scalar(c[l], o.c_cur[j]), l
            np.testing.assert_array_equal(xg[lo:lo + n].view(np.uint32),
                                          o.x[lo:lo + n].view(np.uint32), err_msg=str(l))
        else:
            assert R[l] >= o.R[j] * (1 - SCALAR_TOL), (l, R[l], o.R[j])
    assert n_whole >= 50
    opt.close()


@pytest.mark.parametrize("name", ["base", "large", "large_w32", "gpt2xl"])
def test_full_size_warmup_step_sampled(name):
    """One LAMB warmup step at full size from a seeded synthetic state
    (parameters, momentum, second moment): every sampled chunk's m and v, and
    for whole small tensors the sums of squares, trust ratio, c_bar and the
    updated parameters, against the oracle on the sampled chunks."""
    wl = workload.workloads()[name]
    N, W, C, L = wl.N, wl.W, wl.chunk, wl.L
    gc.collect()
    torch.cuda.empty_cache()              # earlier full-size tests' cached blocks
    free, _ = torch.cuda.mem_get_info()
    gbytes = {"f32": 4, "bf16": 2, "philox": 0}[wl.grad]
    need = pkg.workspace_bytes(layers_of(wl), W, C) + 4 * N + gbytes * W * (N + 8)
    if need > 0.9 * free:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory")
    x = torch.empty(N, device="cuda")
    pkg.gen_params(x, 0, N, wl.param_std, wl.seed)
    opt = pkg.OneBitLamb(x, layers_of(wl), W, C, **wl.hp)
    st = opt.state()
    pkg.gen_params(st["m"], 0, N, STDS["m"], SEEDS["m"])
    pkg.gen_params(st["v"], 0, N, STDS["v"], SEEDS["v"])
    st["v"][:N].mul_(st["v"][:N])
    st["c_bar"].copy_(torch.from_numpy(c_bar_of(L)))
    opt.set_counters(STEP, 3, 0)          # mid-warmup: c_bar follows its EMA
    if wl.grad == "philox":
        g = pkg.PhiloxGrads(wl.seed, wl.layer_std, wl.layer_heavy, wl.heavy_scale)
    else:
        q = 8 if wl.grad == "bf16" else 4
        ld = -(-N // q) * q
        g = torch.empty((W, ld), dtype=torch.int16 if wl.grad == "bf16" else torch.float32,
                        device="cuda")
        pkg.gen_grads(g, STEP, wl.seed, layers_of(wl), wl.layer_std, None, wl.heavy_scale)
    opt.warmup_step(g)
    torch.cuda.synchronize()
    del g

    ks = sample_chunks(wl, small=2 * C)
    frags, NL = fragments(wl, ks)
    idx = np.concatenate([np.arange(k * C, min((k + 1) * C, N)) for k in ks])
    runs = [(k * C, min((k + 1) * C, N)) for k in ks]

    def gather_host(fn):
        return np.concatenate([fn(lo, hi) for lo, hi in runs])

    x0 = gather_host(lambda lo, hi: host_normal(wl.seed, wl.param_std, lo, hi))
    o = oracle.Oracle([f[1] for f in frags], [f[2] for f in frags], W, C, wl.hp, x0)
    o.m[:] = gather_host(lambda lo, hi: host_normal(SEEDS["m"], STDS["m"], lo, hi))
    v = gather_host(lambda lo, hi: host_normal(SEEDS["v"], STDS["v"], lo, hi))
    o.v[:] = v * v
    cb = c_bar_of(L)
    o.c_bar[:] = [cb[f[0]] for f in frags]
    o.t, o.n_warm = STEP, 3
    gh = np.empty((W, NL), np.float32)
    for w in range(W):
        gw = gather_host(lambda lo, hi: workload.gen_grads_range(wl, STEP, w, lo, hi))
        gh[w] = workload.bf16_round(gw) if wl.grad == "bf16" else gw
    o.warmup_step(gh)

    s = opt.state()
    it = torch.from_numpy(idx).cuda()
    for k in ("m", "v"):
        np.testing.assert_array_equal(s[k][it].cpu().numpy().view(np.uint32),
                                      getattr(o, k).view(np.uint32), err_msg=k)
    Sx, Su = s["Sx"].cpu().numpy(), s["Su"].cpu().numpy()
    c, cbar = s["c_cur"].cpu().numpy(), s["c_bar"].cpu().numpy()
    xg = x[it].cpu().numpy()
    n_whole = 0
    for j, (l, lo, n, whole) in enumerate(frags):
        if not whole:
            continue
        n_whole += 1
        assert close_scalar(Sx[l], o.Sx[j]) and close_scalar(Su[l], o.Su[j]), l
        assert close_scalar(c[l], o.c_cur[j]) and close_scalar(cbar[l], o.c_bar[j]), l
        np.testing.assert_array_equal(xg[lo:lo + n].view(np.uint32),
                                      o.x[lo:lo + n].view(np.uint32), err_msg=str(l))
    assert n_whole >= 50
    opt.close()
