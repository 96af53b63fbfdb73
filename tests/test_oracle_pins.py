"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Every check here is either a hand-derived value (tests/golden), a closed
form, an invariant the 1-bit LAMB paper states (arXiv 2104.06069), a special
case that reduces to textbook LAMB, or a library routine.  None re-types the
oracle's own formula.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-6, weight_decay=0.01,
          coeff_min=0.01, coeff_max=10.0, coeff_ema=0.9,
          factor_min=0.5, factor_max=4.0, factor_threshold=0.1)


def ulp32(x):
    x = np.abs(np.asarray(x, dtype=np.float32))
    return np.spacing(x).astype(np.float64)


# ---------------------------------------------------------------------------
# canonical pairwise tree
# ---------------------------------------------------------------------------

def test_cpt_hand_derived():
    """Values derived by hand in tests/golden/cpt_cases.json distinguish the
    granule-aligned pairwise tree from a sequential sum, from an exactly
    rounded sum, from a tree aligned to the segment start and from a
    right-associated level 1."""
    spec = json.load(open(os.path.join(GOLDEN, "cpt_cases.json")))
    for c in spec["cases"]:
        a = np.zeros(c["n"], dtype=np.float32)
        f0, f1, fv = c["fill"]
        a[f0:f1] = np.float32(float.fromhex(fv))
        for i, v in c["set"]:
            a[i] = np.float32(float.fromhex(v))
        got = oracle.cpt_sumsq(a, c["lo"], c["hi"])
        assert got == np.float32(float.fromhex(c["expected"])), c["name"]


def test_cpt_error_bound_and_exact_cases():
    rng = np.random.default_rng(1)
    for n, lo, hi in [(5000, 0, 5000), (5000, 37, 4099), (70000, 255, 69999), (300, 299, 300)]:
        a = rng.standard_normal(n).astype(np.float32)
        got = float(oracle.cpt_sumsq(a, lo, hi))
        sq = [float(np.float32(x) * np.float32(x)) for x in a[lo:hi]]
        exact = math.fsum(sq)
        depth = 8 + math.ceil(math.log2(max(1, (hi - 1) // 256 - lo // 256 + 1)))
        # pairwise summation bound (Higham): depth * u * sum|leaf|
        assert abs(got - exact) <= (depth + 1) * 2.0 ** -24 * exact * 1.01
    # integers below 2^24 add exactly in any order
    a = rng.integers(-40, 40, size=3000).astype(np.float32)
    assert oracle.cpt_sumsq(a, 11, 2999) == np.float32(np.sum(a[11:2999].astype(np.int64) ** 2))
    # empty segment
    assert oracle.cpt_sumsq(a, 5, 5) == 0.0


# ---------------------------------------------------------------------------
# 1-bit compressor (background, error-compensated compression)
# ---------------------------------------------------------------------------

def test_sign_packing_matches_numpy_packbits():
    """bit = !(z < 0), element j of the chunk at word j//32, bit j%32 (LSB
    first); numpy.packbits(bitorder='little') is the library reference."""
    rng = np.random.default_rng(2)
    for C, n in [(256, 256), (256, 37), (1024, 1000), (512, 1)]:
        z = rng.standard_normal(n).astype(np.float32)
        z[::7] = 0.0
        z[3::11] = -0.0
        s, words, err = oracle.compress_chunk(z, 0, C)
        bits = np.zeros(C, dtype=np.uint8)
        bits[:n] = ~(z < 0)
        bits[:n] &= 1
        want = np.packbits(bits, bitorder="little").view("<u4")
        np.testing.assert_array_equal(words, want)


def test_sign_of_nan_and_zero():
    z = np.array([np.nan, 0.0, -0.0, -1.0] + [1.0] * 252, dtype=np.float32)
    _, words, _ = oracle.compress_chunk(z, 0, 256)
    assert words[0] & 0xF == 0b0111


def test_scale_is_rms_and_reconstruction_within_half_ulp():
    """x = s*sigma + e (the error keeps exactly what the 1-bit message
    loses), up to the rounding of one subtraction; s = ||z||_2 / sqrt(n)."""
    rng = np.random.default_rng(3)
    for C, n, k in [(256, 256, 0), (4096, 4096, 3), (2048, 1852, 7)]:
        z = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        s, words, err = oracle.compress_chunk(z, k, C)
        rms = math.sqrt(math.fsum(float(v) ** 2 for v in z) / n)
        assert abs(float(s) - rms) <= 1e-6 * rms
        sigma = np.where(z < 0, -1.0, 1.0)
        recon = sigma * float(s) + err.astype(np.float64)
        assert np.all(np.abs(recon - z.astype(np.float64)) <= 0.5 * ulp32(err) + 1e-45)


def test_constant_vectors_compress_exactly():
    rng = np.random.default_rng(4)
    for C in (256, 1024, 4096):
        a = np.float32(rng.uniform(1e-4, 3.0))
        z = (a * np.where(rng.random(C) < 0.5, -1, 1)).astype(np.float32)
        s, _, err = oracle.compress_chunk(z, 5, C)
        assert s == a
        assert np.all(err == 0)
    # tail chunk (n not a power of two): exact for powers of two
    for n in (1852, 232, 1):
        a = np.float32(2.0 ** -7)
        z = np.full(n, a, dtype=np.float32)
        z[::3] = -a
        s, _, err = oracle.compress_chunk(z, 2, 4096)
        assert s == a and np.all(err == 0)


def test_error_feedback_telescopes():
    """sum_t C[z_t] + e_T = sum_t p_t + e_0 (error feedback keeps nothing
    back), up to one rounding per step."""
    rng = np.random.default_rng(5)
    C = 1024
    e = np.zeros(C, np.float32)
    sent = np.zeros(C, np.float64)
    fed = np.zeros(C, np.float64)
    bound = np.zeros(C, np.float64)
    for t in range(30):
        p = (rng.standard_normal(C) * 1e-2).astype(np.float32)
        z = (p + e).astype(np.float32)
        bound += 0.5 * ulp32(z)
        s, words, e = oracle.compress_chunk(z, 0, C)
        bits = np.unpackbits(words.view(np.uint8), bitorder="little")[:C]
        sent += np.where(bits == 1, 1.0, -1.0) * float(s)
        fed += p
        bound += 0.5 * ulp32(e)
    assert np.all(np.abs(sent + e - fed) <= bound + 1e-12)


def test_packed_volume_is_one_32nd_plus_scales():
    wl = workload.workloads()["tiny"]
    o = oracle.Oracle(wl.offsets, wl.numels, wl.W, wl.chunk, HP, np.zeros(wl.N, np.float32))
    msg = o.signs_w.nbytes + o.scale_w.nbytes
    full = 4 * wl.W * wl.N
    assert msg == wl.W * (4 * (-(-wl.N // 32)) + 4 * wl.K)
    # 1/32 + 1/C at full chunks, within the padding of the last word and chunk
    assert abs(msg / full - (1 / 32 + 1 / wl.chunk)) < 4.0 / wl.N + 4.0 / wl.chunk


# ---------------------------------------------------------------------------
# warmup stage == LAMB (background, LAMB; W=1, compression off)
# ---------------------------------------------------------------------------

def lamb_bruteforce(x, grads, off, numel, hp):
    """Textbook LAMB in float64: Adam moments without bias correction,
    decoupled weight decay inside the update, one clipped trust ratio per
    tensor (clip applied to the whole ratio), coefficient EMA."""
    hp = {k: float(np.float32(v)) for k, v in hp.items()}   # binary32 settings
    x = x.astype(np.float64).copy()
    m = np.zeros_like(x)
    v = np.zeros_like(x)
    cbar = None
    cs = []
    for g in grads:
        gb = g.astype(np.float64).mean(axis=0)
        m = hp["beta1"] * m + (1 - hp["beta1"]) * gb
        v = hp["beta2"] * v + (1 - hp["beta2"]) * gb * gb
        u = m / (np.sqrt(v) + hp["eps"]) + hp["weight_decay"] * x
        c = np.empty(len(off))
        for l, (o, n) in enumerate(zip(off, numel)):
            nx, nu = np.linalg.norm(x[o:o + n]), np.linalg.norm(u[o:o + n])
            r = 1.0 if nx == 0 or nu == 0 else nx / nu
            c[l] = min(max(r, hp["coeff_min"]), hp["coeff_max"])
        for l, (o, n) in enumerate(zip(off, numel)):
            x[o:o + n] -= hp["lr"] * c[l] * u[o:o + n]
        cbar = c.copy() if cbar is None else hp["coeff_ema"] * cbar + (1 - hp["coeff_ema"]) * c
        cs.append(c)
    return x, m, v, cs, cbar


@pytest.mark.parametrize("W", [1, 4])
def test_warmup_equals_bruteforce_lamb(W):
    wl = workload.custom("bf", [("a", (40, 30)), ("b", (30,)), ("c", (700,)), ("d", (3,))],
                         W=W, chunk=256, grad_std=1e-2)
    x0 = workload.gen_params(wl)
    o = oracle.Oracle(wl.offsets, wl.numels, W, wl.chunk, HP, x0)
    grads = []
    for t in range(6):
        g = workload.grads_for_step(wl, t)
        grads.append(g)
        o.warmup_step(g)
    xb, mb, vb, cs, cbar = lamb_bruteforce(x0, grads, wl.offsets, wl.numels, HP)
    # vectors: max|a - b| <= tol * max|b| over each tensor
    for lo, n in zip(wl.offsets, wl.numels):
        for got, want in ((o.x, xb), (o.m, mb), (o.v, vb)):
            sl = slice(lo, lo + n)
            assert np.max(np.abs(got[sl] - want[sl])) <= 1e-5 * np.max(np.abs(want[sl]))
    np.testing.assert_allclose(o.c_cur, cs[-1], rtol=1e-5)
    np.testing.assert_allclose(o.c_bar, cbar, rtol=1e-5)
    assert o.t == 6 and o.n_warm == 6


def test_warmup_one_step_closed_form():
    """From zero moments with wd = 0 and |g| >> eps, u = (1-b1)/sqrt(1-b2)
    * sign(g), so c = clip(||x|| sqrt(1-b2) / ((1-b1) sqrt(n)))."""
    hp = dict(HP, weight_decay=0.0, eps=1e-12)
    rng = np.random.default_rng(6)
    numel = [4096, 777]
    x0 = rng.standard_normal(sum(numel)).astype(np.float32)
    g = (rng.standard_normal((1, sum(numel))) + 3.0).astype(np.float32)
    o = oracle.Oracle([0, 4096], numel, 1, 256, hp, x0)
    o.warmup_step(g)
    for l, (lo, n) in enumerate(zip([0, 4096], numel)):
        w1 = 1.0 - float(np.float32(0.9))      # exact: the binary32 betas
        w2 = 1.0 - float(np.float32(0.999))
        want = np.linalg.norm(x0[lo:lo + n].astype(np.float64)) * math.sqrt(w2) / (w1 * math.sqrt(n))
        want = min(max(want, 0.01), 10.0)
        assert abs(o.c_cur[l] - want) <= 2e-6 * want


def test_warmup_zero_norm_ratio_is_one():
    o = oracle.Oracle([0, 300], [300, 5], 2, 256, HP, np.zeros(305, np.float32))
    g = np.ones((2, 305), np.float32)
    o.warmup_step(g)
    assert np.all(o.c_cur == 1.0)   # ||x|| = 0 -> ratio 1


# ---------------------------------------------------------------------------
# compression stage
# ---------------------------------------------------------------------------

def _fresh(N_layers, W, C, hp=HP, x0=None):
    numel = list(N_layers)
    off = np.concatenate([[0], np.cumsum(numel)[:-1]])
    N = int(sum(numel))
    x0 = np.zeros(N, np.float32) if x0 is None else x0
    return oracle.Oracle(off, numel, W, C, hp, x0)


def test_server_identity_single_worker():
    """W = 1 with zero server error on full chunks: the server's
    recompression sends exactly what the worker sent and keeps no error."""
    rng = np.random.default_rng(7)
    o = _fresh([1024, 512], 1, 256)
    o.m[:] = rng.standard_normal(o.N).astype(np.float32) * 1e-2
    o.v[:] = 1e-4
    o.freeze()
    g = (rng.standard_normal((1, o.N)) * 1e-2).astype(np.float32)
    o.compress_step(g)
    np.testing.assert_array_equal(o.signs_s, o.signs_w[0])
    np.testing.assert_array_equal(o.scale_s, o.scale_w[0])
    assert np.all(o.e_s == 0)


def test_equal_scales_popcount_average():
    """With equal worker scales s the server average is s (2p - W) / W, p the
    number of +1 bits in the element's column (a popcount)."""
    rng = np.random.default_rng(8)
    W, C = 8, 256
    o = _fresh([C], W, C)
    o.freeze()
    a = np.float32(0.01)
    g = (a * np.where(rng.random((W, C)) < 0.5, -1, 1)).astype(np.float32)
    o.compress_step(g)
    s = float(o.scale_w[0, 0])
    assert np.all(o.scale_w[:, 0] == o.scale_w[0, 0])
    bits = np.unpackbits(o.signs_w.view(np.uint8), bitorder="little").reshape(W, -1)[:, :C]
    p = bits.sum(axis=0).astype(np.int64)
    want = s * (2 * p - W) / W
    m_new = o.m.astype(np.float64)
    avg = m_new + o.e_s.astype(np.float64)     # y = avg + 0 = m_new + e_s
    assert np.all(np.abs(avg - want) <= W * np.spacing(np.float32(s)) + 1e-12)


def test_lossless_compression_reduces_to_frozen_variance_momentum_sgd():
    """When every chunk of the momentum has constant magnitude, 1-bit
    compression is exact; with beta2 = 1 the layer factor stays 1, and a
    compression step is momentum SGD preconditioned by the frozen variance
    with coefficient c_bar (1-bit Adam's compression stage scaled by LAMB's
    warmup coefficient)."""
    hp = dict(HP, beta2=1.0)
    rng = np.random.default_rng(9)
    numel = [1024, 2048]
    o = _fresh(numel, 2, 256, hp, x0=rng.standard_normal(3072).astype(np.float32))
    o.v[:] = rng.uniform(1e-6, 1e-4, o.N).astype(np.float32)
    o.c_bar[:] = [0.5, 2.0]
    o.freeze()
    x0 = o.x.astype(np.float64).copy()
    a = np.float32(3e-3)
    sg = np.where(rng.random(o.N) < 0.5, -1, 1)
    g = np.stack([a * sg, a * sg]).astype(np.float32)
    o.compress_step(g)
    m_w = (1 - 0.9) * a * sg          # m starts at 0
    assert np.allclose(o.m, m_w, rtol=1e-6)
    assert np.all(o.e_w == 0) and np.all(o.e_s == 0)
    assert np.all(o.r_prev == 1.0)
    np.testing.assert_array_equal(o.c_cur, o.c_bar)
    cvec = np.repeat(o.c_bar.astype(np.float64), numel)
    u = m_w / (np.sqrt(o.v.astype(np.float64)) + 1e-6) + 0.01 * x0
    np.testing.assert_allclose(o.x, x0 - 1e-3 * cvec * u, rtol=1e-6, atol=1e-9)


def test_fresh_variance_and_ratio_follow_closed_forms():
    """Lossless compression for 30 steps: two workers send the same gradient
    of constant magnitude per chunk, so every chunk compresses exactly (its
    scale is |z|: a pairwise sum of equal squares over a power-of-two chunk is
    exact, and sqrt(fl(z^2)) = |z| in binary floating point), the server
    average of two equal values is exact, and no error is kept.  Then the
    reconstructed gradient is the true gradient g up to one cancellation, so
    the fresh second moment solves its recursion in closed form,
    v_t = beta2^t v0 + (1 - beta2^t) g^2, and the per-tensor ratio is
    R_t = max over the tensor of (sqrt(v0) + eps) / (sqrt(v_t) + eps).
    Tensor 0 has two halves with different |g| (the max picks the half whose
    fresh variance stays smaller); tensor 1's gradient shrinks below the
    frozen variance, so its ratio rises above 1.  The factor then follows the
    soft thresholds: r_t = clip(clip(R_t, 0.5, 4), 0.9 r_{t-1}, 1.1 r_{t-1})."""
    rng = np.random.default_rng(21)
    numel = [2048, 1024]
    o = _fresh(numel, 2, 256, HP, x0=rng.standard_normal(3072).astype(np.float32))
    v0 = np.array([4e-6, 1e-6])
    mag = np.empty(3072)
    mag[:1024], mag[1024:2048], mag[2048:] = 4e-3, 2.5e-3, 2e-4    # |g| per element
    o.v[:2048] = np.float32(v0[0])
    o.v[2048:] = np.float32(v0[1])
    o.freeze()
    sg = np.where(rng.random(3072) < 0.5, -1.0, 1.0)
    g = np.stack([mag * sg, mag * sg]).astype(np.float32)
    g32 = np.abs(g[0]).astype(np.float64)
    b2, eps = 0.999, 1e-6
    r = np.ones(2)
    for t in range(1, 31):
        o.compress_step(g)
        assert np.all(o.e_w == 0) and np.all(o.e_s == 0), t
        v_t = np.empty(3072)
        v_t[:2048] = b2 ** t * v0[0] + (1 - b2 ** t) * g32[:2048] ** 2
        v_t[2048:] = b2 ** t * v0[1] + (1 - b2 ** t) * g32[2048:] ** 2
        np.testing.assert_allclose(o.v_fresh, v_t, rtol=2e-5)
        rho = (np.sqrt(np.repeat(v0, numel)) + eps) / (np.sqrt(v_t) + eps)
        R = np.array([rho[:2048].max(), rho[2048:].max()])
        np.testing.assert_allclose(o.R, R, rtol=2e-5)
        r = np.minimum(np.maximum(np.minimum(np.maximum(R, 0.5), 4.0), 0.9 * r), 1.1 * r)
        np.testing.assert_allclose(o.r_prev, r, rtol=2e-5)
    assert o.R[0] < 1.0 < o.R[1]


def test_beta2_one_keeps_factor_one_over_steps():
    hp = dict(HP, beta2=1.0)
    rng = np.random.default_rng(10)
    o = _fresh([3000, 500], 4, 512, hp, x0=rng.standard_normal(3500).astype(np.float32))
    for t in range(3):
        o.warmup_step((rng.standard_normal((4, 3500)) * 1e-2).astype(np.float32))
    o.freeze()
    cbar = o.c_bar.copy()
    for t in range(4):
        o.compress_step((rng.standard_normal((4, 3500)) * 1e-2).astype(np.float32))
        assert np.all(o.r_prev == 1.0)
        np.testing.assert_array_equal(o.c_cur, cbar)


def _decode(words, scales, N, C):
    """+-scale per element from packed sign words (bit 1 = +1, LSB first)."""
    bits = np.unpackbits(np.ascontiguousarray(words).view(np.uint8), bitorder="little")[:N]
    return np.where(bits == 1, 1.0, -1.0) * np.repeat(np.asarray(scales, np.float64), C)[:N]


def test_error_feedback_telescopes_over_full_steps():
    """Over T compression steps of the full optimizer nothing is held back by
    either error buffer: for every worker w,
        sum_t (what w sent) + e_w,T = sum_t (w's momentum before compression),
    and for the server
        sum_t (the scattered momentum) + e_s,T = sum_t (average of what the
        workers sent),
    where 'sent' is decoded from the exchanged sign words and scales, and a
    worker's momentum before compression is beta1 m_{t-1} + (1-beta1) g_w,t.
    Bounds: the binary32 roundings of each step."""
    rng = np.random.default_rng(23)
    numel = [1500, 700, 1000]        # N = 3200: a ragged last chunk of 128
    W, C = 3, 256
    o = _fresh(numel, W, C, HP, x0=(rng.standard_normal(3200) * 2e-2).astype(np.float32))
    for _ in range(2):
        o.warmup_step((rng.standard_normal((W, o.N)) * 1e-2).astype(np.float32))
    o.freeze()
    N = o.N
    sent_w = np.zeros((W, N)); fed_w = np.zeros((W, N))
    sent_s = np.zeros(N); fed_s = np.zeros(N)
    tol_w = np.zeros((W, N)); tol_s = np.zeros(N)
    for t in range(25):
        g = (rng.standard_normal((W, N)) * 1e-2).astype(np.float32)
        m_old = o.m.astype(np.float64)
        o.compress_step(g)
        dec = np.stack([_decode(o.signs_w[w], o.scale_w[w], N, C) for w in range(W)])
        mw = 0.9 * m_old + (1 - 0.9) * g.astype(np.float64)
        sent_w += dec
        fed_w += mw
        avg = dec.sum(axis=0) / W
        sent_s += o.m.astype(np.float64)
        fed_s += avg
        # a few roundings per step: the momentum, z = m_w + e, e = z -+ s, and
        # for the server the sum over workers, the division and y = avg + e_s
        tol_w += 4 * ulp32(np.abs(mw) + np.abs(dec) + 1e-30)
        tol_s += 4 * ulp32(np.abs(avg) * W + np.abs(o.m) + 1e-30)
    assert np.all(np.abs(sent_w + o.e_w - fed_w) <= tol_w)
    assert np.all(np.abs(sent_s + o.e_s - fed_s) <= tol_s)


def test_warmup_coefficient_average_closed_form():
    """c_bar is the exponential moving average (weight 0.9) of the warmup
    coefficients, started at the first one.  The first step's ratio clips at
    coeff_max (huge parameters); the parameters are then made tiny so every
    later ratio clips at coeff_min:
        c_bar_T = 0.9^(T-1) coeff_max + (1 - 0.9^(T-1)) coeff_min."""
    rng = np.random.default_rng(24)
    o = _fresh([1024], 2, 256, HP, x0=(rng.standard_normal(1024) * 1e3).astype(np.float32))
    for t in range(1, 9):
        o.warmup_step((rng.standard_normal((2, 1024)) * 1e-2).astype(np.float32))
        want_c = 10.0 if t == 1 else 0.01
        assert o.c_cur[0] == np.float32(want_c), t
        want_bar = 0.9 ** (t - 1) * 10.0 + (1 - 0.9 ** (t - 1)) * 0.01
        np.testing.assert_allclose(o.c_bar[0], want_bar, rtol=1e-5)
        if t == 1:
            o.x[:] = (rng.standard_normal(1024) * 1e-7).astype(np.float32)


def test_compression_update_scales_with_the_layer_factor():
    """Two optimizers differ only in the soft-threshold width (0.1 and 0.3);
    the ratio is forced far above factor_max, so the factor rises to 1.1 and
    1.3 in the first step.  Everything else being equal, their parameter steps
    differ by exactly that factor (up to rounding): the update is scaled by
    c = c_bar r, not by c_bar alone.  And the step itself is the frozen-
    variance preconditioned momentum step (the fresh second moment, here 0,
    only steers the factor): dx = -lr c_bar r m / (sqrt(v) + eps)."""
    rng = np.random.default_rng(25)
    x0 = np.zeros(2048, np.float32)       # steps land exactly on zero parameters
    g = (rng.standard_normal((2, 2048)) * 1e-9).astype(np.float32)
    steps = []
    for thr in (0.1, 0.3):
        o = _fresh([2048], 2, 256, dict(HP, factor_threshold=thr), x0=x0.copy())
        o.v[:] = 1e4
        o.m[:] = np.float32(1e-3)
        o.c_bar[:] = 0.5
        o.freeze()
        o.v_fresh[:] = 0.0
        o.compress_step(g)
        np.testing.assert_allclose(o.r_prev, 1.0 + thr, rtol=1e-6)
        steps.append(o.x.astype(np.float64) - x0.astype(np.float64))
        # m after the step: 0.9 * 1e-3 + 0.1 g (|g| ~ 1e-9), compressed per chunk
        want = -1e-3 * 0.5 * (1.0 + thr) * np.abs(o.m.astype(np.float64)) / (100.0 + 1e-6)
        np.testing.assert_allclose(np.abs(steps[-1]), np.abs(want), rtol=1e-5)
        np.testing.assert_allclose(np.abs(o.m), 0.9e-3, rtol=1e-5)
    assert np.all(steps[0] < 0)
    np.testing.assert_allclose(steps[1] / steps[0], 1.3 / 1.1, rtol=1e-6)


def test_soft_threshold_growth_closed_form():
    """With the ratio far above factor_max every step, the factor grows by
    (1 + threshold) per step until it reaches factor_max: r_t =
    min(factor_max, 1.1^t)."""
    rng = np.random.default_rng(11)
    o = _fresh([2048, 300], 2, 256)
    o.v[:] = 1e4
    o.freeze()
    o.v_fresh[:] = 0.0
    for t in range(1, 21):
        o.compress_step((rng.standard_normal((2, o.N)) * 1e-9).astype(np.float32))
        assert np.all(o.R > 100.0)
        want = min(4.0, 1.1 ** t)
        np.testing.assert_allclose(o.r_prev, want, rtol=2e-6)
    # and shrinks by (1 - threshold) when the ratio is far below factor_min
    o2 = _fresh([2048], 2, 256)
    o2.freeze()
    o2.v[:] = 0.0
    o2.v_fresh[:] = 1e4
    for t in range(1, 10):
        o2.compress_step((rng.standard_normal((2, o2.N)) * 1e-9).astype(np.float32))
        np.testing.assert_allclose(o2.r_prev, max(0.5, 0.9 ** t), rtol=2e-6)


def test_nan_ratio_counts_as_infinity():
    """A NaN gradient makes the element's ratio NaN; the per-tensor maximum
    counts it as +Inf (reading R19), so the factor rises by the soft
    threshold only (clip(Inf, fmin, fmax) = fmax, then at most 1.1 r_prev),
    and the other tensor is unaffected."""
    rng = np.random.default_rng(26)
    o = _fresh([1024, 1024], 2, 256, HP, x0=(rng.standard_normal(2048) * 2e-2).astype(np.float32))
    o.v[:] = 1e-4
    o.freeze()
    g = (rng.standard_normal((2, 2048)) * 1e-2).astype(np.float32)
    g[1, 100] = np.nan
    o.compress_step(g)
    assert o.R[0] == np.inf
    assert o.r_prev[0] == np.float32(np.float32(1.1) * np.float32(1.0))
    assert np.isfinite(o.R[1]) and np.isfinite(o.r_prev[1])


def test_layer_factor_clip_definition():
    """clip(x, a, b) = min{max{x, a}, b} (LAMB background, footnote 4),
    applied twice: the hard bounds, then +-threshold around r_prev."""
    f = oracle.layer_factor
    assert f(10.0, 1.0, 0.5, 4.0, 0.1) == np.float32(1.1)
    assert f(1.05, 1.0, 0.5, 4.0, 0.1) == np.float32(1.05)
    assert f(0.1, 1.0, 0.5, 4.0, 0.1) == np.float32(0.9)
    assert f(0.1, 0.52, 0.5, 4.0, 0.1) == np.float32(0.5)
    assert f(float("inf"), 3.9, 0.5, 4.0, 0.1) == np.float32(4.0)


def test_stage_order_enforced():
    o = _fresh([256], 1, 256)
    g = np.zeros((1, 256), np.float32)
    with pytest.raises(RuntimeError):
        o.compress_step(g)
    o.freeze()
    with pytest.raises(RuntimeError):
        o.warmup_step(g)
    with pytest.raises(RuntimeError):
        o.freeze()


# ---------------------------------------------------------------------------
# indexing of the five workloads
# ---------------------------------------------------------------------------

def test_workload_tables():
    """Tensor counts and sizes of the standard parameter lists: BERT-Base
    ~110M, BERT-Large ~340M, GPT-2-XL ~1.56B; chunks tile the flat buffer from
    0 and the last chunk holds the remainder."""
    want = {"tiny": (4, 9448, 37, 232), "base": (206, 110106428, 53763, 1852),
            "large": (398, 336226108, 82087, 1852),
            "large_w32": (398, 336226108, 82087, 1852),
            "gpt2xl": (580, 1557611200, 190139, 704)}
    for name, wl in workload.workloads().items():
        L, N, K, tail = want[name]
        assert (wl.L, wl.N, wl.K) == (L, N, K), name
        assert wl.N - (wl.K - 1) * wl.chunk == tail
        off, num = wl.offsets, wl.numels
        assert off[0] == 0 and np.all(off[1:] == off[:-1] + num[:-1])
    large = workload.workloads()["large_w32"]
    assert int(large.layer_heavy.sum()) == 79


# ---------------------------------------------------------------------------
# 1-bit Adam variant (the predecessor method: Adam warmup, frozen-variance
# compressed momentum, no layerwise coefficient)
# ---------------------------------------------------------------------------

def adam_bruteforce(x, grads, hp):
    """Textbook Adam in float64 without bias correction, decoupled weight
    decay inside the update, at the binary32 settings."""
    hp = {k: float(np.float32(v)) for k, v in hp.items()}
    x = x.astype(np.float64).copy()
    m = np.zeros_like(x)
    v = np.zeros_like(x)
    for g in grads:
        gb = g.astype(np.float64).mean(axis=0)
        m = hp["beta1"] * m + (1 - hp["beta1"]) * gb
        v = hp["beta2"] * v + (1 - hp["beta2"]) * gb * gb
        x -= hp["lr"] * (m / (np.sqrt(v) + hp["eps"]) + hp["weight_decay"] * x)
    return x, m, v


@pytest.mark.parametrize("W", [1, 4])
def test_adam_variant_warmup_equals_bruteforce_adam(W):
    wl = workload.custom("bf", [("a", (40, 30)), ("b", (30,)), ("c", (700,))],
                         W=W, chunk=256, grad_std=1e-2)
    x0 = workload.gen_params(wl)
    o = oracle.Oracle(wl.offsets, wl.numels, W, wl.chunk, HP, x0, variant=1)
    grads = []
    for t in range(6):
        g = workload.grads_for_step(wl, t)
        grads.append(g)
        o.warmup_step(g)
    xb, mb, vb = adam_bruteforce(x0, grads, HP)
    for got, want in ((o.x, xb), (o.m, mb), (o.v, vb)):
        assert np.max(np.abs(got - want)) <= 1e-5 * np.max(np.abs(want))
    assert np.all(o.c_cur == 1.0) and np.all(o.c_bar == 1.0)


def test_adam_variant_lossless_compression_is_frozen_variance_momentum_sgd():
    """With exact 1-bit compression (constant-magnitude momentum chunks) a
    1-bit Adam compression step is momentum SGD preconditioned by the frozen
    variance, coefficient 1 (the 1-bit Adam page: variance frozen after the
    warmup, momentum communicated with error-compensated compression)."""
    rng = np.random.default_rng(12)
    numel = [1024, 2048]
    o = _fresh(numel, 2, 256, HP, x0=rng.standard_normal(3072).astype(np.float32))
    o.variant = 1
    o.v[:] = rng.uniform(1e-6, 1e-4, o.N).astype(np.float32)
    o.c_bar[:] = 0.5           # a LAMB warmup average, which 1-bit Adam must not use
    o.freeze()
    vf0 = o.v_fresh.copy()
    x0 = o.x.astype(np.float64).copy()
    a = np.float32(3e-3)
    sg = np.where(rng.random(o.N) < 0.5, -1, 1)
    o.compress_step(np.stack([a * sg, a * sg]).astype(np.float32))
    m_w = (1 - 0.9) * a * sg
    assert np.allclose(o.m, m_w, rtol=1e-6)
    np.testing.assert_array_equal(o.v_fresh, vf0)      # no fresh variance
    assert np.all(o.c_cur == 1.0)
    u = m_w / (np.sqrt(o.v.astype(np.float64)) + 1e-6) + 0.01 * x0
    np.testing.assert_allclose(o.x, x0 - 1e-3 * u, rtol=1e-6, atol=1e-9)


# ---------------------------------------------------------------------------
# bf16 error-storage variant
# ---------------------------------------------------------------------------

def test_bf16_storage_rounding_matches_torch():
    """Round-to-nearest-even to bfloat16, checked against torch's conversion
    (library routine) on random values, ties, signed zeros and infinities."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(13)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    x[:6] = [0.0, -0.0, np.inf, -np.inf, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]
    ours = np.array([oracle.bf16_round(v) for v in x], dtype=np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))
    assert np.isnan(oracle.bf16_round(float("nan")))


def test_bf16_error_storage_rounds_the_fp32_error_once():
    """From zero errors, one compression step of the bf16-storage variant
    sends the same words and scales as the fp32 variant and keeps the
    fp32 variant's new worker and server errors rounded to bfloat16."""
    rng = np.random.default_rng(14)
    states = []
    for eb in (0, 1):
        o = _fresh([3000, 700], 4, 512, HP, x0=(rng.standard_normal(3700) * 0 + 1).astype(np.float32))
        o.err_bf16 = eb
        o.m[:] = np.linspace(-1e-2, 1e-2, o.N, dtype=np.float32)
        o.v[:] = 1e-4
        o.freeze()
        g = (np.sin(np.arange(4 * o.N, dtype=np.float64)).reshape(4, o.N) * 1e-2).astype(np.float32)
        o.compress_step(g)
        states.append(o)
    a, b = states
    np.testing.assert_array_equal(a.signs_w, b.signs_w)
    np.testing.assert_array_equal(a.scale_w, b.scale_w)
    want = np.array([oracle.bf16_round(v) for v in a.e_w.ravel()], np.float32).reshape(a.e_w.shape)
    np.testing.assert_array_equal(b.e_w.view(np.uint32), want.view(np.uint32))
    # the server sees the same average (same words and scales), so its kept error is the
    # binary32 one rounded once as well
    np.testing.assert_array_equal(a.signs_s, b.signs_s)
    want_s = np.array([oracle.bf16_round(v) for v in a.e_s], np.float32)
    np.testing.assert_array_equal(b.e_s.view(np.uint32), want_s.view(np.uint32))


def test_bf16_error_feedback_telescopes_within_storage_rounding():
    """With bf16 error storage the error feedback still telescopes, up to one
    bf16 rounding (2^-9 relative) of the kept error per step."""
    rng = np.random.default_rng(15)
    C = 1024
    e = np.zeros(C, np.float32)
    sent = np.zeros(C, np.float64)
    fed = np.zeros(C, np.float64)
    bound = np.zeros(C, np.float64)
    for t in range(30):
        p = (rng.standard_normal(C) * 1e-2).astype(np.float32)
        z = (p + e).astype(np.float32)
        bound += 0.5 * ulp32(z)
        s, words, e_full = oracle.compress_chunk(z, 0, C)
        e = np.array([oracle.bf16_round(v) for v in e_full], np.float32)
        bits = np.unpackbits(words.view(np.uint8), bitorder="little")[:C]
        sent += np.where(bits == 1, 1.0, -1.0) * float(s)
        fed += p
        bound += 0.5 * ulp32(e_full) + np.abs(e_full.astype(np.float64)) * 2.0 ** -8
    assert np.all(np.abs(sent + e - fed) <= bound + 1e-12)
