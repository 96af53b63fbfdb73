"""Pins of the seeded input generator (Philox4x32-10 + exact Box-Muller)."""
import math
import statistics

import numpy as np
import pytest

import workload


def test_philox_known_answers():
    """Known-answer vectors of Philox4x32-10 published with the Random123
    library (Salmon et al., SC'11)."""
    P = workload.philox
    assert P([0, 0, 0, 0], [0, 0]) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert P([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2) == [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert P([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0]) == \
        [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_uniform_is_exact_and_open():
    L = workload.lib()
    assert L.wl_uniform(0) == 2.0 ** -24
    assert L.wl_uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert L.wl_uniform(0x80000000) == 0.5 + 2.0 ** -24


def test_log_and_sincos_accuracy():
    L = workload.lib()
    xs = np.concatenate([np.geomspace(2.0 ** -24, 1.0, 4000, endpoint=False),
                         np.linspace(0.5, 1.0, 2000, endpoint=False)]).astype(np.float32)
    err = max(abs(L.wl_log(float(x)) - math.log(float(x))) for x in xs)
    assert err < 2e-6
    import ctypes
    c, s = ctypes.c_float(), ctypes.c_float()
    worst = 0.0
    for v in np.linspace(0.0, 1.0, 5001, endpoint=False).astype(np.float32):
        L.wl_sincos2pi(float(v), ctypes.byref(c), ctypes.byref(s))
        a = 2 * math.pi * float(v)
        worst = max(worst, abs(c.value - math.cos(a)), abs(s.value - math.sin(a)))
    assert worst < 1e-6


def test_normal_distribution():
    """Moments and a Kolmogorov-Smirnov distance against the normal CDF."""
    z = np.concatenate([workload.normal4(7, q, 0, 3, 1) for q in range(60000)]).astype(np.float64)
    assert abs(z.mean()) < 0.01
    assert abs(z.var() - 1.0) < 0.01
    zs = np.sort(z)
    cdf = np.array([statistics.NormalDist().cdf(v) for v in zs[::20]])
    emp = (np.arange(0, len(zs), 20) + 0.5) / len(zs)
    assert np.max(np.abs(cdf - emp)) < 0.01


def test_box_muller_matches_double_precision_formula():
    import ctypes
    L = workload.lib()
    rng = np.random.default_rng(0)
    z0, z1 = ctypes.c_float(), ctypes.c_float()
    for a, b in rng.integers(0, 2 ** 32, size=(3000, 2), dtype=np.uint64):
        L.wl_box_muller(int(a), int(b), ctypes.byref(z0), ctypes.byref(z1))
        u1, u2 = L.wl_uniform(int(a)), L.wl_uniform(int(b))
        r = math.sqrt(-2 * math.log(u1))
        assert abs(z0.value - r * math.cos(2 * math.pi * u2)) < 2e-5
        assert abs(z1.value - r * math.sin(2 * math.pi * u2)) < 2e-5


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * 1e-3).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]   # ties to even
    L = workload.lib()
    ours = np.array([L.wl_bf16_rne(float(v)) for v in x], dtype=np.uint16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_grad_streams_are_distinct_and_scaled():
    wl = workload.workloads()["tiny"]
    g00 = workload.gen_grads(wl, 0, 0)
    g01 = workload.gen_grads(wl, 0, 1)
    g10 = workload.gen_grads(wl, 1, 0)
    assert not np.array_equal(g00, g01) and not np.array_equal(g00, g10)
    assert abs(g00.std() - 1e-2) < 1e-3
    x = workload.gen_params(wl)
    assert abs(x.std() - 2e-2) < 2e-3
    np.testing.assert_array_equal(workload.gen_params(wl, 100, 200), x[100:200])


def test_heavy_tailed_layers():
    wl = workload.custom("h", [("a", (4000,)), ("b", (40000,))], W=1, chunk=256,
                         grad="philox", grad_std=1e-3, heavy_every=2, heavy_scale=1e-3)
    g = workload.gen_grads(wl, 0, 0)
    normal, heavy = g[:4000], g[4000:]
    # Student-t(3): variance 3 * scale^2, excess kurtosis large
    assert 0.5e-3 < normal.std() < 1.5e-3
    k = np.mean(heavy.astype(np.float64) ** 4) / np.mean(heavy.astype(np.float64) ** 2) ** 2
    assert k > 6.0
