"""GPU parity of the whole hot path against the CPU oracle, step by step, on
seeded workloads that span many chunks with ragged tails (N not a multiple of
4, 32 or C), misaligned tensor boundaries, every chunk size, every gradient
storage, and the degenerate cases (one worker, one element, a chunk holding
more tensors than the kernel keeps in shared memory)."""
import numpy as np
import pytest

import workload
from harness import Pair

pytestmark = pytest.mark.gpu


def bert_mini(W=8, chunk=2048, grad="f32", **kw):
    t = workload.bert_tensors(2, 64, 256, 1000) + [("extra", (5,))]
    return workload.custom("bert_mini", t, W=W, chunk=chunk, grad=grad, grad_std=1e-3, **kw)


def run(wl, n_warm, n_comp, expect_bitwise=True, variant=0, error_storage=0):
    p = Pair(wl, variant=variant, error_storage=error_storage)
    diffs = 0
    for i in range(n_warm):
        p.warmup()
        diffs += p.compare(f"warmup {i}")
    p.freeze()
    diffs += p.compare("freeze")
    for i in range(n_comp):
        p.compress()
        diffs += p.compare(f"compress {i}")
    if expect_bitwise:
        assert diffs == 0, f"{diffs} float elements differ in some bit"
    return p


def test_tiny_workload_full_run():
    """The toy workload as specified: 4 tensors, W=4, C=256, 5 warmup steps,
    freeze, 5 compression steps."""
    wl = workload.workloads()["tiny"]
    run(wl, wl.warmup_steps, wl.compress_steps)


def test_bert_mini_twenty_steps():
    """BERT-shaped table (odd tensor offsets, N % 4 == 3), W=8, C=2048,
    10 warmup + 10 compression steps: parameters after 20 steps."""
    wl = bert_mini()
    assert wl.N % 4 == 3
    run(wl, 10, 10)


@pytest.mark.parametrize("chunk", [256, 512, 1024, 4096, 8192])
def test_every_chunk_size(chunk):
    wl = bert_mini(W=3, chunk=chunk)
    run(wl, 2, 3)


def test_bf16_gradients():
    t = workload.gpt2_tensors(2, 48, 192, 500, n_pos=64)
    wl = workload.custom("gpt2_mini", t, W=8, chunk=8192, grad="bf16", grad_std=1e-3)
    assert wl.N > 3 * wl.chunk
    run(wl, 3, 4)


@pytest.mark.parametrize("chunk", [256, 512, 1024, 2048, 8192])
def test_in_kernel_gradients_at_other_chunk_sizes(chunk):
    """In-kernel gradients at the chunk sizes whose kernels draw them in the
    compressing threads themselves (no draw warps): normal and Student-t
    tensors, tiles that hold both kinds and tiles of only one."""
    t = workload.bert_tensors(1, 64, 256, 700) + [("tail", (37,))]
    wl = workload.custom("w5_philox", t, W=5, chunk=chunk, grad="philox", grad_std=1e-3,
                         fan_in_scaled=True, heavy_every=5, heavy_scale=1e-3)
    assert wl.N % chunk != 0
    run(wl, 2, 3)


@pytest.mark.parametrize("chunk", [256, 512, 1024, 2048, 4096, 8192])
@pytest.mark.parametrize("grad", ["f32", "bf16", "philox"])
@pytest.mark.parametrize("variant,errors", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_every_kernel_instantiation(variant, errors, grad, chunk):
    """Every combination the dispatch can launch (method variant x error
    storage x gradient kind x chunk size) on one small ragged table, W = 3:
    each compiled kernel instantiation runs against the oracle at least
    once."""
    t = workload.bert_tensors(1, 32, 128, 300, max_pos=64) + [("tail", (37,))]
    kw = dict(heavy_every=5, heavy_scale=1e-3, fan_in_scaled=True) if grad == "philox" else {}
    wl = workload.custom("sweep", t, W=3, chunk=chunk, grad=grad, grad_std=1e-3, **kw)
    run(wl, 1, 2, variant=variant, error_storage=errors)


def test_in_kernel_philox_gradients_with_heavy_tails():
    """Gradients drawn inside the kernels (W=32), per-tensor std scaled by
    1/sqrt(fan_in), every fifth tensor Student-t(3)."""
    t = workload.bert_tensors(2, 128, 512, 800)
    wl = workload.custom("large_mini_w32", t, W=32, chunk=4096, grad="philox", grad_std=1e-3,
                         fan_in_scaled=True, heavy_every=5, heavy_scale=1e-3)
    run(wl, 3, 3)


def test_single_worker():
    run(bert_mini(W=1, chunk=1024), 3, 3)


def test_single_element_and_tiny_tables():
    for tensors in ([("a", (1,))], [("a", (3,))], [("a", (2,)), ("b", (1,)), ("c", (5,))]):
        wl = workload.custom("small", tensors, W=2, chunk=256, grad_std=1e-2)
        run(wl, 2, 2)


def test_many_tensors_in_one_chunk():
    """A chunk that meets more tensors than the per-chunk shared-memory slots
    (200 tensors of 5 elements), so the per-tensor maximum also takes the
    global-atomic path."""
    t = [("big", (3000,))] + [(f"s{i}", (5,)) for i in range(200)] + [("tail", (777,))]
    wl = workload.custom("many", t, W=4, chunk=2048, grad_std=1e-2)
    run(wl, 2, 3)


def test_odd_worker_count_and_large_w():
    run(bert_mini(W=37, chunk=512), 1, 2)


def test_a_quarter_million_small_tensors():
    """250,000 tensors of 1 to 8 elements (W = 2, C = 1024): every chunk holds
    over a hundred tensors, far past the per-tile shared-memory slots of the
    per-tensor ratio maximum, and the per-tensor kernels run a quarter of a
    million CTAs or threads."""
    rng = np.random.default_rng(21)
    t = [(f"t{i}", (int(n),)) for i, n in enumerate(rng.integers(1, 9, 250_000))]
    run(workload.custom("many_small", t, W=2, chunk=1024, grad_std=1e-3), 1, 2)


def _small_table():
    return workload.bert_tensors(1, 32, 128, 300, max_pos=64) + [("tail", (37,))]


@pytest.mark.parametrize("W,chunk,grad,errors", [(256, 4096, "f32", 0), (255, 4096, "f32", 1),
                                                 (256, 1024, "bf16", 0), (255, 4096, "philox", 0)])
def test_maximum_worker_count(W, chunk, grad, errors):
    """The largest worker counts the C ABI accepts (256, and 255, which is
    not a power of two: the server average is a true division), in the
    stored-gradient, bfloat16-error three-CTA and in-kernel-gradient
    shapes."""
    kw = dict(heavy_every=5, heavy_scale=1e-3, fan_in_scaled=True) if grad == "philox" else {}
    wl = workload.custom("max_w", _small_table(), W=W, chunk=chunk, grad=grad, grad_std=1e-3, **kw)
    run(wl, 1, 2, error_storage=errors)


# ---- 1-bit Adam variant ------------------------------------------------------

def test_adam_variant_tiny_and_bert_mini():
    wl = workload.workloads()["tiny"]
    run(wl, wl.warmup_steps, wl.compress_steps, variant=1)
    run(bert_mini(W=8, chunk=2048), 4, 6, variant=1)


def test_adam_variant_in_kernel_gradients():
    t = workload.bert_tensors(1, 128, 512, 800)
    wl = workload.custom("adam_w32", t, W=32, chunk=4096, grad="philox", grad_std=1e-3,
                         fan_in_scaled=True, heavy_every=5, heavy_scale=1e-3)
    run(wl, 2, 2, variant=1)


# ---- non-finite inputs ---------------------------------------------------------

@pytest.mark.parametrize("error_storage", [0, 1])
def test_nonfinite_gradients_propagate_like_the_oracle(error_storage):
    """A NaN and an Inf gradient in one worker's chunk: NaN sends +1 (sign
    bit rule), the chunk's scale and errors become NaN, the server chunk
    follows, the tensor's ratio max counts NaN as +Inf; every word and every
    NaN position agrees with the oracle.  With bfloat16 error storage the
    stored error bits themselves, NaNs included (0x7FC0), equal the
    oracle's."""
    import numpy as np
    import torch
    wl = bert_mini(W=4, chunk=1024)
    p = Pair(wl, error_storage=error_storage)
    for _ in range(2):
        p.warmup()
    p.freeze()
    g_host = workload.grads_for_step(wl, p.t)
    g_host[1, 5000] = np.nan
    g_host[2, 70000] = np.inf
    g_dev = torch.zeros((wl.W, p.ld), device="cuda")
    g_dev[:, :wl.N] = torch.from_numpy(g_host).cuda()
    p.gpu.compress_step(g_dev)
    p.orc.compress_step(g_host)
    p.t += 1
    st = p.gpu_state()
    o = p.orc
    nw = st["nw"]
    np.testing.assert_array_equal(st["signs_w"][:, :nw], o.signs_w)
    np.testing.assert_array_equal(st["signs_s"][:nw], o.signs_s)
    for k in ("m", "e_s", "v_fresh"):
        np.testing.assert_array_equal(np.isnan(st[k][:wl.N]), np.isnan(getattr(o, k)), err_msg=k)
        fin = ~np.isnan(getattr(o, k))
        np.testing.assert_array_equal(st[k][:wl.N][fin], getattr(o, k)[fin], err_msg=k)
    np.testing.assert_array_equal(np.isnan(st["e_w"][:, :wl.N]), np.isnan(o.e_w))
    if error_storage:
        for k in ("e_w", "e_s"):
            got = np.ascontiguousarray(st[k][..., :wl.N]).view(np.uint32)
            want = np.ascontiguousarray(getattr(o, k)).view(np.uint32)
            assert np.isnan(getattr(o, k)).any(), k
            np.testing.assert_array_equal(got, want, err_msg=k)
    np.testing.assert_array_equal(np.isnan(st["scale_w"]), np.isnan(o.scale_w))
    np.testing.assert_array_equal(np.isnan(st["x"]), np.isnan(o.x))
    fin = ~np.isnan(o.x)
    np.testing.assert_array_equal(st["x"][fin], o.x[fin])
    assert np.isinf(o.R).any()
    np.testing.assert_array_equal(st["R_last"], o.R)


# ---- bfloat16 error storage ---------------------------------------------------

@pytest.mark.parametrize("variant", [0, 1])
def test_bf16_error_storage(variant):
    """Worker and server errors kept in bfloat16 (round to nearest even at
    store): bit-exact against the oracle's bf16-storage variant, 20 steps on
    the mini BERT table and the toy table, both method variants."""
    run(bert_mini(W=8, chunk=2048), 10, 10, variant=variant, error_storage=1)
    wl = workload.workloads()["tiny"]
    run(wl, wl.warmup_steps, wl.compress_steps, variant=variant, error_storage=1)


@pytest.mark.parametrize("variant", [0, 1])
def test_bf16_error_storage_4096(variant):
    """bfloat16 errors with 4096-element chunks and W = 16 (the BERT-Large
    shape of that option: three CTAs per SM, a 4-slot ring, and for 1-bit
    LAMB the server's late reads)."""
    run(bert_mini(W=16, chunk=4096), 4, 6, variant=variant, error_storage=1)


@pytest.mark.parametrize("W", [1, 2, 37])
@pytest.mark.parametrize("variant,errors", [(0, 1), (1, 0), (1, 1)])
def test_three_cta_shape_worker_counts(W, variant, errors):
    """The three-CTA, 4-slot shape (C = 4096 with bfloat16 errors or 1-bit
    Adam) with one, two and an odd number of workers: the copy ring's
    schedule changes with W (one worker item of two slots, or many), and
    the late server reads keep two slots to the end of every tile."""
    run(bert_mini(W=W, chunk=4096), 2, 3, variant=variant, error_storage=errors)


def test_bf16_error_storage_with_bf16_and_in_kernel_gradients():
    t = workload.gpt2_tensors(2, 48, 192, 500, n_pos=64)
    run(workload.custom("gpt2_mini", t, W=8, chunk=8192, grad="bf16", grad_std=1e-3), 2, 3,
        error_storage=1)
    t = workload.bert_tensors(1, 128, 512, 800)
    wl = workload.custom("w32", t, W=32, chunk=4096, grad="philox", grad_std=1e-3,
                         fan_in_scaled=True, heavy_every=5, heavy_scale=1e-3)
    run(wl, 1, 2, error_storage=1)


# ---- degenerate values -----------------------------------------------------------

def test_degenerate_values():
    """Zero, negative-zero, subnormal and constant gradients; an all-zero
    parameter tensor (trust ratio 1); parameter scales that clip the warmup
    trust ratio at both bounds; gradients that grow 100x after the freeze so
    the layerwise factor falls to its lower soft threshold.  Every step is
    compared with the oracle element by element, and all float state must be
    bit-identical."""
    import torch
    t = [("zero_x", (3000,)), ("zero_g", (5000,)), ("subnormal", (4096,)),
         ("const", (2055,)), ("negzero", (1000,)), ("tiny_x", (6000,)),
         ("huge_x", (4100,)), ("grows", (7000,)), ("normal", (9001,))]
    wl = workload.custom("degenerate", t, W=4, chunk=1024, grad_std=1e-2)
    off = {n: (int(o), int(o + k)) for (n, _), o, k in zip(t, wl.offsets, wl.numels)}
    p = Pair(wl)
    for name, scale in (("zero_x", 0.0), ("tiny_x", 1e-5), ("huge_x", 1e4)):
        a, b = off[name]
        p.x[a:b] *= scale
        p.orc.x[a:b] *= np.float32(scale)
    assert np.array_equal(p.x.cpu().numpy().view(np.uint32), p.orc.x.view(np.uint32))

    def grads(step, stage):
        g = workload.grads_for_step(wl, step)
        a, b = off["zero_g"]; g[:, a:b] = 0.0
        a, b = off["subnormal"]
        g[:, a:b] = np.where(g[:, a:b] < 0, -1e-40, 3e-41).astype(np.float32)
        a, b = off["const"]; g[:, a:b] = 3e-3
        a, b = off["negzero"]; g[:, a:b] = -0.0
        if stage == 1:
            a, b = off["grows"]; g[:, a:b] *= 100.0
        return g

    def step(kind, stage):
        g = grads(p.t, stage)
        dev = torch.from_numpy(g).cuda()
        if kind == "warmup":
            p.gpu.warmup_step(dev)
            p.orc.warmup_step(g)
        else:
            p.gpu.compress_step(dev)
            p.orc.compress_step(g)
        p.t += 1

    diffs = 0
    L = {n: i for i, (n, _) in enumerate(t)}
    for i in range(3):
        step("warmup", 0)
        diffs += p.compare(f"warmup {i}")
        if i == 0:
            assert p.orc.c_cur[L["zero_x"]] == np.float32(1.0)   # ||x|| = 0: ratio 1
    c = p.orc.c_cur
    assert c[L["tiny_x"]] == np.float32(wl.hp["coeff_min"])
    assert c[L["huge_x"]] == np.float32(wl.hp["coeff_max"])
    p.freeze()
    diffs += p.compare("freeze")
    for i in range(4):
        step("compress", 1)
        diffs += p.compare(f"compress {i}")
    r = p.orc.r_prev
    # soft threshold: r falls by at most 10 % a step from 1, floor 0.5
    assert r[L["grows"]] == np.float32(np.float32(np.float32(np.float32(0.9) * np.float32(0.9))
                                                  * np.float32(0.9)) * np.float32(0.9))
    assert diffs == 0, f"{diffs} float elements differ in some bit"
