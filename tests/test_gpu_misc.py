"""GPU: on-device generator equals the host generator bit for bit;
determinism; checkpoint/resume; non-finite detection; call-order errors."""
import ctypes

import numpy as np
import pytest
import torch

import communication_compressed_optimizer_gb300 as pkg
import workload
from communication_compressed_optimizer_gb300 import _abi
from harness import Pair, device_grads, grad_ld, layers_of

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host_generator():
    t = workload.bert_tensors(1, 96, 384, 700) + [("odd", (7,))]
    for grad, heavy in (("f32", 0), ("bf16", 0), ("f32", 3)):
        wl = workload.custom("gen", t, W=5, chunk=256, grad=grad, grad_std=1e-3,
                             fan_in_scaled=True, heavy_every=heavy, heavy_scale=2e-3)
        ld = grad_ld(wl) + 8
        dt = torch.int16 if grad == "bf16" else torch.float32
        out = torch.zeros((wl.W, ld), dtype=dt, device="cuda")
        for step in (0, 7):
            pkg.gen_grads(out, step, wl.seed, layers_of(wl), wl.layer_std,
                          wl.layer_heavy if heavy else None, wl.heavy_scale)
            got = out.cpu().numpy()
            for w in range(wl.W):
                want = workload.gen_grads(wl, step, w, bf16_bits=(grad == "bf16"))
                if grad == "bf16":
                    np.testing.assert_array_equal(got[w, :wl.N].view(np.uint16), want)
                else:
                    np.testing.assert_array_equal(got[w, :wl.N].view(np.uint32), want.view(np.uint32))
                assert not np.any(got[w, wl.N:])
    # parameters, including a range that does not start on a multiple of 4
    wl = workload.workloads()["tiny"]
    x = torch.empty(wl.N - 5, device="cuda")
    pkg.gen_params(x, 5, wl.N, wl.param_std, wl.seed)
    np.testing.assert_array_equal(x.cpu().numpy().view(np.uint32),
                                  workload.gen_params(wl, 5, wl.N).view(np.uint32))


def test_device_philox_stream_many_counters():
    """2^24 consecutive elements (2^22 Philox counters) of one stream, device
    vs host, bit for bit."""
    wl = workload.custom("one", [("a", (1 << 24,))], W=1, chunk=256, grad_std=1.0)
    out = torch.empty((1, wl.N), device="cuda")
    pkg.gen_grads(out, 3, 12345, layers_of(wl), wl.layer_std)
    wl.seed = 12345
    want = workload.gen_grads(wl, 3, 0)
    np.testing.assert_array_equal(out.cpu().numpy()[0].view(np.uint32), want.view(np.uint32))


def test_device_transform_division_and_square_root_are_exact():
    """The device transform's divisions by (f+1) and by 3 and its square
    roots (Markstein's method) give the IEEE results on every input the
    transform can produce, enumerated completely by lamb1b_gen_selfcheck; its
    packed normals and Student-t values equal the plain one-operation-at-a-time
    evaluation over 2^22 counters."""
    counts = torch.full((5,), -1, dtype=torch.int64, device="cuda")
    rc = _abi.load().lamb1b_gen_selfcheck(ctypes.c_void_p(counts.data_ptr()), 2718,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, _abi.load().lamb1b_error_string(rc)
    assert counts.cpu().tolist() == [0, 0, 0, 0, 0]


def _bert_mini(W=4, chunk=1024):
    t = workload.bert_tensors(1, 64, 256, 500) + [("extra", (5,))]
    return workload.custom("bm", t, W=W, chunk=chunk, grad_std=1e-3)


def _run_gpu_only(wl, n_warm, n_comp, **opts):
    x = torch.from_numpy(workload.gen_params(wl)).cuda()
    opt = pkg.OneBitLamb(x, layers_of(wl), wl.W, wl.chunk, **dict(wl.hp, **opts))
    ld = grad_ld(wl)
    t = 0
    for _ in range(n_warm):
        opt.warmup_step(device_grads(wl, t, ld))
        t += 1
    opt.freeze_variance()
    for _ in range(n_comp):
        opt.compress_step(device_grads(wl, t, ld))
        t += 1
    torch.cuda.synchronize()
    return opt, x


@pytest.mark.parametrize("shape", ["512x2", "three_cta_bf16err", "draw_warps"])
def test_bitwise_deterministic(shape):
    """Two runs of the same steps leave the same bits everywhere (with the
    CPU parity this stands in for a race checker): the 512 x 2 tile, the
    three-CTA shape with late server reads, and the in-kernel-gradient
    kernel with its draw warps."""
    opts = {}
    if shape == "512x2":
        wl = _bert_mini(W=6, chunk=2048)
    elif shape == "three_cta_bf16err":
        wl = _bert_mini(W=6, chunk=4096)
        opts = dict(error_storage=1)
    else:
        t = workload.bert_tensors(1, 128, 512, 800)
        wl = workload.custom("w32", t, W=32, chunk=4096, grad="philox", grad_std=1e-3,
                             fan_in_scaled=True, heavy_every=5, heavy_scale=1e-3)
    a, xa = _run_gpu_only(wl, 3, 4, **opts)
    b, xb = _run_gpu_only(wl, 3, 4, **opts)
    assert torch.equal(xa.view(torch.int32), xb.view(torch.int32))
    assert torch.equal(a.workspace, b.workspace)


def _same_bits(a, b):
    it = torch.int32 if a.element_size() == 4 else torch.int16
    return torch.equal(a.contiguous().view(it), b.contiguous().view(it))


@pytest.mark.parametrize("chunk,variant,errors", [(1024, 0, 0), (4096, 0, 1), (4096, 1, 0), (2048, 1, 1)])
def test_checkpoint_resume_is_bitwise(chunk, variant, errors):
    """Save every state buffer after 3 warmup + 2 compression steps, restore
    them into a new context, run 4 more: bit for bit the uninterrupted run,
    for both method variants and both error storages."""
    wl = _bert_mini(chunk=chunk)
    opts = dict(variant=variant, error_storage=errors)
    ld = grad_ld(wl)
    ref, xr = _run_gpu_only(wl, 3, 6, **opts)
    # interrupted run: 3 warmup + 2 compression steps, save, restore, 4 more
    a, xa = _run_gpu_only(wl, 3, 2, **opts)
    sa = a.state()
    saved = {k: v.clone() for k, v in sa.items() if isinstance(v, torch.Tensor)}
    counters = (sa["t"], sa["n_warmup"], sa["stage"])
    x_saved = xa.clone()
    del a
    xb = x_saved.clone()
    b = pkg.OneBitLamb(xb, layers_of(wl), wl.W, wl.chunk, **dict(wl.hp, **opts))
    sb = b.state()
    for k, v in saved.items():
        sb[k].copy_(v)
    b.set_counters(*counters)
    t = counters[0]
    for _ in range(4):
        b.compress_step(device_grads(wl, t, ld))
        t += 1
    torch.cuda.synchronize()
    assert torch.equal(xb.view(torch.int32), xr.view(torch.int32))
    sr = ref.state()
    sb = b.state()
    for k in ("m", "v", "v_fresh", "e_s", "e_w", "signs_w", "signs_s", "scale_w", "scale_s",
              "r_prev", "c_cur", "c_bar"):
        assert _same_bits(sb[k], sr[k]), k


@pytest.mark.parametrize("chunk,variant,errors", [(1024, 0, 0), (4096, 0, 1), (4096, 1, 0)])
def test_copy_wait_timeout_is_reported_and_a_checkpoint_recovers(chunk, variant, errors):
    """Failure path without a GPU fault: the first CTA leaves out one of its
    shared-memory bulk copies, so its bounded wait for it runs out.  The step
    reports LAMB1B_ERR_TIMEOUT, the context stays usable, and restoring the
    state saved before the step continues bit for bit like an uninterrupted
    run.  Skipped copies: the first tile's momentum, a worker's gradient, a
    worker's error, the server error, and for 1-bit LAMB the fresh second
    moment (one of the two slots its server holds to the end of the tile).
    Shapes: a 7-slot ring, and the three-CTA shape's 4-slot ring."""
    wl = _bert_mini(chunk=chunk)
    opts = dict(variant=variant, error_storage=errors)
    ld = grad_ld(wl)
    ref, xr = _run_gpu_only(wl, 3, 4, **opts)
    a, xa = _run_gpu_only(wl, 3, 2, **opts)
    sa = a.state()
    saved = {k: v.clone() for k, v in sa.items() if isinstance(v, torch.Tensor)}
    counters = (sa["t"], sa["n_warmup"], sa["stage"])
    x_saved = xa.clone()
    t = counters[0]
    # copy positions of the first tile: 0 momentum, 1 + 2w gradient of worker
    # w, 2 + 2w its error, 1 + 2W server error, 2 + 2W frozen v, 3 + 2W v_fresh
    W = wl.W
    skips = (0, 5, 2 * W, 1 + 2 * W) + (() if variant else (3 + 2 * W,))
    for skip in skips:
        a.set_fault_injection(skip, 2000)
        a.compress_step(device_grads(wl, t, ld))
        with pytest.raises(pkg.Lamb1bError) as e:
            a.check_status()
        assert e.value.code == _abi.ERR_TIMEOUT, skip
        a.check_status()                      # cleared
        cur = a.state()
        for k, v in saved.items():
            cur[k].copy_(v)
        xa.copy_(x_saved)
        a.set_counters(*counters)
    a.set_fault_injection(-1, 0)
    for _ in range(2):
        a.compress_step(device_grads(wl, t, ld))
        t += 1
    a.check_status()
    torch.cuda.synchronize()
    assert torch.equal(xa.view(torch.int32), xr.view(torch.int32))
    sr, sb = ref.state(), a.state()
    for k in ("m", "v", "v_fresh", "e_s", "e_w", "signs_w", "signs_s", "scale_w", "scale_s",
              "r_prev", "c_cur", "c_bar"):
        assert _same_bits(sb[k], sr[k]), k


def test_copy_wait_timeout_with_draw_warps_recovers():
    """The same failure path in the in-kernel-gradient kernel (C = 4096: 512
    compressing threads plus 512 draw threads per CTA).  When the first CTA's
    compressing threads give up on a left-out copy they tell its draw warps
    to stop, so the CTA leaves instead of waiting; the step reports
    LAMB1B_ERR_TIMEOUT, and a restored checkpoint continues bit for bit.
    Skipped copies: the first tile's momentum, a worker's error, the server
    error, the fresh second moment."""
    t = workload.bert_tensors(1, 128, 512, 800)
    wl = workload.custom("w32", t, W=32, chunk=4096, grad="philox", grad_std=1e-3,
                         fan_in_scaled=True, heavy_every=5, heavy_scale=1e-3)
    ld = grad_ld(wl)
    ref, xr = _run_gpu_only(wl, 2, 4)
    a, xa = _run_gpu_only(wl, 2, 2)
    sa = a.state()
    saved = {k: v.clone() for k, v in sa.items() if isinstance(v, torch.Tensor)}
    counters = (sa["t"], sa["n_warmup"], sa["stage"])
    x_saved = xa.clone()
    t0 = counters[0]
    W = wl.W
    # copy positions of the first tile (gradients are drawn, not copied): 0
    # momentum, 1 + w worker w's error, 1 + W server error, 2 + W frozen
    # preconditioner, 3 + W fresh second moment
    for skip in (0, 5, 1 + W, 3 + W):
        a.set_fault_injection(skip, 2000)
        a.compress_step(device_grads(wl, t0, ld))
        with pytest.raises(pkg.Lamb1bError) as e:
            a.check_status()
        assert e.value.code == _abi.ERR_TIMEOUT, skip
        a.check_status()
        cur = a.state()
        for k, v in saved.items():
            cur[k].copy_(v)
        xa.copy_(x_saved)
        a.set_counters(*counters)
    a.set_fault_injection(-1, 0)
    for step in range(2):
        a.compress_step(device_grads(wl, t0 + step, ld))
    a.check_status()
    torch.cuda.synchronize()
    assert torch.equal(xa.view(torch.int32), xr.view(torch.int32))
    sr, sb = ref.state(), a.state()
    for k in ("m", "v_fresh", "e_s", "e_w", "signs_w", "signs_s", "scale_w", "scale_s",
              "r_prev", "c_cur"):
        assert torch.equal(sb[k].view(torch.int32), sr[k].view(torch.int32)), k


def test_compress_step_replays_from_a_cuda_graph():
    """A compression step only enqueues kernels on the caller's stream (no
    host synchronisation, no allocation), so it can be captured once in a
    CUDA graph and replayed: three replays of a captured step give the same
    device state, bit for bit, as three direct calls with the same gradients.
    (The host step counter advances on direct calls only.)"""
    wl = _bert_mini()
    ld = grad_ld(wl)
    a, xa = _run_gpu_only(wl, 3, 1)
    b, xb = _run_gpu_only(wl, 3, 1)
    g = device_grads(wl, 50, ld)
    for _ in range(3):
        a.compress_step(g)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        b.compress_step(g)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(xa.view(torch.int32), xb.view(torch.int32))
    sa, sb = a.state(), b.state()
    for k in ("m", "v", "v_fresh", "e_s", "e_w", "signs_w", "signs_s", "scale_w", "scale_s",
              "r_prev", "c_cur", "c_bar", "R_last"):
        assert torch.equal(sa[k].view(torch.int32), sb[k].view(torch.int32)), k


def test_fault_injection_arguments():
    wl = _bert_mini()
    x = torch.from_numpy(workload.gen_params(wl)).cuda()
    opt = pkg.OneBitLamb(x, layers_of(wl), wl.W, wl.chunk, **wl.hp)
    with pytest.raises(pkg.Lamb1bError):
        opt.set_fault_injection(-2, 0)
    opt.set_fault_injection(-1, 0)


def test_nonfinite_gradients_are_flagged():
    wl = _bert_mini()
    x = torch.from_numpy(workload.gen_params(wl)).cuda()
    opt = pkg.OneBitLamb(x, layers_of(wl), wl.W, wl.chunk, **dict(wl.hp, check_finite=1))
    ld = grad_ld(wl)
    g = device_grads(wl, 0, ld)
    opt.warmup_step(g)
    opt.check_status()                       # clean
    g[1, 123] = float("nan")
    opt.warmup_step(g)
    with pytest.raises(pkg.Lamb1bError) as e:
        opt.check_status()
    assert e.value.code == _abi.ERR_NONFINITE
    opt.check_status()                       # cleared
    opt.freeze_variance()
    g = device_grads(wl, 2, ld)
    g[0, 7] = float("inf")
    opt.compress_step(g)
    with pytest.raises(pkg.Lamb1bError):
        opt.check_status()


def test_call_order_and_argument_errors():
    wl = _bert_mini()
    x = torch.from_numpy(workload.gen_params(wl)).cuda()
    opt = pkg.OneBitLamb(x, layers_of(wl), wl.W, wl.chunk, **wl.hp)
    ld = grad_ld(wl)
    g = device_grads(wl, 0, ld)
    with pytest.raises(pkg.Lamb1bError) as e:
        opt.compress_step(g)
    assert e.value.code == _abi.ERR_STATE
    with pytest.raises(pkg.Lamb1bError) as e:
        opt.warmup_step(torch.zeros((wl.W, wl.N - 8), device="cuda"))   # ld < N
    assert e.value.code == _abi.ERR_ARG
    gbad = torch.zeros((wl.W, ld + 1), device="cuda")[:, :ld + 1]
    with pytest.raises(pkg.Lamb1bError) as e:
        opt.warmup_step(gbad)                    # ld*4 not a multiple of 16
    assert e.value.code == _abi.ERR_ALIGN
    opt.warmup_step(g)
    opt.freeze_variance()
    with pytest.raises(pkg.Lamb1bError) as e:
        opt.freeze_variance()
    assert e.value.code == _abi.ERR_STATE
    with pytest.raises(pkg.Lamb1bError) as e:
        opt.warmup_step(g)
    assert e.value.code == _abi.ERR_STATE
    # a failed check changed nothing: the step counter is still 1
    assert opt.state()["t"] == 1
    # host memory is not accepted as parameters (checked through the C ABI)
    import ctypes
    L = _abi.load()
    h = pkg._hparams(wl.W, wl.chunk, dict(pkg.DEFAULT_HP))
    arr = pkg._layers_array(layers_of(wl))
    host = np.zeros(wl.N + 64, np.float32)
    hp_ptr = (host.ctypes.data + 255) // 256 * 256
    ws = torch.empty(pkg.workspace_bytes(layers_of(wl), wl.W, wl.chunk), dtype=torch.uint8,
                     device="cuda")
    ctx = ctypes.c_void_p()
    rc = L.lamb1b_init(ctypes.byref(ctx), arr, len(arr), ctypes.byref(h), ctypes.c_void_p(hp_ptr),
                       ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
    assert rc == _abi.ERR_ARG and ctx.value is None
    # nor as gradients: rejected on the host before any launch
    hg = np.zeros(wl.W * ld + 64, np.float32)
    d = _abi.GradsDesc()
    d.kind, d.ld = pkg.GRAD_F32, ld
    d.ptr = (hg.ctypes.data + 255) // 256 * 256
    assert L.lamb1b_compress_step(opt._ctx, ctypes.byref(d), None) == _abi.ERR_ARG
    std_host = np.ones(wl.L + 16, np.float32)
    d = _abi.GradsDesc()
    d.kind, d.layer_std, d.heavy_scale = pkg.GRAD_PHILOX, (std_host.ctypes.data + 15) // 16 * 16, 1e-3
    assert L.lamb1b_compress_step(opt._ctx, ctypes.byref(d), None) == _abi.ERR_ARG
    assert opt.state()["t"] == 1
    # the generator and the allocation-free sums check their device pointers too
    assert L.lamb1b_gen_params(ctypes.c_void_p(hp_ptr), 0, 64, 1.0, 0, None) == _abi.ERR_ARG
    out = torch.zeros(len(arr), device="cuda")
    assert L.lamb1b_tensor_sumsq_noalloc(ctypes.c_void_p(hp_ptr), arr, len(arr),
                                         ctypes.c_void_p(out.data_ptr()), None) == _abi.ERR_ARG
    assert L.lamb1b_tensor_sumsq_noalloc(ctypes.c_void_p(x.data_ptr()), arr, len(arr),
                                         ctypes.c_void_p(hp_ptr), None) == _abi.ERR_ARG


def test_trace_events_time_every_kernel_of_a_step():
    """lamb1b_set_trace_events: four events around the three kernels of a
    step, recorded on the step's stream; then tracing off again."""
    wl = _bert_mini()
    x = torch.from_numpy(workload.gen_params(wl)).cuda()
    opt = pkg.OneBitLamb(x, layers_of(wl), wl.W, wl.chunk, **wl.hp)
    ld = grad_ld(wl)
    stream = torch.cuda.Stream()
    for stage in ("warmup", "compress"):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        opt.set_trace_events(ev)
        g = device_grads(wl, 0 if stage == "warmup" else 2, ld)
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            if stage == "warmup":
                opt.warmup_step(g, stream=stream)
            else:
                opt.compress_step(g, stream=stream)
        stream.synchronize()
        times = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
        assert all(t >= 0 for t in times) and ev[0].elapsed_time(ev[3]) > 0
        opt.set_trace_events(None)
        if stage == "warmup":
            opt.freeze_variance(stream=stream)
    with pytest.raises(pkg.Lamb1bError):
        _abi.check("lamb1b_set_trace_events", _abi.load().lamb1b_set_trace_events(opt._ctx, None, 4))
