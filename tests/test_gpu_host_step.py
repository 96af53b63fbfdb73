"""The compression step from host gradients, lamb1b_compress_step_host.

Its results must be the bits of lamb1b_compress_step on the same gradients
in device memory: checked step by step (the server message read back into
pinned host memory) and on the whole state afterwards, with fp32 and bf16
gradients, two staging buffers used in turn on a separate copy stream (a
step's copy overlapping the previous step's kernels), and more staging
buffers than the context remembers (the copy then waits for everything on
the step stream).  Argument errors are refused before anything is enqueued.
"""
import ctypes

import numpy as np
import pytest
import torch

import communication_compressed_optimizer_gb300 as pkg
import workload
from communication_compressed_optimizer_gb300 import _abi
from harness import layers_of

pytestmark = pytest.mark.gpu


def _mini(grad="f32"):
    t = workload.bert_tensors(2, 64, 256, 1000) + [("extra", (5,))]
    return workload.custom("host_step", t, W=4, chunk=1024, grad=grad, grad_std=1e-3)


def _host_grads(wl, t, ld):
    """Step t's gradients of every worker as a pinned host tensor [W, ld]."""
    if wl.grad == "bf16":
        g = np.zeros((wl.W, ld), np.uint16)
        for w in range(wl.W):
            g[w, :wl.N] = workload.gen_grads(wl, t, w, bf16_bits=True)
        return torch.from_numpy(g.view(np.int16)).pin_memory()
    return torch.from_numpy(workload.grads_for_step(wl, t, ld)).pin_memory()


def _pair(wl):
    x0 = torch.from_numpy(workload.gen_params(wl))
    xa, xb = x0.clone().cuda(), x0.clone().cuda()
    a = pkg.OneBitLamb(xa, layers_of(wl), wl.W, wl.chunk, **wl.hp)
    b = pkg.OneBitLamb(xb, layers_of(wl), wl.W, wl.chunk, **wl.hp)
    return a, b, xa, xb


def _bits(t):
    return t.contiguous().view(torch.int32).cpu().numpy() if t.element_size() == 4 else \
        t.contiguous().view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("grad,n_staging", [("f32", 2), ("bf16", 2), ("f32", 5)])
def test_host_step_equals_the_device_step_bit_for_bit(grad, n_staging):
    wl = _mini(grad)
    q = 8 if grad == "bf16" else 4
    ld = -(-wl.N // q) * q
    a, b, xa, xb = _pair(wl)
    for t in range(2):
        g = _host_grads(wl, t, ld).cuda()
        a.warmup_step(g)
        b.warmup_step(g)
    a.freeze_variance()
    b.freeze_variance()
    staging = [torch.empty((wl.W, ld), dtype=g.dtype, device="cuda") for _ in range(n_staging)]
    copy_stream = torch.cuda.Stream()
    nw, K = -(-wl.N // 32), -(-wl.N // wl.chunk)
    words = torch.empty(nw, dtype=torch.int32).pin_memory()
    scales = torch.empty(K, dtype=torch.float32).pin_memory()
    for i in range(6):
        h = _host_grads(wl, 2 + i, ld)
        a.compress_step(h.cuda())
        b.compress_step_host(h, staging[i % n_staging], words, scales, copy_stream=copy_stream)
        torch.cuda.synchronize()
        sa = a.state(sync=False)
        np.testing.assert_array_equal(words.numpy(), _bits(sa["signs_s"][:nw]), err_msg=f"step {i}")
        np.testing.assert_array_equal(scales.numpy().view(np.int32), _bits(sa["scale_s"][:K]))
    sa, sb = a.state(), b.state()
    for k in ("m", "v", "v_fresh", "e_w", "e_s", "signs_w", "signs_s", "scale_w", "scale_s", "c_cur",
              "r_prev", "R_last"):
        np.testing.assert_array_equal(_bits(sa[k]), _bits(sb[k]), err_msg=k)
    np.testing.assert_array_equal(_bits(xa), _bits(xb))
    a.close()
    b.close()


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_host_step_argument_errors():
    wl = _mini()
    ld = -(-wl.N // 4) * 4
    a, b, xa, xb = _pair(wl)
    lib = _abi.load()
    h = _host_grads(wl, 0, ld)
    staging = torch.empty((wl.W, ld), device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(ptr, stage_ptr, kind=pkg.GRAD_F32, stream=st):
        d = _abi.GradsDesc()
        d.kind, d.ptr, d.ld = kind, ptr, ld
        return lib.lamb1b_compress_step_host(a._ctx, ctypes.byref(d), ctypes.c_void_p(stage_ptr), None, None,
                                             stream, stream)

    assert call(h.data_ptr(), staging.data_ptr()) == _abi.ERR_STATE        # before the freeze
    a.warmup_step(h.cuda())
    a.freeze_variance()
    pageable = np.zeros((wl.W, ld), np.float32)
    assert call(pageable.ctypes.data, staging.data_ptr()) == _abi.ERR_ARG   # not pinned
    assert call(staging.data_ptr(), staging.data_ptr()) == _abi.ERR_ARG     # device memory as host
    assert call(h.data_ptr(), h.data_ptr()) == _abi.ERR_ARG                 # staging in host memory
    assert call(h.data_ptr(), staging.data_ptr() + 4) == _abi.ERR_ALIGN
    assert call(h.data_ptr(), staging.data_ptr(), kind=pkg.GRAD_PHILOX) == _abi.ERR_ARG
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    rcs = []
    with torch.cuda.graph(graph, stream=s):
        rcs.append(call(h.data_ptr(), staging.data_ptr(), stream=ctypes.c_void_p(s.cuda_stream)))
    assert rcs == [_abi.ERR_ARG]
    assert a.state(sync=False)["t"] == 1          # nothing above ran a step
    assert call(h.data_ptr(), staging.data_ptr()) == 0
    assert a.state(sync=False)["t"] == 2
    torch.cuda.synchronize()
    a.close()
    b.close()
