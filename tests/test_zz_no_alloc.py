"""The allocation-free entry point, lamb1b_tensor_sumsq_noalloc.

It serves callers that may not allocate device memory themselves (for
example a plug-in inside a framework whose caching allocator owns the GPU's
memory, or a latency-critical loop where cudaMalloc/cudaFree would
synchronise the device): its scratch is a fixed array inside the library.
Here it is checked, through the C ABI, against the per-tensor sums of squares
that the warmup step (lamb1b_warmup_step) computes for its trust ratio, on
consecutive calls, including a call with a different tensor table that
reuses the scratch the previous call left behind.

The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

import communication_compressed_optimizer_gb300 as pkg
import workload
from communication_compressed_optimizer_gb300 import _abi
from harness import close_scalar, device_grads, grad_ld, layers_of

pytestmark = pytest.mark.gpu


def noalloc_sumsq(x, layers):
    out = torch.full((len(layers),), float("nan"), device="cuda")
    arr = pkg._layers_array(layers)
    rc = _abi.load().lamb1b_tensor_sumsq_noalloc(
        ctypes.c_void_p(x.data_ptr()), arr, len(layers), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out


def tables():
    a = workload.custom("a", workload.bert_tensors(2, 64, 256, 1000) + [("extra", (5,))],
                        W=4, chunk=1024, grad_std=1e-3)
    b = workload.workloads()["tiny"]
    return a, b


def test_noalloc_matches_warmup_step_norms_on_consecutive_calls():
    for wl in tables():
        x = torch.from_numpy(workload.gen_params(wl)).cuda()
        opt = pkg.OneBitLamb(x, layers_of(wl), wl.W, wl.chunk, **wl.hp)
        ld = grad_ld(wl)
        for t in range(2):
            x_before = x.clone()
            opt.warmup_step(device_grads(wl, t, ld))
            rc, out = noalloc_sumsq(x_before, layers_of(wl))
            assert rc == 0, pkg._abi.load().lamb1b_error_string(rc)
            torch.cuda.synchronize()
            want = opt.state()["Sx"].cpu().numpy()
            assert close_scalar(out.cpu().numpy(), want)
        opt.close()


def test_noalloc_rejects_inputs_beyond_its_limits():
    x = torch.zeros(64, device="cuda")
    rc, _ = noalloc_sumsq(x, [(i, 1) for i in range(4097)])       # too many tensors
    assert rc == _abi.ERR_ARG
    rc, _ = noalloc_sumsq(x, [(0, 1 << 30)])                       # too long for the scratch
    assert rc == _abi.ERR_ARG
    rc, _ = noalloc_sumsq(x[1:], [(0, 8)])                         # misaligned vector
    assert rc == _abi.ERR_ALIGN
