"""The allocation-free entry point, lamb1b_tensor_sumsq_noalloc.

It serves callers that may not allocate device memory themselves (for
example a plug-in inside a framework whose caching allocator owns the GPU's
memory, or a latency-critical loop where cudaMalloc/cudaFree would
synchronise the device): its scratch is a fixed array inside the library.

Checked through the C ABI, bit for bit, against the CPU oracle's canonical
pairwise-tree sum of squares of every tensor (oracle.cpt_sumsq), on calls in
a row with different tables (each call reuses the scratch the previous one
left behind): a BERT-shaped table with odd offsets, a table whose tensors
start and end inside 256-element granules and one of whose tensors meets
more than 256 granules (the per-thread sequential part of the level-1
tree), and a table that fills most of the scratch's 2^22 half-granule
partial sums.  It is also checked bit for bit against the sums of squares
the warmup step computes for its trust ratio, which it promises to
reproduce.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import communication_compressed_optimizer_gb300 as pkg
import oracle
import workload
from communication_compressed_optimizer_gb300 import _abi
from harness import device_grads, grad_ld, layers_of

pytestmark = pytest.mark.gpu

MAX_HALVES = 1 << 22


def noalloc_sumsq(x, layers):
    out = torch.full((len(layers),), float("nan"), device="cuda")
    arr = pkg._layers_array(layers)
    rc = _abi.load().lamb1b_tensor_sumsq_noalloc(
        ctypes.c_void_p(x.data_ptr()), arr, len(layers), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out


def table(sizes):
    off = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    return list(zip(off.tolist(), [int(s) for s in sizes]))


def halves(layers):
    return sum(2 * ((o + n - 1) // 256 - o // 256 + 1) for o, n in layers)


def oracle_sums(xh, layers):
    return np.array([oracle.cpt_sumsq(xh, o, o + n) for o, n in layers], dtype=np.float32)


def check_against_oracle(xh, layers):
    x = torch.from_numpy(xh).cuda()
    rc, out = noalloc_sumsq(x, layers)
    assert rc == 0, _abi.load().lamb1b_error_string(rc)
    got = out.cpu().numpy()
    want = oracle_sums(xh, layers)
    bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
    assert bad.size == 0, (bad[:5], got[bad[:5]], want[bad[:5]])
    del x


def test_noalloc_equals_the_oracle_bit_for_bit_on_calls_in_a_row():
    rng = np.random.default_rng(11)
    # 1: BERT-shaped, odd offsets after the NSP/decoder biases
    t1 = workload.bert_tensors(2, 64, 256, 1000) + [("extra", (5,))]
    l1 = table([int(np.prod(s)) for _, s in t1])
    # 2: boundaries inside granules, a tensor over > 256 granules (70,001
    # elements meet 275), single-element and exactly-one-granule tensors
    l2 = table([100, 300, 70001, 1, 256, 5, 129, 4096 * 70 + 3, 77])
    assert max((o + n - 1) // 256 - o // 256 + 1 for o, n in l2) > 256
    for layers, scale in ((l1, 0.02), (l2, 1.0), (l1, 3.0)):
        N = layers[-1][0] + layers[-1][1]
        xh = (rng.standard_normal(N, dtype=np.float32) * np.float32(scale)).astype(np.float32)
        check_against_oracle(xh, layers)


def test_noalloc_near_its_scratch_limit():
    # 15 tensors of ragged sizes that together meet nearly 2^21 granules
    sizes = [int(v) for v in np.random.default_rng(3).integers(30_000_000, 36_000_000, 15)]
    layers = table(sizes)
    h = halves(layers)
    assert 0.9 * MAX_HALVES < h <= MAX_HALVES, h
    N = sum(sizes)
    xh = np.random.default_rng(4).random(N, dtype=np.float32)
    xh -= np.float32(0.5)
    check_against_oracle(xh, layers)


def test_noalloc_equals_warmup_step_norms_bit_for_bit():
    wl = workload.custom("a", workload.bert_tensors(2, 64, 256, 1000) + [("extra", (5,))],
                         W=4, chunk=1024, grad_std=1e-3)
    x = torch.from_numpy(workload.gen_params(wl)).cuda()
    opt = pkg.OneBitLamb(x, layers_of(wl), wl.W, wl.chunk, **wl.hp)
    ld = grad_ld(wl)
    for t in range(2):
        x_before = x.clone()
        opt.warmup_step(device_grads(wl, t, ld))
        rc, out = noalloc_sumsq(x_before, layers_of(wl))
        assert rc == 0, _abi.load().lamb1b_error_string(rc)
        torch.cuda.synchronize()
        want = opt.state()["Sx"][:wl.L]
        assert torch.equal(out.view(torch.int32), want.view(torch.int32))
    opt.close()


def test_noalloc_rejects_inputs_beyond_its_limits():
    x = torch.zeros(64, device="cuda")
    rc, _ = noalloc_sumsq(x, [(i, 1) for i in range(4097)])       # too many tensors
    assert rc == _abi.ERR_ARG
    rc, _ = noalloc_sumsq(x, [(0, 1 << 30)])                       # too long for the scratch
    assert rc == _abi.ERR_ARG
    rc, _ = noalloc_sumsq(x[1:], [(0, 8)])                         # misaligned vector
    assert rc == _abi.ERR_ALIGN


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_noalloc_refuses_a_capturing_stream():
    """The tables are staged from host memory local to the call, which a
    graph replay could not read: under stream capture the call returns
    LAMB1B_ERR_ARG and enqueues nothing."""
    x = torch.ones(1024, device="cuda")
    out = torch.full((1,), -1.0, device="cuda")
    arr = pkg._layers_array([(0, 1024)])
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    rcs = []
    with torch.cuda.graph(graph, stream=s):
        rcs.append(_abi.load().lamb1b_tensor_sumsq_noalloc(
            ctypes.c_void_p(x.data_ptr()), arr, 1, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(s.cuda_stream)))
    assert rcs == [_abi.ERR_ARG]
    torch.cuda.synchronize()
    assert out.item() == -1.0
    rc, got = noalloc_sumsq(x, [(0, 1024)])       # the same call outside a capture
    assert rc == 0 and got.item() == 1024.0
