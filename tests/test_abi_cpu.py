"""The C-ABI library loads, exports every entry point the headers declare, and
rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

import communication_compressed_optimizer_gb300 as pkg
from communication_compressed_optimizer_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(lamb1b_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    L = _abi.load()
    names = declared_functions()
    assert "lamb1b_compress_step" in names and "lamb1b_gen_grads" in names
    for n in sorted(names):
        assert hasattr(L, n), n
    assert set(_abi.EXPORTED) <= names


def test_library_is_in_tree():
    assert os.path.commonpath([pkg.library_path(), ROOT]) == ROOT
    assert os.path.exists(pkg.library_path())


def _layers(numels):
    arr = (_abi.Layer * len(numels))()
    o = 0
    for i, n in enumerate(numels):
        arr[i].offset, arr[i].numel = o, n
        o += n
    return arr


def _hp(**kw):
    d = dict(pkg.DEFAULT_HP, **kw)
    return pkg._hparams(d.pop("W", 4), d.pop("chunk", 256), d)


def test_workspace_bytes_and_validation():
    L = _abi.load()
    arr = _layers([4096, 256, 4096, 1000])
    n = L.lamb1b_workspace_bytes(arr, 4, ctypes.byref(_hp()))
    N, K, W = 9448, 37, 4
    Np = K * 256
    assert n >= 4 * Np * (4 + W)          # m, v, v_fresh, e_s, e_w
    assert n % 256 == 0
    # more workers, more bytes
    assert L.lamb1b_workspace_bytes(arr, 4, ctypes.byref(_hp(W=8))) > n
    bad = [dict(W=0), dict(W=257), dict(chunk=100), dict(chunk=384), dict(chunk=16384),
           dict(beta1=1.0), dict(beta2=1.5), dict(eps=-1.0), dict(coeff_min=2.0, coeff_max=1.0),
           dict(factor_min=5.0), dict(factor_threshold=-0.1), dict(lr=float("nan")),
           dict(check_finite=2), dict(variant=2)]
    for kw in bad:
        assert L.lamb1b_workspace_bytes(arr, 4, ctypes.byref(_hp(**kw))) == 0, kw
    # tables: gaps, overlaps, empty tensors, no tensors
    broken = _layers([10, 10])
    broken[1].offset = 11
    assert L.lamb1b_workspace_bytes(broken, 2, ctypes.byref(_hp())) == 0
    assert L.lamb1b_workspace_bytes(_layers([10, 0]), 2, ctypes.byref(_hp())) == 0
    assert L.lamb1b_workspace_bytes(arr, 0, ctypes.byref(_hp())) == 0
    assert L.lamb1b_workspace_bytes(None, 4, ctypes.byref(_hp())) == 0


def test_init_rejects_bad_arguments_before_any_cuda_call():
    L = _abi.load()
    arr = _layers([300, 5])
    h = _hp()
    need = L.lamb1b_workspace_bytes(arr, 2, ctypes.byref(h))
    ctx = ctypes.c_void_p()
    fake = ctypes.c_void_p(0x10000)     # never dereferenced: checks fail first
    rc = L.lamb1b_init(ctypes.byref(ctx), arr, 2, ctypes.byref(h), None, fake, need, None)
    assert rc == _abi.ERR_ARG
    rc = L.lamb1b_init(ctypes.byref(ctx), arr, 2, ctypes.byref(h), ctypes.c_void_p(0x10004),
                       fake, need, None)
    assert rc == _abi.ERR_ALIGN
    rc = L.lamb1b_init(ctypes.byref(ctx), arr, 2, ctypes.byref(h), fake,
                       ctypes.c_void_p(0x10010), need, None)
    assert rc == _abi.ERR_ALIGN
    rc = L.lamb1b_init(ctypes.byref(ctx), arr, 2, ctypes.byref(h), fake, fake, need - 1, None)
    assert rc == _abi.ERR_WORKSPACE
    assert ctx.value is None
    assert L.lamb1b_init(None, arr, 2, ctypes.byref(h), fake, fake, need, None) == _abi.ERR_ARG


def test_null_context_calls():
    L = _abi.load()
    g = _abi.GradsDesc()
    assert L.lamb1b_warmup_step(None, ctypes.byref(g), None) == _abi.ERR_ARG
    assert L.lamb1b_compress_step(None, ctypes.byref(g), None) == _abi.ERR_ARG
    assert L.lamb1b_freeze_variance(None, None) == _abi.ERR_ARG
    assert L.lamb1b_state_view(None, None) == _abi.ERR_ARG
    assert L.lamb1b_set_counters(None, 0, 0, 0) == _abi.ERR_ARG
    assert L.lamb1b_check_status(None, None) == _abi.ERR_ARG
    assert L.lamb1b_set_fault_injection(None, -1, 0) == _abi.ERR_ARG
    assert L.lamb1b_sync_momentum(None, None) == _abi.ERR_ARG
    assert L.lamb1b_destroy(None) == 0
    for code in range(0, -9, -1):
        assert L.lamb1b_error_string(code)
    assert L.lamb1b_gen_params(None, 0, 10, 1.0, 0, None) == _abi.ERR_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi._build, "LIB", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _abi.load()
