"""The C ABI without a GPU: the library loads, exports every function that
include/mha.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mha.h")

NULL = None
OK, INVALID, UNSUPPORTED = mha.MHA_OK, mha.MHA_ERR_INVALID_ARG, mha.MHA_ERR_UNSUPPORTED
BF16, F32 = mha.MHA_BF16, mha.MHA_F32


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    mha_build.build()
    return mha.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sdpa_forward", "mha_create", "mha_forward", "mha_destroy", "mha_check",
              "mha_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(mha.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} is declared but not exported"


def test_status_strings(lib):
    for code, name in [(0, "MHA_OK"), (1, "MHA_ERR_INVALID_ARG"), (2, "MHA_ERR_UNSUPPORTED"),
                       (3, "MHA_ERR_CUDA"), (4, "MHA_ERR_OOM"), (5, "MHA_ERR_TIMEOUT"),
                       (6, "MHA_ERR_DEVICE")]:
        assert mha.status_string(code) == name


P = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced
MIS = ctypes.c_void_p(0x10008)    # misaligned


def sdpa(lib, Q=P, K=P, V=P, O=P, B=1, H=1, Lq=4, Lk=4, d=64, scale=0.0, mask=0, kl=NULL,
         dt=BF16, odt=BF16):
    return lib.sdpa_forward(Q, K, V, O, B, H, Lq, Lk, d, scale, mask, kl, dt, odt, NULL)


@pytest.mark.parametrize("kw,code", [
    (dict(Q=NULL), INVALID), (dict(O=NULL), INVALID), (dict(K=MIS), INVALID),
    (dict(B=-1), INVALID), (dict(Lk=0), INVALID), (dict(d=0), INVALID),
    (dict(scale=-1.0), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID), (dict(mask=4), INVALID), (dict(mask=-1), INVALID),
    (dict(mask=1, Lq=4, Lk=5), INVALID), (dict(mask=2, kl=NULL), INVALID),
    (dict(mask=2, kl=ctypes.c_void_p(0x10002)), INVALID),
    (dict(dt=7), INVALID), (dict(odt=9), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(d=32), UNSUPPORTED), (dict(d=256, dt=F32, odt=F32), UNSUPPORTED),
    (dict(dt=F32, odt=BF16), UNSUPPORTED),
])
def test_sdpa_rejects_before_launch(lib, kw, code):
    assert sdpa(lib, **kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(Lq=0)])
def test_empty_inputs_are_a_no_op(lib, kw):
    # nothing to compute: OK without touching the (null) pointers or the GPU
    assert sdpa(lib, Q=NULL, K=NULL, V=NULL, O=NULL, **kw) == OK


def test_mha_create_validation(lib):
    h = ctypes.c_void_p()
    assert lib.mha_create(None, 512, BF16, 1, 1, 1) == INVALID
    assert lib.mha_create(ctypes.byref(h), 0, BF16, 1, 1, 1) == INVALID
    assert lib.mha_create(ctypes.byref(h), 512, 5, 1, 1, 1) == INVALID
    assert lib.mha_create(ctypes.byref(h), 512, BF16, 0, 1, 1) == INVALID
    assert h.value is None


def test_mha_forward_null_handle(lib):
    assert lib.mha_forward(None, P, P, P, P, P, P, 1, 4, 4, 8, 0, NULL, P, NULL) == INVALID
    assert lib.mha_destroy(None) == OK


def test_wait_limit_setter(lib):
    prev = lib.mha_set_wait_limit_ms(1234)
    assert lib.mha_set_wait_limit_ms(prev) == 1234


def test_binding_fails_loudly_without_library(monkeypatch):
    from transformer_head_scaled_03_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", "/nonexistent/libmha_gb300.so")
    with pytest.raises(RuntimeError, match="missing"):
        _binding.lib()
