"""mha_forward_noalloc, the entry point for callers that cannot allocate
device memory (a host that owns all device memory through its own pool, a
plugin whose execution step may not allocate, a latency-bound loop that
cannot take cudaMalloc's implicit synchronisation).

It is called here through the C ABI (ctypes on the library itself).  It runs
the same kernels as mha_forward -- whose workspace comes from cudaMalloc in
mha_create -- on the same inputs, so on consecutive calls that share the
library's fixed device array it must return exactly (bit for bit) what
mha_forward returns, and agree with the fp64 oracle within the parity
tolerances.  A call made after a warm-up call must leave the device's free
memory unchanged.  This file
sorts last so that a run stopping at its first failure has already run every
other test; it also builds and loads the library itself, so it passes when
run alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build
from transformer_head_scaled_03_gb300.inputs import Draws
from tests.gpu_util import assert_parity, to_dev, to_np

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 32 * 1024 * 1024   # MHA_NOALLOC_SCRATCH_BYTES in include/mha.h


@pytest.fixture(scope="module")
def lib():
    mha_build.build()
    L = ctypes.CDLL(mha.LIB_PATH)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    L.mha_forward_noalloc.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                      vp, vp, vp]
    L.mha_forward_noalloc.restype = i32
    return L


def ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def host_inputs(seed, dtype, B, Lq, Lk, D, cross):
    g = Draws(seed)
    st = "bf16" if dtype == torch.bfloat16 else "f32"
    xq = g.normal((B, Lq, D), dtype=st)
    xkv = g.normal((B, Lk, D), dtype=st) if cross else xq
    Ws = [g.normal((D, D), std=1.0 / np.sqrt(D), dtype=st) for _ in range(4)]
    return xq, xkv, Ws


def inputs(seed, dtype, B, Lq, Lk, D, cross):
    xq, xkv, Ws = host_inputs(seed, dtype, B, Lq, Lk, D, cross)
    dxq = to_dev(xq, dtype)
    return dxq, (to_dev(xkv, dtype) if cross else dxq), [to_dev(W, dtype) for W in Ws]


def with_handle(dtype, xq, xkv, Ws, h, mask, kl):
    B, Lq, D = xq.shape
    handle = mha.mha_create(D, dtype, B, Lq, xkv.shape[1])
    try:
        out = mha.mha_forward(handle, xq, xkv, *Ws, h=h, mask_kind=mask, key_lengths=kl)
        assert mha.mha_check(handle) == mha.MHA_OK
        return to_np(out)
    finally:
        handle.close()


def call_noalloc(lib, dtype, xq, xkv, Ws, h, mask, kl, out):
    B, Lq, D = xq.shape
    code = mha.MHA_BF16 if dtype == torch.bfloat16 else mha.MHA_F32
    st = lib.mha_forward_noalloc(D, code, ptr(xq), ptr(xkv), *(ptr(W) for W in Ws), B, Lq,
                                 xkv.shape[1], h, mask, ptr(kl), ptr(out),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mha.MHA_OK, mha.status_string(st)


def without_alloc(lib, dtype, xq, xkv, Ws, h, mask, kl):
    out = torch.empty_like(xq)
    call_noalloc(lib, dtype, xq, xkv, Ws, h, mask, kl, out)
    assert mha.mha_check() == mha.MHA_OK
    return to_np(out)


CASES = [
    # dtype, B, Lq, Lk, D, h, mask, lengths, cross
    (torch.bfloat16, 2, 200, 200, 512, 8, mha.MASK_CAUSAL, None, False),
    (torch.bfloat16, 2, 100, 300, 256, 2, mha.MASK_KEY_PADDING, [17, 300], True),
    (torch.float32, 1, 128, 128, 512, 8, mha.MASK_NONE, None, False),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_matches_handle_path_on_consecutive_calls(lib, case):
    """Bit for bit equal to mha_forward on two calls in a row (same kernels,
    same inputs), and within the parity bar of the fp64 oracle."""
    dtype, B, Lq, Lk, D, h, mask, lengths, cross = case
    hx = host_inputs(900 + CASES.index(case), dtype, B, Lq, Lk, D, cross)
    xq = to_dev(hx[0], dtype)
    xkv = to_dev(hx[1], dtype) if cross else xq
    Ws = [to_dev(W, dtype) for W in hx[2]]
    kl = torch.tensor(lengths, dtype=torch.int32, device="cuda") if lengths else None
    ref = with_handle(dtype, xq, xkv, Ws, h, mask, kl)
    first = without_alloc(lib, dtype, xq, xkv, Ws, h, mask, kl)
    second = without_alloc(lib, dtype, xq, xkv, Ws, h, mask, kl)
    assert np.array_equal(first, ref), float(np.max(np.abs(first - ref)))
    assert np.array_equal(second, ref), float(np.max(np.abs(second - ref)))
    lens = np.asarray(lengths, np.int32) if lengths else None
    expect = oracle.mha(hx[0], hx[1], *hx[2], h=h, mask_kind=mask, key_lengths=lens)
    assert_parity(first, expect, dtype, "against the oracle")


def test_a_call_allocates_no_device_memory(lib):
    """After a warm-up call (which may load kernel code), a second call leaves
    the device's free memory exactly where it was."""
    xq, xkv, Ws = inputs(920, torch.bfloat16, 2, 256, 256, 512, False)
    out = torch.empty_like(xq)
    call_noalloc(lib, torch.bfloat16, xq, xkv, Ws, 8, mha.MASK_CAUSAL, None, out)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    call_noalloc(lib, torch.bfloat16, xq, xkv, Ws, 8, mha.MASK_CAUSAL, None, out)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert mha.mha_check() == mha.MHA_OK
    assert free_after == free_before, (free_before, free_after)


def test_array_left_by_another_shape_does_not_leak(lib):
    """A call after a call of another shape (the array still holds the
    earlier intermediates) gives the same result as before."""
    a = inputs(910, torch.bfloat16, 1, 256, 256, 512, False)
    b = inputs(911, torch.bfloat16, 3, 64, 64, 1024, False)
    before = without_alloc(lib, torch.bfloat16, a[0], a[1], a[2], 8, mha.MASK_NONE, None)
    without_alloc(lib, torch.bfloat16, b[0], b[1], b[2], 16, mha.MASK_CAUSAL, None)
    after = without_alloc(lib, torch.bfloat16, a[0], a[1], a[2], 8, mha.MASK_NONE, None)
    assert np.array_equal(after, before)


def test_rejects_sizes_beyond_the_array(lib):
    # bf16, B1 L2048 D4096: 4 * 16 MiB of intermediates > 32 MiB
    B, L, D = 1, 2048, 4096
    assert 4 * B * L * D * 2 > SCRATCH_LIMIT
    x = torch.zeros((B, L, D), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((D, D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    st = lib.mha_forward_noalloc(D, mha.MHA_BF16, ptr(x), ptr(x), ptr(W), ptr(W), ptr(W), ptr(W),
                                 B, L, L, 32, mha.MASK_NONE, None, ptr(out), None)
    assert st == mha.MHA_ERR_INVALID_ARG
