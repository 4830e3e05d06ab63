"""sdpa_forward_host: attention from host buffers, the copies overlapped with
the attention chunk by chunk.

Every head is independent, so a chunked run must give bit for bit what
sdpa_forward gives on device-resident copies of the same inputs.  Those in
turn are within the forward's bar of the fp64 oracle (tests/test_sdpa_gpu.py).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build
from transformer_head_scaled_03_gb300.inputs import Draws
from tests.gpu_util import assert_parity

pytestmark = pytest.mark.gpu

NONE, CAUSAL, PAD = mha.MASK_NONE, mha.MASK_CAUSAL, mha.MASK_KEY_PADDING


@pytest.fixture(scope="module", autouse=True)
def built():
    mha_build.build()
    mha.lib()


def host_inputs(seed, B, H, Lq, Lk, d, dtype):
    g = Draws(seed)
    arrs = [g.normal((B, H, L, d)) for L in (Lq, Lk, Lk)]
    return arrs, [torch.from_numpy(a).to(dtype).pin_memory() for a in arrs]


CASES = [
    # B, H, Lq, Lk, d, mask, lengths, in dtype, out dtype     chunking
    (1, 8, 300, 300, 128, CAUSAL, None, torch.bfloat16, torch.bfloat16),   # 8 chunks of 1 head
    (10, 2, 200, 333, 64, PAD, list(range(33, 333, 30)), torch.bfloat16, torch.float32),  # items
    (2, 3, 50, 70, 32, NONE, None, torch.float32, torch.float32),          # fp32, 6 chunks
    (3, 5, 129, 129, 64, CAUSAL | PAD, [129, 1, 64], torch.bfloat16, torch.bfloat16),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[:6]) for c in CASES])
def test_host_call_matches_device_call(case):
    B, H, Lq, Lk, d, mask, lengths, idt, odt = case
    (Q, K, V), (Qh, Kh, Vh) = host_inputs(1500 + CASES.index(case), B, H, Lq, Lk, d, idt)
    lens_h = torch.tensor(lengths, dtype=torch.int32).pin_memory() if lengths else None
    Oh = mha.sdpa_forward_host(Qh, Kh, Vh, mask_kind=mask, lengths_h=lens_h, out_dtype=odt)
    torch.cuda.current_stream().synchronize()
    assert mha.mha_check() == mha.MHA_OK
    kl = lens_h.cuda() if lens_h is not None else None
    Od = torch.empty((B, H, Lq, d), dtype=odt, device="cuda")
    mha.sdpa_forward(Qh.cuda(), Kh.cuda(), Vh.cuda(), mask_kind=mask, key_lengths=kl,
                     out_dtype=odt, out=Od)
    assert torch.equal(Oh, Od.cpu()), "chunked host call differs from the device call"
    if idt == torch.bfloat16:
        ref = oracle.sdpa(Qh.float().numpy(), Kh.float().numpy(), Vh.float().numpy(),
                          mask_kind=mask, key_lengths=None if lengths is None else np.asarray(
                              lengths, np.int32))
        assert_parity(Oh.float().numpy(), ref, idt, "host call")   # tensor-core bar


def test_back_to_back_calls_share_a_workspace():
    """Two calls on one stream, one workspace, no synchronisation between
    them: the second call's copies in must wait for the first call's
    attention, and both outputs must be right."""
    B, H, L, d = 1, 16, 512, 128
    lib = mha.lib()
    (_, (Q1, K1, V1)) = host_inputs(1600, B, H, L, L, d, torch.bfloat16)
    (_, (Q2, K2, V2)) = host_inputs(1601, B, H, L, L, d, torch.bfloat16)
    need = int(lib.sdpa_forward_host_workspace_bytes(B, H, L, L, d, mha.MHA_BF16, mha.MHA_BF16))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = [torch.empty((B, H, L, d), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    for (q, k, v), o in zip(((Q1, K1, V1), (Q2, K2, V2)), outs):
        st = lib.sdpa_forward_host(p(q), p(k), p(v), p(o), B, H, L, L, d, 0.0, CAUSAL, None,
                                   mha.MHA_BF16, mha.MHA_BF16, p(ws), need, s)
        assert st == mha.MHA_OK
    torch.cuda.current_stream().synchronize()
    for (q, k, v), o in zip(((Q1, K1, V1), (Q2, K2, V2)), outs):
        Od = mha.sdpa_forward(q.cuda(), k.cuda(), v.cuda(), mask_kind=CAUSAL)
        assert torch.equal(o, Od.cpu())


def test_rejects_bad_workspace():
    lib = mha.lib()
    B, H, L, d = 1, 2, 64, 64
    (_, (Q, K, V)) = host_inputs(1700, B, H, L, L, d, torch.bfloat16)
    O = torch.empty_like(Q).pin_memory()
    need = int(lib.sdpa_forward_host_workspace_bytes(B, H, L, L, d, mha.MHA_BF16, mha.MHA_BF16))
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    call = lambda w, n: lib.sdpa_forward_host(p(Q), p(K), p(V), p(O), B, H, L, L, d, 0.0, NONE,
                                              None, mha.MHA_BF16, mha.MHA_BF16, w, n, s)
    assert call(p(ws, 16), need) == mha.MHA_ERR_INVALID_ARG      # not 256-byte aligned
    assert call(p(ws), need - 256) == mha.MHA_ERR_INVALID_ARG    # too small
    assert call(p(ws), need) == mha.MHA_OK
    torch.cuda.current_stream().synchronize()
