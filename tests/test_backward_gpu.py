"""sdpa_forward_lse and sdpa_backward on the GPU against the fp64 oracle.

The backward pass reads the GPU forward's bf16 output O and its row
log-sum-exp.  It rounds P and dS to bf16 for the tensor-core products and
accumulates in fp32; the oracle differentiates the exact forward.

The bar comes from the roundings on the GPU side, each at most 2^-9 relative
(half a bf16 ulp):
  - P before dV;
  - dS before dK and dQ;
  - O, which enters D = <dO, O>;
  - a bf16 dK or dV output.
Two or three of these stack on each gradient.  So the bar is: relative RMS
error <= 2^-7 per gradient, and max|err| <= 2^-6 of the gradient's largest
entry.  dS = P (dP - D) subtracts nearly equal terms, so a few entries carry
more than the RMS.  The log-sum-exp is fp32 arithmetic on fp32 scores: within
1e-4 (log2 units) of the fp64 value.  A natural-log or missing-max slip moves
it by O(1)."""
import numpy as np
import pytest
import torch

import oracle
import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build
from transformer_head_scaled_03_gb300.inputs import Draws
from tests.gpu_util import assert_parity, to_dev, to_np

pytestmark = pytest.mark.gpu

NONE, CAUSAL, PAD = mha.MASK_NONE, mha.MASK_CAUSAL, mha.MASK_KEY_PADDING
RMS_REL, MAX_REL, LSE_ABS = 2.0 ** -7, 2.0 ** -6, 1e-4


@pytest.fixture(scope="module", autouse=True)
def built():
    mha_build.build()
    mha.lib()


def lse_reference(Q, K, scale, mask, lens):
    """fp64 base-2 log-sum-exp of the scaled, masked scores (the definition)."""
    Qd, Kd = Q.astype(np.float64), K.astype(np.float64)
    s = np.einsum("bhid,bhjd->bhij", Qd, Kd) * scale
    Lq, Lk = s.shape[-2:]
    blocked = np.zeros(s.shape, dtype=bool)
    if mask & CAUSAL:
        blocked |= np.triu(np.ones((Lq, Lk), dtype=bool), 1)[None, None]
    if mask & PAD:
        blocked |= (np.arange(Lk)[None, None, None, :] >= np.asarray(lens)[:, None, None, None])
    s = np.where(blocked, -np.inf, s)
    m = s.max(-1, keepdims=True)
    return (np.log(np.exp(s - m).sum(-1)) + m[..., 0]) / np.log(2.0)


def rel_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), "non-finite gradient"
    diff = got - ref
    scale = float(np.max(np.abs(ref))) or 1.0
    rms = float(np.sqrt(np.sum(diff * diff) / max(np.sum(ref * ref), 1e-300)))
    return float(np.max(np.abs(diff))) / scale, rms


def run_backward(seed, B, H, Lq, Lk, d, mask, lengths=None, grad_dtype=torch.bfloat16):
    g = Draws(seed)
    Q, K, V, dO = (g.normal(s) for s in ((B, H, Lq, d), (B, H, Lk, d), (B, H, Lk, d),
                                         (B, H, Lq, d)))
    lens = None if lengths is None else np.asarray(lengths, np.int32)
    kl = None if lens is None else torch.from_numpy(lens).cuda()
    q, k, v, do = (to_dev(a, torch.bfloat16) for a in (Q, K, V, dO))
    O, lse = mha.sdpa_forward_lse(q, k, v, mask_kind=mask, key_lengths=kl)
    dQ, dK, dV = mha.sdpa_backward(q, k, v, O, do, lse, mask_kind=mask, key_lengths=kl,
                                   grad_dtype=grad_dtype)
    assert mha.mha_check() == mha.MHA_OK
    return (Q, K, V, dO, lens), (to_np(O), to_np(lse)), (to_np(dQ), to_np(dK), to_np(dV))


CASES = [
    # B, H, Lq, Lk, d, mask, lengths, grad dtype
    (1, 2, 128, 128, 64, NONE, None, torch.bfloat16),
    (2, 2, 200, 300, 64, NONE, None, torch.float32),        # cross, ragged tiles
    (1, 2, 257, 257, 128, CAUSAL, None, torch.bfloat16),
    (2, 1, 300, 300, 64, CAUSAL, None, torch.float32),
    (3, 2, 130, 384, 128, PAD, [384, 129, 1], torch.bfloat16),
    (2, 2, 256, 256, 128, PAD | CAUSAL, [200, 256], torch.float32),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[:7]) for c in CASES])
def test_backward_parity(case):
    B, H, Lq, Lk, d, mask, lengths, gdt = case
    (Q, K, V, dO, lens), (O, lse), grads = run_backward(800 + CASES.index(case), B, H, Lq, Lk, d,
                                                       mask, lengths, gdt)
    scale = 1.0 / np.sqrt(d)
    assert_parity(O, oracle.sdpa(Q, K, V, mask_kind=mask, key_lengths=lens), torch.bfloat16,
                  "forward O")
    lse_err = float(np.max(np.abs(lse - lse_reference(Q, K, scale, mask, lens))))
    print(f"\n{case[:7]} lse: max|err| {lse_err:.3e}")
    assert lse_err <= LSE_ABS, lse_err
    refs = oracle.sdpa_backward(Q, K, V, dO, mask_kind=mask, key_lengths=lens)
    for name, got, ref in zip(("dQ", "dK", "dV"), grads, refs):
        mx, rms = rel_errors(got, ref)
        print(f"\n{case[:7]} {name}: max|err|/max|ref| {mx:.3e} rms rel {rms:.3e}")
        assert mx <= MAX_REL and rms <= RMS_REL, (name, mx, rms)


@pytest.mark.parametrize("shape", [(1, 2, 2048, 64), (1, 1, 4096, 128)])
def test_backward_long_causal_heads(shape):
    """Long causal heads (many key and query tiles, dQ summed over 16-32 key
    tiles), every gradient entry against the oracle."""
    B, H, L, d = shape
    (Q, K, V, dO, lens), _, grads = run_backward(850 + L, B, H, L, L, d, CAUSAL)
    refs = oracle.sdpa_backward(Q, K, V, dO, mask_kind=CAUSAL)
    for name, got, ref in zip(("dQ", "dK", "dV"), grads, refs):
        mx, rms = rel_errors(got, ref)
        print(f"\n{shape} {name}: max|err|/max|ref| {mx:.3e} rms rel {rms:.3e}")
        assert mx <= MAX_REL and rms <= RMS_REL, (name, mx, rms)


def test_backward_blocked_keys_get_zero_gradient():
    """Keys beyond a batch item's length get exactly zero dK and dV."""
    _, _, (dQ, dK, dV) = run_backward(870, 2, 2, 100, 300, 64, PAD, [40, 300])
    assert np.all(dK[0, :, 40:] == 0) and np.all(dV[0, :, 40:] == 0)


def test_backward_rejects_bad_arguments():
    q = torch.zeros((1, 1, 8, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mha.MhaError):           # d = 96
        mha.sdpa_backward(q, q, q, q, q, torch.zeros((1, 1, 8), device="cuda"))
    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    lib = mha.lib()
    import ctypes
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    ws = torch.zeros(4, dtype=torch.uint8, device="cuda")   # too small for 8 rows
    lse = torch.zeros((1, 1, 8), device="cuda")
    dq = torch.zeros((1, 1, 8, 64), device="cuda")
    st = lib.sdpa_backward(p(q), p(q), p(q), p(q), p(q), p(lse), p(dq), p(q), p(q), 1, 1, 8, 8,
                           64, 0.0, 0, None, mha.MHA_BF16, p(ws), 4, None)
    assert st == mha.MHA_ERR_INVALID_ARG
