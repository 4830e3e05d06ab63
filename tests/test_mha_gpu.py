"""mha_forward (projections with head-split stores, attention with the
concat store, output projection) on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build
from transformer_head_scaled_03_gb300.inputs import WORKLOADS, Draws, mha_inputs
from tests.gpu_util import assert_parity, to_dev, to_np

pytestmark = pytest.mark.gpu

NONE, CAUSAL, PAD = mha.MASK_NONE, mha.MASK_CAUSAL, mha.MASK_KEY_PADDING


@pytest.fixture(scope="module", autouse=True)
def built():
    mha_build.build()
    mha.lib()


def run_mha(seed, dtype, B, Lq, Lk, D, h, mask=NONE, lengths=None, cross=False):
    g = Draws(seed)
    st = "bf16" if dtype == torch.bfloat16 else "f32"
    xq = g.normal((B, Lq, D), dtype=st)
    xkv = g.normal((B, Lk, D), dtype=st) if cross else xq
    Ws = [g.normal((D, D), std=1.0 / np.sqrt(D), dtype=st) for _ in range(4)]
    lens = None if lengths is None else np.asarray(lengths, np.int32)
    handle = mha.mha_create(D, dtype, B, Lq, Lk)
    try:
        dxq = to_dev(xq, dtype)
        dxkv = to_dev(xkv, dtype) if cross else dxq
        dW = [to_dev(W, dtype) for W in Ws]
        kl = torch.from_numpy(lens).cuda() if lens is not None else None
        out = mha.mha_forward(handle, dxq, dxkv, *dW, h=h, mask_kind=mask, key_lengths=kl)
        assert mha.mha_check(handle) == mha.MHA_OK
        got = to_np(out)
    finally:
        handle.close()
    ref = oracle.mha(xq, xkv, *Ws, h=h, mask_kind=mask, key_lengths=lens)
    return got, ref


CASES = [
    # dtype, B, Lq, Lk, D, h, mask, lengths, cross
    (torch.bfloat16, 1, 128, 128, 512, 8, NONE, None, False),
    (torch.bfloat16, 2, 200, 200, 256, 2, CAUSAL, None, False),
    (torch.bfloat16, 2, 100, 300, 512, 4, PAD, [17, 300], True),
    (torch.bfloat16, 1, 129, 257, 1024, 16, NONE, None, True),
    (torch.bfloat16, 3, 64, 64, 384, 3, PAD | CAUSAL, [1, 64, 40], False),
    (torch.float32, 1, 128, 128, 512, 8, NONE, None, False),
    (torch.float32, 2, 70, 70, 96, 3, CAUSAL, None, False),
    (torch.float32, 2, 33, 90, 128, 4, PAD, [90, 5], True),
    # fp32 projections in both GEMM forms and both load paths: 32 x 64 tiles
    # (enough rows to fill the GPU) and the split-k 16 x 32 tiles, with
    # D a multiple of 4 (16-byte copies) and not (element loads; d = 30)
    (torch.float32, 8, 512, 512, 256, 4, NONE, None, False),
    (torch.float32, 4, 300, 300, 90, 3, NONE, None, False),
    (torch.float32, 3, 50, 70, 90, 3, PAD, [70, 1, 33], True),
    # fp32 self-attention: key padding with a length of 1, causal + padding,
    # 512 rows, d = 128
    (torch.float32, 4, 100, 100, 256, 4, PAD, [100, 1, 57, 99], False),
    (torch.float32, 3, 64, 64, 192, 6, PAD | CAUSAL, [64, 7, 33], False),
    (torch.float32, 2, 256, 256, 384, 6, CAUSAL, None, False),
    (torch.float32, 1, 200, 200, 512, 4, NONE, None, False),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{'bf16' if c[0] == torch.bfloat16 else 'f32'}-{c[1:]}" for c in CASES])
def test_mha_parity(case):
    dtype, B, Lq, Lk, D, h, mask, lengths, cross = case
    got, ref = run_mha(300 + CASES.index(case), dtype, B, Lq, Lk, D, h, mask, lengths, cross)
    assert_parity(got, ref, dtype, str(case))


def test_mha_base_shape_fp32_workload():
    """The base-shape layer (B1 L128 D512 h8, fp32, W ~ N(0, 1/512)) on its
    own seeded inputs, full output against the oracle within 1e-4."""
    w = WORKLOADS[1]
    x, Wq, Wk, Wv, Wo = mha_inputs(w)
    handle = mha.mha_create(w.D, torch.float32, w.B, w.Lq, w.Lk)
    try:
        dx = to_dev(x, torch.float32)
        out = mha.mha_forward(handle, dx, dx, *(to_dev(W, torch.float32) for W in (Wq, Wk, Wv, Wo)),
                              h=w.H)
        assert mha.mha_check(handle) == mha.MHA_OK
        got = to_np(out)
    finally:
        handle.close()
    ref = oracle.mha(x, x, Wq, Wk, Wv, Wo, h=w.H)
    max_abs, rms = assert_parity(got, ref, torch.float32, "base-shape fp32 layer")
    print(f"\n{w.name}: all {got.size} outputs, max|err| {max_abs:.3e}, rms rel {rms:.3e}")


def test_mha_rejects_sizes_above_handle_maxima():
    handle = mha.mha_create(256, torch.bfloat16, 1, 64, 64)
    try:
        x = torch.zeros((1, 65, 256), dtype=torch.bfloat16, device="cuda")
        W = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(mha.MhaError):
            mha.mha_forward(handle, x, x, W, W, W, W, h=4)
    finally:
        handle.close()


@pytest.mark.parametrize("dtype,B,L,D,h", [(torch.bfloat16, 2, 300, 512, 8),
                                           (torch.float32, 1, 128, 512, 8)])
def test_mha_permutation_equivariance(dtype, B, L, D, h):
    """Self-attention with no mask and no positional encoding is
    permutation-equivariant ("The Transformer" (rayaq.ca), "Embeddings and
    positions": reorder the words and every output is reordered with them).
    Permuting the positions of x on the device permutes the rows of the
    layer's output the same way, within the parity bar of the dtype; the
    two results differ only in the order the keys are summed in."""
    g = Draws(350 + L)
    st = "bf16" if dtype == torch.bfloat16 else "f32"
    x = g.normal((B, L, D), dtype=st)
    Ws = [to_dev(g.normal((D, D), std=1.0 / np.sqrt(D), dtype=st), dtype) for _ in range(4)]
    perm = np.stack([g.rng.permutation(L) for _ in range(B)])
    xp = np.stack([x[b, perm[b]] for b in range(B)])
    handle = mha.mha_create(D, dtype, B, L, L)
    try:
        dx, dxp = to_dev(x, dtype), to_dev(xp, dtype)
        out = to_np(mha.mha_forward(handle, dx, dx, *Ws, h=h))
        out_p = to_np(mha.mha_forward(handle, dxp, dxp, *Ws, h=h))
        assert mha.mha_check(handle) == mha.MHA_OK
    finally:
        handle.close()
    moved = np.stack([out[b, perm[b]] for b in range(B)])
    assert not np.array_equal(xp, x)
    max_abs, rms = assert_parity(out_p, moved, dtype, "permuted positions")
    print(f"\npermutation {st}: max|out(Px) - P out(x)| {max_abs:.3e}, rms rel {rms:.3e}")
