"""encoder_forward (MHA with biases, residual + LayerNorm, ReLU FFN,
residual + LayerNorm) on the GPU against the fp64 oracle.

Tolerances: an fp32 layer, max|err| <= 1e-4.  A bf16 layer is graded on its
output kept in fp32 (out_dtype float32): max|err| <= 2e-2 and RMS relative
<= 1e-2, the bar for bf16 inputs with fp32 accumulation.  Its bf16 output is
that same result rounded once more; the test reports its error and bounds it
by the bar plus the rounding's own half-ulp, 2^-8 of the largest |y|
(LayerNorm outputs reach |y| ~ 5, where half an ulp is 0.0156)."""
import numpy as np
import pytest
import torch

import oracle
import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build
from transformer_head_scaled_03_gb300.inputs import Draws, round_to_bf16
from tests.gpu_util import errors, to_dev, to_np

pytestmark = pytest.mark.gpu

from tests.gpu_util import BF16_MAX_ABS as BF16_MAX, BF16_RMS_REL as BF16_RMS, F32_MAX_ABS as F32_MAX


@pytest.fixture(scope="module", autouse=True)
def built():
    mha_build.build()
    mha.lib()


def make_params(g, D, F, st):
    p = {}
    for n in ("Wq", "Wk", "Wv", "Wo"):
        p[n] = g.normal((D, D), std=1.0 / np.sqrt(D), dtype=st)
    p["W1"] = g.normal((D, F), std=1.0 / np.sqrt(D), dtype=st)
    p["W2"] = g.normal((F, D), std=1.0 / np.sqrt(F), dtype=st)
    for n in ("bq", "bk", "bv", "bo", "b2", "ln1_beta", "ln2_beta"):
        p[n] = g.normal((D,), std=0.1, dtype=st)
    p["b1"] = g.normal((F,), std=0.1, dtype=st)
    for n in ("ln1_gamma", "ln2_gamma"):
        v = 1.0 + g.normal((D,), std=0.1, dtype="f32")
        p[n] = v if st == "f32" else round_to_bf16(v)
    return p


CASES = [
    # dtype, B, L, D, h, F, mask, lengths
    (torch.bfloat16, 2, 128, 512, 8, 2048, mha.MASK_NONE, None),
    (torch.bfloat16, 1, 200, 256, 4, 1024, mha.MASK_CAUSAL, None),
    (torch.bfloat16, 3, 64, 512, 4, 512, mha.MASK_KEY_PADDING, [64, 10, 33]),
    # d_model 384: the fused epilogue's MMA split 256 + 128 columns, 100 rows
    (torch.bfloat16, 1, 100, 384, 6, 1536, mha.MASK_NONE, None),
    # d_model 1024: the seven-launch form (residual + LayerNorm as own launches)
    (torch.bfloat16, 2, 96, 1024, 8, 1024, mha.MASK_CAUSAL, None),
    # more 128-row tiles than SMs: CTAs of the fused epilogue GEMMs take a
    # second tile (the accumulator handed back, the next tile's residual
    # prefetched); 20480 and 19968 rows, d_model 256 and 512
    (torch.bfloat16, 128, 160, 256, 4, 512, mha.MASK_NONE, None),
    (torch.bfloat16, 48, 416, 512, 8, 1024, mha.MASK_KEY_PADDING, [200 + 4 * i for i in range(48)]),
    # d_model 320 and 192 (an odd number of 64-column blocks): the fused
    # epilogue GEMMs in their single-CTA form (even counts run as CTA pairs),
    # the second with more 128-row tiles than SMs
    (torch.bfloat16, 2, 150, 320, 5, 640, mha.MASK_CAUSAL, None),
    (torch.bfloat16, 64, 320, 192, 3, 384, mha.MASK_NONE, None),
    # d_model 128: the CTA-pair form with one 128-column chunk (one block of
    # W per CTA); d_model 64: the single-CTA form, where the second epilogue
    # warp of each lane quarter has no chunk of its own
    (torch.bfloat16, 4, 96, 128, 2, 256, mha.MASK_CAUSAL, None),
    (torch.bfloat16, 2, 100, 64, 1, 128, mha.MASK_KEY_PADDING, [100, 37]),
    (torch.float32, 1, 128, 512, 8, 2048, mha.MASK_NONE, None),
    (torch.float32, 2, 50, 96, 3, 200, mha.MASK_CAUSAL, None),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_encoder_layer_parity(case):
    dtype, B, L, D, h, F, mk, lengths = case
    st = "bf16" if dtype == torch.bfloat16 else "f32"
    g = Draws(700 + CASES.index(case))
    x = g.normal((B, L, D), dtype=st)
    p = make_params(g, D, F, st)
    lens = np.asarray(lengths, np.int32) if lengths else None
    layer = mha.EncoderLayer(D, h, F, dtype, B, L)
    try:
        dx = to_dev(x, dtype)
        dp = {k: to_dev(v, dtype) for k, v in p.items()}
        kl = torch.from_numpy(lens).cuda() if lens is not None else None
        out = layer.forward(dx, dp, mask_kind=mk, key_lengths=kl)
        out32 = (layer.forward(dx, dp, mask_kind=mk, key_lengths=kl, out_dtype=torch.float32)
                 if dtype == torch.bfloat16 else None)
        assert mha.mha_check() == mha.MHA_OK
        got = to_np(out)
        got32 = to_np(out32) if out32 is not None else None
        rounded = out32.to(torch.bfloat16) if out32 is not None else None
    finally:
        layer.close()
    ref = oracle.encoder_layer(x, p, h, mask_kind=mk, key_lengths=lens)
    max_abs, rms = errors(got, ref)
    if dtype == torch.bfloat16:
        max32, rms32 = errors(got32, ref)
        assert max32 <= BF16_MAX and rms32 <= BF16_RMS, (case, "fp32 out", max32, rms32)
        bound = BF16_MAX + 2.0 ** -8 * float(np.max(np.abs(ref)))
        assert max_abs <= bound and rms <= BF16_RMS, (case, "bf16 out", max_abs, bound, rms)
        if D <= 512:
            # one kernel computes both; only the final store differs
            assert torch.equal(rounded, out), case
        print(f"\nencoder {case[1:6]} bf16: fp32 out max|err| {max32:.3e} rms rel {rms32:.3e}; "
              f"bf16 out max|err| {max_abs:.3e} (bound {bound:.3e}) rms rel {rms:.3e}")
    else:
        assert max_abs <= F32_MAX, (case, max_abs)
        print(f"\nencoder {case[1:6]} {st}: max|err| {max_abs:.3e} rms rel {rms:.3e}")


def test_encoder_rejects_unsupported_shapes():
    with pytest.raises(mha.MhaError):
        mha.EncoderLayer(512, 8, 2000, torch.bfloat16, 1, 16)   # d_ff not a multiple of 64
    with pytest.raises(mha.MhaError):
        mha.EncoderLayer(512, 2, 2048, torch.bfloat16, 1, 16)   # head size 256
    D, F = 96, 128
    layer = mha.EncoderLayer(D, 3, F, torch.float32, 1, 16)
    try:
        p = {k: torch.from_numpy(v).cuda()
             for k, v in make_params(Draws(1), D, F, "f32").items()}
        with pytest.raises(mha.MhaError):                       # B above the maximum
            layer.forward(torch.zeros((2, 16, D), device="cuda"), p)
        with pytest.raises(mha.MhaError):                       # L above the maximum
            layer.forward(torch.zeros((1, 17, D), device="cuda"), p)
    finally:
        layer.close()


def test_encoder_layer_is_deterministic():
    """The layer's sums have fixed orders (no atomics; the two epilogue warps
    of a row merge their statistics in one order; CTA pairs split rows and
    columns, never a sum across CTAs), so repeated calls give the same bits.
    20,480 rows at d_model 256: more CTA-pair tiles than pairs resident."""
    B, L, D, h, F = 64, 320, 256, 4, 1024
    st = "bf16"
    g = Draws(77)
    p = {k: torch.from_numpy(v).to(torch.bfloat16).cuda()
         for k, v in make_params(g, D, F, st).items()}
    x = torch.from_numpy(g.normal((B, L, D), dtype=st)).to(torch.bfloat16).cuda()
    lens = torch.from_numpy(g.integers(L // 2, L, B)).cuda()
    layer = mha.EncoderLayer(D, h, F, torch.bfloat16, B, L)
    try:
        outs = [layer.forward(x, p, mask_kind=mha.MASK_KEY_PADDING, key_lengths=lens,
                              out_dtype=torch.float32).clone() for _ in range(4)]
        assert mha.mha_check() == mha.MHA_OK
    finally:
        layer.close()
    assert bool(torch.isfinite(outs[0]).all())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
