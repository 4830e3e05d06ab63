"""encoder_forward (MHA with biases, residual + LayerNorm, ReLU FFN,
residual + LayerNorm) on the GPU against the fp64 oracle.

Tolerances: fp32 max|err| <= 1e-4.  bf16: max|err| <= 5e-2 and RMS relative
<= 1e-2 -- the layer output is a LayerNorm output with |y| up to ~5, where a
bf16 half-ulp alone is 0.0156, and four intermediate tensors (Q/K/V, context,
x1, the FFN hidden activation) are rounded to bf16 on the way."""
import numpy as np
import pytest
import torch

import oracle
import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build
from transformer_head_scaled_03_gb300.inputs import Draws, round_to_bf16
from tests.gpu_util import errors, to_dev, to_np

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_RMS, F32_MAX = 5e-2, 1e-2, 1e-4


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
        out = layer.forward(to_dev(x, dtype), {k: to_dev(v, dtype) for k, v in p.items()},
                            mask_kind=mk,
                            key_lengths=torch.from_numpy(lens).cuda() if lens is not None else None)
        assert mha.mha_check() == mha.MHA_OK
        got = to_np(out)
    finally:
        layer.close()
    ref = oracle.encoder_layer(x, p, h, mask_kind=mk, key_lengths=lens)
    max_abs, rms = errors(got, ref)
    if dtype == torch.bfloat16:
        assert max_abs <= BF16_MAX and rms <= BF16_RMS, (case, max_abs, rms)
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
