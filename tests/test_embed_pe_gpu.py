"""sinusoidal_pe and embed_pe_forward (token embedding x sqrt(D) + positional
encoding, one pass) on the GPU against the fp64 oracle.

Tolerances, from the arithmetic: the PE table is the fp64 value rounded to
fp32 (|err| <= 2^-24 for |v| <= 1, so 1e-7).  x is fma(e, sqrt(D), pe) in
fp32 rounded once to the storage type: bf16 |err| <= 2^-8 |x| (half an ulp)
+ 1e-6, fp32 |err| <= 1e-6 (|x| + 1)."""
import numpy as np
import pytest
import torch

import oracle
import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build
from transformer_head_scaled_03_gb300.inputs import Draws
from tests.gpu_util import assert_parity, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    mha_build.build()
    mha.lib()


@pytest.mark.parametrize("n_pos,D,first", [(5000, 512, 0), (300, 7, 100), (33, 4096, 32735)])
def test_pe_table(n_pos, D, first):
    got = to_np(mha.sinusoidal_pe(n_pos, D, first_pos=first))
    ref = oracle.sinusoidal_pe(n_pos, D, first_pos=first)
    err = float(np.max(np.abs(got - ref)))
    assert err <= 1e-7, err
    assert mha.mha_check() == mha.MHA_OK


def check_x(got, ref, dtype):
    err = np.abs(got - ref)
    if dtype == torch.bfloat16:
        bound = 2.0 ** -8 * np.abs(ref) + 1e-6
    else:
        bound = 1e-6 * (np.abs(ref) + 1.0)
    worst = float(np.max(err - bound))
    assert worst <= 0.0, f"max|err| {float(err.max()):.3e} exceeds the bound by {worst:.3e}"
    return float(err.max())


@pytest.mark.parametrize("dtype,B,L,D,vocab,off", [
    (torch.bfloat16, 3, 200, 512, 1000, 37),
    (torch.bfloat16, 2, 50, 100, 64, 0),      # D not a multiple of 8: element-wise path
    (torch.float32, 2, 77, 96, 500, 5),
    (torch.bfloat16, 1, 1, 4096, 10, 4095),
])
def test_embed_pe_parity(dtype, B, L, D, vocab, off):
    g = Draws(1100 + D)
    st = "bf16" if dtype == torch.bfloat16 else "f32"
    table = g.normal((vocab, D), std=1.0 / np.sqrt(D), dtype=st)
    ids = g.integers(0, vocab - 1, (B, L))
    pe = mha.sinusoidal_pe(off + L, D)
    x = mha.embed_pe(torch.from_numpy(ids).cuda(), to_dev(table, dtype), pe, pos_offset=off)
    assert mha.mha_check() == mha.MHA_OK
    ref = oracle.embed_pe(ids, table, pos_offset=off)
    err = check_x(to_np(x), ref, dtype)
    print(f"\nembed_pe {st} B{B} L{L} D{D}: max|err| {err:.3e}")


def test_embed_pe_bad_token_reports_device_error():
    D, vocab = 64, 10
    table = torch.ones((vocab, D), dtype=torch.bfloat16, device="cuda")
    pe = mha.sinusoidal_pe(4, D)
    ids = torch.tensor([[1, 10, 2, -1]], dtype=torch.int32, device="cuda")
    assert mha.mha_check() == mha.MHA_OK
    x = mha.embed_pe(ids, table, pe)
    assert mha.mha_check() == mha.MHA_ERR_DEVICE
    assert torch.all(x[0, 1] == 0) and torch.all(x[0, 3] == 0)
    assert torch.all(x[0, 0] != 0)
    assert mha.mha_check() == mha.MHA_OK
    with pytest.raises(mha.MhaError):          # the table is too short for the window
        mha.embed_pe(ids, table, pe, pos_offset=1)


def test_embed_pe_encoder_workload_shape():
    """The encoder workload's input at full size (B32 L512, d_model 512, the
    pages' 37000-token vocabulary), every output element."""
    B, L, D, vocab = 32, 512, 512, 37000
    g = Draws(1200)
    table = g.normal((vocab, D), std=1.0 / np.sqrt(D))
    ids = g.integers(0, vocab - 1, (B, L))
    pe = mha.sinusoidal_pe(L, D)
    x = mha.embed_pe(torch.from_numpy(ids).cuda(), to_dev(table, torch.bfloat16), pe)
    assert mha.mha_check() == mha.MHA_OK
    err = check_x(to_np(x), oracle.embed_pe(ids, table), torch.bfloat16)
    print(f"\nembed_pe encoder shape: max|err| {err:.3e}")


def test_embedding_then_encoder_layer():
    """Tokens -> embed_pe -> encoder_forward against the oracle's embed_pe ->
    encoder_layer.  The library stores x once in the layer's type (bf16), so
    the oracle's layer reads its own fp64 x rounded to bf16 the same way
    (round to nearest even); the encoder's bars apply: the fp32 output
    within 2e-2, the bf16 output within that plus its half-ulp."""
    from tests.test_encoder_gpu import BF16_MAX, BF16_RMS, make_params
    from tests.gpu_util import errors
    from transformer_head_scaled_03_gb300.inputs import round_to_bf16
    B, L, D, h, F, vocab = 2, 96, 256, 4, 1024, 300
    g = Draws(1300)
    table = g.normal((vocab, D), std=1.0 / np.sqrt(D))
    ids = g.integers(0, vocab - 1, (B, L))
    p = make_params(g, D, F, "bf16")
    pe = mha.sinusoidal_pe(L, D)
    x = mha.embed_pe(torch.from_numpy(ids).cuda(), to_dev(table, torch.bfloat16), pe)
    layer = mha.EncoderLayer(D, h, F, torch.bfloat16, B, L)
    try:
        dp = {k: to_dev(v, torch.bfloat16) for k, v in p.items()}
        out = layer.forward(x, dp)
        out32 = layer.forward(x, dp, out_dtype=torch.float32)
        assert mha.mha_check() == mha.MHA_OK
        got, got32 = to_np(out), to_np(out32)
    finally:
        layer.close()
    x_ref = round_to_bf16(oracle.embed_pe(ids, table).astype(np.float32))
    ref = oracle.encoder_layer(x_ref, p, h)
    max32, rms32 = errors(got32, ref)
    assert max32 <= BF16_MAX and rms32 <= BF16_RMS, (max32, rms32)
    max_abs, rms = errors(got, ref)
    bound = BF16_MAX + 2.0 ** -8 * float(np.max(np.abs(ref)))
    assert max_abs <= bound and rms <= BF16_RMS, (max_abs, bound, rms)
    print(f"\ntokens -> encoder layer: fp32 out max|err| {max32:.3e}; bf16 out max|err| "
          f"{max_abs:.3e} (bound {bound:.3e}) rms rel {rms:.3e}")
