"""sdpa_forward on the GPU against the fp64 oracle, element by element, on
seeded inputs that span several 128-row/128-key tiles and ragged tails, plus
the invariants that must hold exactly on the device."""
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


@pytest.fixture(scope="module", autouse=True)
def built():
    mha_build.build()
    mha.lib()


def make(seed, B, H, Lq, Lk, d, dtype, mask, lengths=None):
    g = Draws(seed)
    st = "bf16" if dtype == torch.bfloat16 else "f32"
    Q = g.normal((B, H, Lq, d), dtype=st)
    K = g.normal((B, H, Lk, d), dtype=st)
    V = g.normal((B, H, Lk, d), dtype=st)
    if mask & PAD and lengths is None:
        lengths = g.integers(1, Lk, B)
    lens = None if lengths is None else np.asarray(lengths, dtype=np.int32)
    return Q, K, V, lens


def run_case(seed, B, H, Lq, Lk, d, dtype, mask, lengths=None, out_dtype=None, scale=0.0):
    Q, K, V, lens = make(seed, B, H, Lq, Lk, d, dtype, mask, lengths)
    kl = torch.from_numpy(lens).cuda() if lens is not None else None
    O = mha.sdpa_forward(to_dev(Q, dtype), to_dev(K, dtype), to_dev(V, dtype), scale=scale,
                         mask_kind=mask, key_lengths=kl, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert mha.mha_check() == mha.MHA_OK
    ref = oracle.sdpa(Q, K, V, scale=scale, mask_kind=mask, key_lengths=lens)
    return to_np(O), ref


BF16_CASES = [
    # B, H, Lq, Lk, d, mask, lengths
    (1, 1, 1, 1, 64, NONE, None),
    (1, 2, 3, 5, 64, NONE, None),
    (2, 2, 128, 128, 64, NONE, None),
    (1, 3, 129, 300, 64, NONE, None),
    (2, 2, 200, 700, 128, NONE, None),
    (1, 2, 4, 1000, 128, NONE, None),
    (1, 1, 1, 1, 128, CAUSAL, None),
    (1, 2, 2, 2, 64, CAUSAL, None),
    (1, 2, 127, 127, 128, CAUSAL, None),
    (1, 1, 129, 129, 128, CAUSAL, None),
    (2, 2, 257, 257, 64, CAUSAL, None),
    (1, 2, 1000, 1000, 64, CAUSAL, None),
    (1, 1, 640, 640, 128, CAUSAL, None),
    (4, 2, 300, 300, 64, PAD, [1, 127, 128, 129]),
    (3, 2, 130, 256, 128, PAD, [256, 255, 1]),
    (3, 2, 256, 256, 64, PAD | CAUSAL, [1, 200, 256]),
    (2, 1, 384, 384, 128, PAD | CAUSAL, [383, 129]),
    # each query tile of a two-tile CTA stops at its own diagonal (or at the
    # key length, when that comes first)
    (1, 2, 450, 450, 64, CAUSAL, None),
    (2, 1, 450, 450, 128, CAUSAL, None),
    (2, 3, 260, 260, 64, PAD | CAUSAL, [190, 65]),
    (2, 2, 520, 520, 128, PAD | CAUSAL, [300, 520]),
]


@pytest.mark.parametrize("case", BF16_CASES, ids=[str(c[:6]) for c in BF16_CASES])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["obf16", "of32"])
def test_bf16_parity(case, out_dtype):
    B, H, Lq, Lk, d, mask, lengths = case
    got, ref = run_case(101 + BF16_CASES.index(case), B, H, Lq, Lk, d, torch.bfloat16, mask,
                        lengths, out_dtype=out_dtype)
    assert_parity(got, ref, torch.bfloat16, f"{case} {out_dtype}")


def test_bf16_explicit_scale():
    got, ref = run_case(7, 2, 2, 300, 300, 64, torch.bfloat16, CAUSAL, scale=0.05)
    assert_parity(got, ref, torch.bfloat16, "scale 0.05")


F32_CASES = [
    (1, 1, 1, 1, 17, NONE, None),
    (2, 3, 33, 70, 64, NONE, None),
    (1, 2, 100, 100, 100, CAUSAL, None),
    (2, 2, 65, 65, 128, CAUSAL, None),
    (3, 2, 40, 97, 64, PAD, [1, 32, 97]),
    (2, 1, 50, 50, 8, PAD | CAUSAL, [3, 50]),
]


@pytest.mark.parametrize("case", F32_CASES, ids=[str(c[:6]) for c in F32_CASES])
def test_f32_parity(case):
    B, H, Lq, Lk, d, mask, lengths = case
    got, ref = run_case(201 + F32_CASES.index(case), B, H, Lq, Lk, d, torch.float32, mask,
                        lengths)
    assert_parity(got, ref, torch.float32, str(case))


# ------------------------------------------------------------------ invariants

@pytest.mark.parametrize("d", [64, 128])
def test_causal_rows_ignore_future_keys_bitwise(d):
    B, H, L = 1, 2, 384
    Q, K, V, _ = make(31, B, H, L, L, d, torch.bfloat16, CAUSAL)
    base = to_np(mha.sdpa_forward(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                                  to_dev(V, torch.bfloat16), mask_kind=CAUSAL))
    g = Draws(32)
    for i in (0, 127, 128, 200, 383):
        K2, V2 = K.copy(), V.copy()
        K2[:, :, i + 1:] = g.normal(K2[:, :, i + 1:].shape) * 4
        V2[:, :, i + 1:] = g.normal(V2[:, :, i + 1:].shape) * 4
        got = to_np(mha.sdpa_forward(to_dev(Q, torch.bfloat16), to_dev(K2, torch.bfloat16),
                                     to_dev(V2, torch.bfloat16), mask_kind=CAUSAL))
        assert np.array_equal(got[:, :, : i + 1], base[:, :, : i + 1]), f"row <= {i} changed"


@pytest.mark.parametrize("d", [64, 128])
def test_single_visible_key_returns_value_row_exactly(d):
    B, H, Lq, Lk = 2, 2, 200, 300
    Q, K, V, _ = make(41, B, H, Lq, Lk, d, torch.bfloat16, PAD)
    kl = torch.ones(B, dtype=torch.int32, device="cuda")
    O = to_np(mha.sdpa_forward(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                               to_dev(V, torch.bfloat16), mask_kind=PAD, key_lengths=kl))
    assert np.array_equal(O, np.broadcast_to(V[:, :, :1].astype(np.float64), O.shape))
    # causal row 0 sees only key 0
    Q, K, V, _ = make(42, B, H, Lq, Lq, d, torch.bfloat16, CAUSAL)
    O = to_np(mha.sdpa_forward(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                               to_dev(V, torch.bfloat16), mask_kind=CAUSAL))
    assert np.array_equal(O[:, :, 0], V[:, :, 0].astype(np.float64))


def test_zero_query_gives_mean_of_visible_values():
    B, H, L, d = 1, 2, 300, 64
    _, K, V, _ = make(51, B, H, L, L, d, torch.bfloat16, NONE)
    Q = np.zeros((B, H, L, d), np.float32)
    O = to_np(mha.sdpa_forward(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                               to_dev(V, torch.bfloat16), mask_kind=CAUSAL,
                               out_dtype=torch.float32))
    prefix = np.cumsum(V.astype(np.float64), axis=2) / np.arange(1, L + 1)[None, None, :, None]
    assert np.max(np.abs(O - prefix)) <= 2e-2


def test_key_length_outside_range_reports_device_error():
    B, H, L, d = 2, 1, 64, 64
    Q, K, V, _ = make(61, B, H, L, L, d, torch.bfloat16, NONE)
    kl = torch.tensor([0, L + 1], dtype=torch.int32, device="cuda")
    O = mha.sdpa_forward(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                         to_dev(V, torch.bfloat16), mask_kind=PAD, key_lengths=kl)
    assert mha.mha_check() == mha.MHA_ERR_DEVICE
    assert torch.count_nonzero(O).item() == 0     # affected rows are zeros, no NaN
    assert mha.mha_check() == mha.MHA_OK          # the word was cleared


def test_empty_batch_is_a_no_op():
    Q = torch.empty((0, 2, 5, 64), dtype=torch.bfloat16, device="cuda")
    O = mha.sdpa_forward(Q, Q, Q)
    assert O.shape == (0, 2, 5, 64)


# Shapes with many more (b, h, query block) CTAs than SMs and short key
# ranges: several waves, with CTAs of different lengths sharing an SM.
# Causal runs mix block lengths; key padding gives items of different
# lengths, including single-key and full-length ones.
MULTI_ITEM_CASES = [
    # B, H, Lq, Lk, d, mask, lengths
    (40, 4, 700, 700, 64, CAUSAL, None),
    (40, 4, 700, 700, 128, CAUSAL, None),
    (24, 8, 300, 300, 64, PAD, None),
    (30, 6, 513, 513, 128, PAD | CAUSAL, None),
    (160, 1, 100, 1000, 64, NONE, None),       # one query tile per item
    (20, 10, 256, 129, 128, PAD, [1] * 10 + [129] * 10),
]


@pytest.mark.parametrize("case", MULTI_ITEM_CASES, ids=[str(c[:6]) for c in MULTI_ITEM_CASES])
def test_bf16_parity_several_items_per_cta(case):
    B, H, Lq, Lk, d, mask, lengths = case
    got, ref = run_case(500 + MULTI_ITEM_CASES.index(case), B, H, Lq, Lk, d, torch.bfloat16,
                        mask, lengths)
    max_abs, rms = assert_parity(got, ref, torch.bfloat16, str(case))
    print(f"\n{case[:6]}: max|err| {max_abs:.3e} rms rel {rms:.3e}")
