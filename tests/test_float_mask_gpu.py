"""sdpa_forward_float_mask: an additive float mask [.., Lq, Lk] added to the
scaled scores, against the fp64 oracle; the causal mask in float form must
give exactly what mask_kind = causal gives."""
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


def random_mask(g, shape, frac_blocked=0.3):
    m = g.normal(shape, std=3.0, dtype="f32")
    blocked = g.rng.random(shape) < frac_blocked
    m[blocked] = -np.inf
    m[..., 0] = 0.0   # key 0 stays visible in every row
    return m.astype(np.float32)


CASES = [
    # dtype, B, H, Lq, Lk, d, mask shape kind, mask_kind, lengths
    (torch.bfloat16, 2, 2, 200, 300, 64, "head", mha.MASK_NONE, None),
    (torch.bfloat16, 1, 3, 257, 257, 128, "bcast", mha.MASK_NONE, None),
    (torch.bfloat16, 3, 2, 130, 256, 64, "batch", mha.MASK_KEY_PADDING, [256, 100, 1]),
    (torch.bfloat16, 1, 2, 384, 384, 128, "head", mha.MASK_CAUSAL, None),
    (torch.bfloat16, 2, 1, 64, 130, 64, "bcast", mha.MASK_NONE, None),     # Lk % 4 != 0
    (torch.float32, 2, 2, 70, 90, 64, "head", mha.MASK_NONE, None),
    (torch.float32, 1, 2, 33, 33, 128, "bcast", mha.MASK_CAUSAL, None),
]
SHAPES = {"head": lambda B, H, Lq, Lk: (B, H, Lq, Lk), "bcast": lambda B, H, Lq, Lk: (Lq, Lk),
          "batch": lambda B, H, Lq, Lk: (B, 1, Lq, Lk)}


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_float_mask_parity(case):
    dtype, B, H, Lq, Lk, d, kind, mk, lengths = case
    g = Draws(600 + CASES.index(case))
    st = "bf16" if dtype == torch.bfloat16 else "f32"
    Q, K, V = (g.normal(s, dtype=st) for s in ((B, H, Lq, d), (B, H, Lk, d), (B, H, Lk, d)))
    m = random_mask(g, SHAPES[kind](B, H, Lq, Lk))
    lens = np.asarray(lengths, np.int32) if lengths else None
    kl = torch.from_numpy(lens).cuda() if lens is not None else None
    O = mha.sdpa_forward(to_dev(Q, dtype), to_dev(K, dtype), to_dev(V, dtype), mask_kind=mk,
                         key_lengths=kl, add_mask=torch.from_numpy(m).cuda())
    assert mha.mha_check() == mha.MHA_OK
    ref = oracle.sdpa(Q, K, V, mask_kind=mk, key_lengths=lens, add_mask=m)
    assert_parity(to_np(O), ref, dtype, str(case))


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 64), (torch.bfloat16, 128),
                                     (torch.float32, 64)])
def test_causal_float_mask_equals_causal_kind_bitwise(dtype, d):
    g = Draws(650 + d)
    st = "bf16" if dtype == torch.bfloat16 else "f32"
    L = 300
    Q, K, V = (g.normal((2, 2, L, d), dtype=st) for _ in range(3))
    causal = np.triu(np.full((L, L), -np.inf, np.float32), 1)
    a = mha.sdpa_forward(to_dev(Q, dtype), to_dev(K, dtype), to_dev(V, dtype),
                         add_mask=torch.from_numpy(causal).cuda())
    b = mha.sdpa_forward(to_dev(Q, dtype), to_dev(K, dtype), to_dev(V, dtype),
                         mask_kind=mha.MASK_CAUSAL)
    assert torch.equal(a, b)


def test_fully_blocked_row_is_zero():
    g = Draws(660)
    Q, K, V = (g.normal((1, 1, 8, 64)) for _ in range(3))
    m = np.zeros((8, 8), np.float32)
    m[3, :] = -np.inf
    O = to_np(mha.sdpa_forward(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                               to_dev(V, torch.bfloat16), add_mask=torch.from_numpy(m).cuda()))
    assert np.all(O[0, 0, 3] == 0.0) and np.all(np.isfinite(O))
    ref = oracle.sdpa(Q, K, V, add_mask=m)
    rows = [0, 1, 2, 4, 5, 6, 7]
    assert_parity(O[:, :, rows], ref[:, :, rows], torch.bfloat16, "other rows")
