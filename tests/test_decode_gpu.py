"""sdpa_decode (a few new queries against a key/value cache, bottom-right
causal, keys split across a thread-block cluster and merged through
distributed shared memory) on the GPU against the fp64 oracle.

Tolerance: the bf16 bar (max|err| <= 2e-2, RMS rel <= 1e-2) for both output
types -- the inputs are bf16 and the weights are rounded to bf16 before the
P V product, as in sdpa_forward."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build
from transformer_head_scaled_03_gb300.inputs import WORKLOADS, Draws, sdpa_inputs
from tests.gpu_util import assert_parity, to_dev, to_np

pytestmark = pytest.mark.gpu

BR, PAD = oracle.MASK_CAUSAL_BOTTOM_RIGHT, oracle.MASK_KEY_PADDING


@pytest.fixture(scope="module", autouse=True)
def built():
    mha_build.build()
    mha.lib()


def run_decode(seed, d, B, H, Lq, Lk, lengths, causal, splits, out_dtype, q_scale=1.0):
    g = Draws(seed)
    Q = g.normal((B, H, Lq, d)) * np.float32(q_scale)
    K = g.normal((B, H, Lk, d))
    V = g.normal((B, H, Lk, d))
    lens = None if lengths is None else np.asarray(lengths, np.int32)
    kl = None if lens is None else torch.from_numpy(lens).cuda()
    O = mha.sdpa_decode(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                        to_dev(V, torch.bfloat16), kv_lengths=kl, causal=causal,
                        out_dtype=out_dtype, num_splits=splits)
    assert mha.mha_check() == mha.MHA_OK
    mk = (BR if causal else 0) | (PAD if lens is not None else 0)
    ref = oracle.sdpa(Q, K, V, mask_kind=mk, key_lengths=lens)
    return to_np(O), ref


BF, F32 = torch.bfloat16, torch.float32
CASES = [
    # d, B, H, Lq, Lk, lengths, causal, splits, out dtype
    (128, 2, 3, 1, 1000, [1000, 517], True, 0, BF),
    (128, 2, 2, 16, 777, [16, 777], True, 3, F32),        # len = Lq, the minimum
    (64, 3, 4, 5, 2048, [129, 128, 2048], True, 16, BF),  # tile edges, 16-CTA cluster
    (64, 1, 2, 16, 300, None, True, 1, F32),               # no padding: len = Lk
    (128, 2, 2, 7, 4096, [4000, 1], False, 8, BF),         # cross-attention, one key
    (64, 4, 2, 3, 130, [3, 130, 64, 127], True, 2, F32),
    (128, 1, 1, 2, 200, [150], True, 16, F32),             # more splits than tiles
    (64, 2, 8, 1, 8192, [8192, 5000], True, 0, BF),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_decode_parity(case):
    d, B, H, Lq, Lk, lengths, causal, splits, odt = case
    got, ref = run_decode(900 + CASES.index(case), d, B, H, Lq, Lk, lengths, causal, splits, odt)
    max_abs, rms = assert_parity(got, ref, torch.bfloat16, str(case))
    print(f"\ndecode {case}: max|err| {max_abs:.3e} rms rel {rms:.3e}")


def test_decode_sharp_scores_every_split_count():
    """Peaked rows (queries x4: scaled-score std ~ 4) with the maximum in a
    different split per head: the exact merge must reproduce the single
    softmax for every split count."""
    for splits in (1, 2, 5, 8, 16):
        got, ref = run_decode(950, 128, 1, 4, 4, 3000, [2900], True, splits, F32, q_scale=4.0)
        assert_parity(got, ref, torch.bfloat16, f"splits {splits}")


def test_decode_bad_lengths_report_device_error():
    g = Draws(960)
    B, H, Lq, Lk, d = 3, 2, 4, 256, 64
    Q, K, V = (to_dev(g.normal(s), torch.bfloat16) for s in
               ((B, H, Lq, d), (B, H, Lk, d), (B, H, Lk, d)))
    assert mha.mha_check() == mha.MHA_OK
    for bad in ([0, 10, 10], [10, Lk + 1, 10], [10, 10, Lq - 1]):
        kl = torch.tensor(bad, dtype=torch.int32, device="cuda")
        O = mha.sdpa_decode(Q, K, V, kv_lengths=kl, causal=True, out_dtype=torch.float32)
        assert mha.mha_check() == mha.MHA_ERR_DEVICE
        i = next(k for k, v in enumerate(bad) if v < Lq or v > Lk)
        assert torch.all(O[i] == 0)
    assert mha.mha_check() == mha.MHA_OK


def test_decode_rejects_bad_arguments():
    lib = mha.lib()
    g = Draws(961)
    Q = to_dev(g.normal((1, 1, 17, 64)), torch.bfloat16)
    K = to_dev(g.normal((1, 1, 64, 64)), torch.bfloat16)
    with pytest.raises(mha.MhaError):          # Lq > 16
        mha.sdpa_decode(Q, K, K)
    Q = to_dev(g.normal((1, 1, 2, 96)), torch.bfloat16)
    K = to_dev(g.normal((1, 1, 64, 96)), torch.bfloat16)
    with pytest.raises(mha.MhaError):          # d = 96
        mha.sdpa_decode(Q, K, K)
    Q = to_dev(g.normal((1, 1, 2, 64)), torch.bfloat16)
    K = to_dev(g.normal((1, 1, 64, 64)), torch.bfloat16)
    O = torch.empty_like(Q)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    call = lambda mask, lens, splits=0: lib.sdpa_decode(p(Q), p(K), p(K), p(O), 1, 1, 2, 64, 64,
                                                        0.0, mask, lens, mha.MHA_BF16, splits,
                                                        None)
    assert call(mha.MASK_CAUSAL, None) == mha.MHA_ERR_INVALID_ARG        # top-left causal
    assert call(mha.MASK_KEY_PADDING, None) == mha.MHA_ERR_INVALID_ARG   # lengths missing
    assert call(0, None, splits=17) == mha.MHA_ERR_INVALID_ARG
    assert call(mha.MASK_CAUSAL_BOTTOM_RIGHT, None) == mha.MHA_OK
    assert mha.mha_check() == mha.MHA_OK
    assert 1 <= mha.decode_splits(8, 32, 32768, 128) <= 16


@pytest.mark.parametrize("wid", [6, 7, 8])
def test_decode_workload_sampled_heads(wid):
    """The decode workloads at full size, called as the benchmark calls them
    (default split count), against the oracle on every query row of a
    seeded sample of (b, h) pairs."""
    w = WORKLOADS[wid]
    Q, K, V, lens, _ = sdpa_inputs(w)
    kl = torch.from_numpy(lens).cuda()
    O = mha.sdpa_decode(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                        to_dev(V, torch.bfloat16), kv_lengths=kl, causal=True)
    assert mha.mha_check() == mha.MHA_OK
    g = Draws(w.seed + 4000)
    bhs = g.choice(w.B * w.H, min(24, w.B * w.H))
    # the sampled heads as a batch of single-head items (lengths follow b)
    pick = lambda a, L: a.reshape(w.B * w.H, L, w.d)[bhs][:, None]
    ref = oracle.sdpa(pick(Q, w.Lq), pick(K, w.Lk), pick(V, w.Lk), mask_kind=w.mask,
                      key_lengths=lens[bhs // w.H])
    got = to_np(O.reshape(w.B * w.H, w.Lq, w.d)[torch.from_numpy(bhs).cuda()])[:, None]
    max_abs, rms = assert_parity(got, ref, torch.bfloat16, w.name)
    print(f"\n{w.name}: {bhs.size} heads x {w.Lq} rows, max|err| {max_abs:.3e}, "
          f"rms rel {rms:.3e}")
