"""The four attention workloads at full size, called exactly as bench.py
calls them, against the fp64 oracle: every output of the key-padding
encoder, decoder causal and cross-attention workloads, and seeded row
samples (plus fixed tile-edge rows) of the long-context workload, whose
8.8 TFLOP the oracle cannot finish in seconds."""
import numpy as np
import pytest
import torch

import oracle
import transformer_head_scaled_03_gb300 as mha
from transformer_head_scaled_03_gb300 import build as mha_build
from transformer_head_scaled_03_gb300.inputs import WORKLOADS, sample_rows, sdpa_inputs
from tests.gpu_util import assert_parity, errors, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    mha_build.build()
    mha.lib()


def gpu_run(w, Q, K, V, lens, out_dtype=torch.bfloat16):
    kl = torch.from_numpy(lens).cuda() if lens is not None else None
    O = mha.sdpa_forward(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                         to_dev(V, torch.bfloat16), mask_kind=w.mask, key_lengths=kl,
                         out_dtype=out_dtype)
    assert mha.mha_check() == mha.MHA_OK
    return O


@pytest.mark.parametrize("wid", [2, 3, 4])
def test_workload_full_output(wid):
    """Every output element of the workload (B32 L512 key padding: 16.8 M
    values; B16 L2048 causal: 33.6 M; B64 Lq256 Lk1024: 8.4 M)."""
    w = WORKLOADS[wid]
    Q, K, V, lens, _ = sdpa_inputs(w)
    if lens is not None:
        assert lens.min() >= 256 and lens.max() <= 512
    got = to_np(gpu_run(w, Q, K, V, lens))
    ref = oracle.sdpa(Q, K, V, mask_kind=w.mask, key_lengths=lens)
    assert oracle.default().last_bad_rows == 0
    max_abs, rms = assert_parity(got, ref, torch.bfloat16, w.name)
    print(f"\n{w.name}: all {got.size} outputs, max|err| {max_abs:.3e}, rms rel {rms:.3e}")


def test_long_context_sampled_rows():
    w = WORKLOADS[5]
    Q, K, V, lens, dims = sdpa_inputs(w)
    rows = sample_rows(w.B, w.H, w.Lq, 64, seed=w.seed + 1000)
    O = gpu_run(w, Q, K, V, lens)
    got = to_np(O.reshape(-1, w.d)[torch.from_numpy(rows).cuda()])
    ref = oracle.sdpa_rows(Q, K, V, rows, mask_kind=w.mask, key_lengths=lens)
    max_abs, rms = assert_parity(got, ref, torch.bfloat16, w.name)
    print(f"\n{w.name}: {rows.size} rows, max|err| {max_abs:.3e}, rms rel {rms:.3e}")


def test_long_context_fp32_output_sampled_rows():
    """Same workload with the output kept in fp32: isolates kernel error from
    the final bf16 rounding of the output."""
    w = WORKLOADS[5]
    Q, K, V, lens, dims = sdpa_inputs(w)
    rows = sample_rows(w.B, w.H, w.Lq, 16, seed=w.seed + 2000)
    O = gpu_run(w, Q, K, V, lens, out_dtype=torch.float32)
    got = to_np(O.reshape(-1, w.d)[torch.from_numpy(rows).cuda()])
    ref = oracle.sdpa_rows(Q, K, V, rows, mask_kind=w.mask, key_lengths=lens)
    max_abs, rms = assert_parity(got, ref, torch.bfloat16, w.name + " fp32 out")
    print(f"\n{w.name} fp32 out: max|err| {max_abs:.3e}, rms rel {rms:.3e}")
