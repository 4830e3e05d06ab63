"""Failure detection without faulting the GPU: a pipeline wait that nothing
completes gives up after its limit, the device error word reports
MHA_ERR_TIMEOUT to the host, and the context keeps working."""
import time

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


def test_wait_that_never_completes_reports_timeout_and_context_survives():
    assert mha.mha_check() == mha.MHA_OK
    t0 = time.perf_counter()
    mha.selftest_wait_timeout(200)
    status = mha.mha_check()
    elapsed = time.perf_counter() - t0
    assert status == mha.MHA_ERR_TIMEOUT
    assert 0.15 <= elapsed < 5.0          # gave up after about the limit
    assert mha.mha_check() == mha.MHA_OK  # the word was cleared
    # the context is still usable: a normal call after the timeout is correct
    g = Draws(77)
    Q, K, V = (g.normal((1, 2, 200, 64)) for _ in range(3))
    O = mha.sdpa_forward(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                         to_dev(V, torch.bfloat16), mask_kind=mha.MASK_CAUSAL)
    assert mha.mha_check() == mha.MHA_OK
    assert_parity(to_np(O), oracle.sdpa(Q, K, V, mask_kind=oracle.MASK_CAUSAL),
                  torch.bfloat16, "after timeout")


def test_selftest_rejects_bad_limit():
    with pytest.raises(mha.MhaError):
        mha.selftest_wait_timeout(0)
