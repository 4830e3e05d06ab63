"""Shared helpers of the GPU parity tests."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances of the parity bar.
#   fp32 inputs: max |err| <= 1e-4
#   bf16 inputs, fp32 accumulation: max |err| <= 2e-2 and RMS relative error
#   sqrt(sum (o - o_ref)^2 / sum o_ref^2) <= 1e-2
F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_RMS_REL = 1e-2


def to_dev(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    """float32 array of storage-type values -> device tensor (exact)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dtype).cuda()


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0, 0.0
    assert np.all(np.isfinite(got)), "non-finite output"
    diff = got - ref
    max_abs = float(np.max(np.abs(diff)))
    denom = float(np.sum(ref * ref))
    rms_rel = float(np.sqrt(np.sum(diff * diff) / denom)) if denom > 0 else float(np.sqrt(np.sum(diff * diff)))
    return max_abs, rms_rel


def assert_parity(got, ref, dtype: torch.dtype, what: str = ""):
    max_abs, rms_rel = errors(got, ref)
    if dtype == torch.bfloat16:
        assert max_abs <= BF16_MAX_ABS and rms_rel <= BF16_RMS_REL, \
            f"{what}: max|err| {max_abs:.3e} (<= {BF16_MAX_ABS}), rms rel {rms_rel:.3e} (<= {BF16_RMS_REL})"
    else:
        assert max_abs <= F32_MAX_ABS, f"{what}: max|err| {max_abs:.3e} (<= {F32_MAX_ABS})"
    return max_abs, rms_rel
