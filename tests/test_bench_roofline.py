"""Host-side roofline bookkeeping of bench.py (CPU): the algorithmic bytes of
each attention workload and the choice of bound against the measured peaks."""
import numpy as np
import pytest

import bench
from transformer_head_scaled_03_gb300.inputs import WORKLOADS, sdpa_inputs

PEAK_TF, PEAK_GBS = 1918.6, 6673.2   # the measured bf16 burst and HBM copy rates


def test_algorithmic_bytes_by_hand():
    # causal and no-mask workloads read Q, K, V and write O once (bf16)
    for wid in (3, 4, 5):
        w = WORKLOADS[wid]
        expect = 2 * w.H * w.d * (2 * w.B * w.Lq + 2 * w.B * w.Lk)
        assert w.sdpa_bytes() == expect
    # key padding reads only the rows below each item's length
    w = WORKLOADS[2]
    lens = np.array([256, 512] * (w.B // 2), dtype=np.int32)
    assert w.sdpa_bytes(lens) == 2 * w.H * w.d * (2 * w.B * w.Lq + 2 * int(lens.sum()))


@pytest.mark.parametrize("wid,bound", [(2, "hbm"), (3, "tensor"), (4, "hbm"), (5, "tensor")])
def test_bound_of_each_workload(wid, bound):
    w = WORKLOADS[wid]
    lens = sdpa_inputs(w)[3] if w.mask & 2 else None
    flops, nbytes = w.flops(lens), w.sdpa_bytes(lens)
    r = bench.attention_roofline(flops, nbytes, 500.0, PEAK_TF, PEAK_GBS, "measured")
    assert r["bound"] == bound


def test_hbm_bound_reports_the_same_time_in_bytes():
    # 1 GFLOP over 10 MB at 100 TFLOP/s: 10 us, i.e. 1000 GB/s
    r = bench.attention_roofline(1e9, 1e7, 100.0, PEAK_TF, PEAK_GBS, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(1000.0)
    assert r["frac"] == pytest.approx(1000.0 / PEAK_GBS, abs=1e-4)
    r = bench.attention_roofline(1e12, 1e7, 100.0, PEAK_TF, PEAK_GBS, "measured")
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(100.0 / PEAK_TF, abs=1e-4)


def test_nominal_fraction_beside_the_measured_one():
    r = bench.attention_roofline(1e9, 1e7, 100.0, PEAK_TF, PEAK_GBS, "measured")
    assert r["frac_nominal"] == pytest.approx(1000.0 / bench.NOMINAL_HBM_GBS, abs=1e-4)
    r = bench.attention_roofline(1e12, 1e7, 100.0, PEAK_TF, PEAK_GBS, "measured")
    assert r["frac_nominal"] == pytest.approx(100.0 / bench.NOMINAL_BF16_TFLOPS, abs=1e-4)


@pytest.mark.parametrize("wid", [2, 3, 4, 5])
def test_one_oracle_sample_per_workload(wid):
    """The CPU-baseline leg and the reference arm time the same rows."""
    w = WORKLOADS[wid]
    a, na = bench.oracle_sample(w)
    b, nb = bench.oracle_sample(w)
    assert na == nb and np.array_equal(a, b)
    assert a.size == w.B * w.H * na
    assert np.all((a >= 0) & (a < w.B * w.H * w.Lq))


def test_config_names_the_mask_and_l2_treatment():
    lens = sdpa_inputs(WORKLOADS[2])[3]
    c = bench.sdpa_config(WORKLOADS[2], lens, 1)
    assert c["mask"] == "key_padding" and c["l2"] == "L2 flushed between steps"
    c = bench.sdpa_config(WORKLOADS[5], None, 1)
    assert c["mask"] == "causal" and c["l2"] == "inputs larger than L2"
    assert bench.sdpa_config(WORKLOADS[4], None, 1)["l2"] == "L2 flushed between steps"
    assert bench.sdpa_config(WORKLOADS[3], None, 1)["l2"] == "L2 flushed between steps"
