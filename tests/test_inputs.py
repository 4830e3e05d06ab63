"""The seeded input recipe (CPU): the workloads' shapes, distributions and
structure as stated for them -- bf16-representable values, key lengths drawn
inclusively from their range, the long-context outlier dimensions shared by
Q and K and scaled by exactly 8, and weights with variance 1/D -- and that
the draws are deterministic per seed."""
import numpy as np

from transformer_head_scaled_03_gb300.inputs import (WORKLOADS, Draws, mha_inputs,
                                                     round_to_bf16, sdpa_inputs)


def _is_bf16(a):
    return np.array_equal(a.view(np.uint32) & np.uint32(0xFFFF), np.zeros(a.shape, np.uint32))


def test_round_to_bf16_ties_to_even_and_idempotent():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: ties go to even (1)
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 0.0], dtype=np.float32)
    r = round_to_bf16(x)
    assert r[0] == np.float32(1.0) and r[1] == np.float32(1.0 + 2.0 ** -6) and r[2] == -2.5
    assert np.array_equal(round_to_bf16(r), r) and _is_bf16(r)


def test_draws_are_deterministic_per_seed():
    a = Draws(7).normal((3, 5))
    b = Draws(7).normal((3, 5))
    c = Draws(8).normal((3, 5))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_key_padding_lengths_inclusive_range():
    w = WORKLOADS[2]
    Q, K, V, lens, dims = sdpa_inputs(w, B=4096, H=1, Lq=1, Lk=512, d=8)
    assert lens.dtype == np.int32 and lens.shape == (4096,)
    assert lens.min() == 256 and lens.max() == 512   # both ends reachable
    assert dims is None and _is_bf16(Q) and _is_bf16(K) and _is_bf16(V)


def test_long_context_outliers_shared_by_q_and_k():
    w = WORKLOADS[5]
    Q, K, V, lens, dims = sdpa_inputs(w, B=1, H=4, Lq=4096, Lk=4096, d=128)
    assert lens is None and dims.shape == (4, 4)
    assert all(len(set(dims[h])) == 4 for h in range(4))
    base_q, base_k, _, _, _ = sdpa_inputs(
        WORKLOADS[3], seed=w.seed, B=1, H=4, Lq=4096, Lk=4096, d=128)
    for h in range(4):
        other = np.setdiff1d(np.arange(128), dims[h])
        # the chosen dims of Q and K are the plain draws times 8 (exact in bf16)
        assert np.array_equal(Q[0, h][:, dims[h]], base_q[0, h][:, dims[h]] * 8)
        assert np.array_equal(K[0, h][:, dims[h]], base_k[0, h][:, dims[h]] * 8)
        assert np.array_equal(Q[0, h][:, other], base_q[0, h][:, other])
        assert np.array_equal(V[0, h], sdpa_inputs(WORKLOADS[3], seed=w.seed, B=1, H=4, Lq=4096,
                                                   Lk=4096, d=128)[2][0, h])
    # scaled-score spread: sqrt((124 + 4 * 64^2) / 128) ~ 11.4 (the literal x8 reading)
    s = np.einsum("qd,kd->qk", Q[0, 0, :256].astype(np.float64),
                  K[0, 0, :256].astype(np.float64)) / np.sqrt(128.0)
    assert abs(s.std() - np.sqrt((124 + 4 * 64 ** 2) / 128)) < 1.5


def test_base_shape_weights_have_variance_one_over_d():
    w = WORKLOADS[1]
    x, *Ws = mha_inputs(w)
    assert x.shape == (1, 128, 512) and all(W.shape == (512, 512) for W in Ws)
    for W in Ws:
        assert abs(W.var() * 512 - 1.0) < 0.02
    assert abs(x.std() - 1.0) < 0.02
