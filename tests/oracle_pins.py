"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics,
none of which re-types the oracle's own formula.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees.  ``tests/test_oracle_pins.py`` runs them on the oracle;
``tests/test_oracle_mutants.py`` runs them on deliberately broken copies of
the oracle and requires every copy to fail at least one pin.

Sources of the pinned facts:
  - rows of weights sum to 1, weights >= 0: "32 Transformer" (ml-canon-en),
    PyTorch snippet comment; "The Transformer" (hoshank.vercel.app), symbol
    table of the attention equation.
  - the printed 4x4 causal mask and "-inf gives weight exactly 0":
    "The Transformer" (rayaq.ca), "Masks: who may look at whom".
  - key padding masks keys per batch item: same section.
  - permutation: swapping two words swaps their outputs and nothing else:
    "The Transformer" (rayaq.ca), "Embeddings and positions".
  - score variance d_k before scaling and 1 after: "32 Transformer",
    "Why we divide by sqrt(dk)"; hoshank, "The Mathematics".
  - one-hot collapse of sharply peaked rows: rayaq.ca, "Worked example".
  - the multi-head assembly (projection x @ W, head i = column block i,
    concat, @ Wo): "32 Transformer", "PyTorch Implementation"; hoshank,
    multi-head equation.
  - library routines: torch's CPU float64 ``scaled_dot_product_attention``
    and ``multi_head_attention_forward`` (an independent implementation).
  - positional encoding: PE(0, 2i) = 0 and PE(0, 2i+1) = 1; each dimension
    pair is a point on the unit circle turning at its own frequency, the
    frequencies falling geometrically from 1 rad per position, so a shift of
    k positions is one fixed rotation per pair (the "signal for relative
    position"): "How Transformers Work" (worksonmygpu.com), "Positional
    encoding"; "The Transformer" (hoshank.vercel.app), "The Mathematics".
    The embedding lookup is cross-checked against torch's embedding.
  - backward pass: torch's float64 autograd of scaled_dot_product_attention
    (library routine); central finite differences of sum(dO * O); the
    softmax-gradient structure (each row of dS sums to zero, so the key
    gradients of a head sum to zero and the value gradients sum to the sum
    of dO); blocked keys get no gradient; a saturated row's gradient
    vanishes at its inactive positions ("32 Transformer" (ml-canon-en),
    "Why we divide by sqrt(dk)").
  - decoding: the decoder sees earlier positions only and generates left to
    right, so attending from the last Lq positions against the cached keys
    and values reproduces those rows of the full causal pass: "How
    Transformers Work" (worksonmygpu.com), "What changed since 2017"; "The
    Transformer" (hoshank.vercel.app), "The Breakthrough"; torch's
    ``causal_lower_right`` bias is the library cross-check.
"""
from __future__ import annotations

import math
import os

import numpy as np

from oracle import MASK_CAUSAL, MASK_CAUSAL_BOTTOM_RIGHT, MASK_KEY_PADDING, MASK_NONE

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _qkv(rng, B, H, Lq, Lk, d):
    return (rng.standard_normal((B, H, Lq, d)), rng.standard_normal((B, H, Lk, d)),
            rng.standard_normal((B, H, Lk, d)))


def _allclose(a, b, tol, what):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max|err| {err:.3e} > {tol:.1e}"


def read_mask_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "causal_mask_4x4.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([float(t) for t in line.split()])
    return np.array(rows)


# ---------------------------------------------------------------- SDPA pins

def pin_rows_sum_to_one(orc):
    rng = _rng(1)
    B, H, Lq, Lk, d = 2, 3, 5, 7, 8
    Q, K, V = _qkv(rng, B, H, Lq, Lk, d)
    lens = np.array([3, 7], dtype=np.int32)
    for mk in (MASK_NONE, MASK_KEY_PADDING):
        _, W = orc.sdpa(Q, K, V, mask_kind=mk, key_lengths=lens, return_weights=True)
        assert np.all(W >= 0.0), "negative weight"
        _allclose(W.sum(-1), np.ones((B, H, Lq)), 1e-12, "row sums")
    Q, K, V = _qkv(rng, B, H, 6, 6, d)
    _, W = orc.sdpa(Q, K, V, mask_kind=MASK_CAUSAL, return_weights=True)
    assert np.all(W >= 0.0)
    _allclose(W.sum(-1), np.ones((B, H, 6)), 1e-12, "causal row sums")


def pin_printed_causal_mask(orc):
    mask = read_mask_fixture()
    assert mask.shape == (4, 4)
    rng = _rng(2)
    for trial in range(5):
        Q, K, V = _qkv(rng, 1, 2, 4, 4, 16)
        _, W = orc.sdpa(Q * (1 + 3 * trial), K, V, mask_kind=MASK_CAUSAL,
                        return_weights=True)
        blocked = np.isneginf(mask)
        for h in range(2):
            assert np.all(W[0, h][blocked] == 0.0), "blocked key has nonzero weight"
            assert np.all(W[0, h][~blocked] > 0.0), "visible key has zero weight"


def pin_causal_future_independence(orc):
    rng = _rng(3)
    B, H, L, d = 2, 2, 9, 8
    Q, K, V = _qkv(rng, B, H, L, L, d)
    O = orc.sdpa(Q, K, V, mask_kind=MASK_CAUSAL)
    for i in (0, 3, 7):
        K2, V2 = K.copy(), V.copy()
        K2[:, :, i + 1:] = rng.standard_normal(K2[:, :, i + 1:].shape) * 5
        V2[:, :, i + 1:] = rng.standard_normal(V2[:, :, i + 1:].shape) * 5
        O2 = orc.sdpa(Q, K2, V2, mask_kind=MASK_CAUSAL)
        assert np.array_equal(O[:, :, : i + 1], O2[:, :, : i + 1]), \
            f"row <= {i} depends on a future key"
        if i + 1 < L:
            assert not np.array_equal(O[:, :, i + 1:], O2[:, :, i + 1:])


def pin_key_padding(orc):
    rng = _rng(4)
    B, H, Lq, Lk, d = 3, 2, 5, 8, 8
    Q, K, V = _qkv(rng, B, H, Lq, Lk, d)
    full = np.full(B, Lk, dtype=np.int32)
    assert np.array_equal(orc.sdpa(Q, K, V, mask_kind=MASK_KEY_PADDING, key_lengths=full),
                          orc.sdpa(Q, K, V)), "len = Lk differs from no mask"
    lens = np.array([2, 5, 8], dtype=np.int32)
    O = orc.sdpa(Q, K, V, mask_kind=MASK_KEY_PADDING, key_lengths=lens)
    K2, V2 = K.copy(), V.copy()
    for b, n in enumerate(lens):
        K2[b, :, n:] = 7.0
        V2[b, :, n:] = -9.0
    O2 = orc.sdpa(Q, K2, V2, mask_kind=MASK_KEY_PADDING, key_lengths=lens)
    assert np.array_equal(O, O2), "padded keys changed the output"
    # and a padded key does matter once it is inside the length
    O3 = orc.sdpa(Q, K2, V2, mask_kind=MASK_KEY_PADDING, key_lengths=lens + np.array([1, 1, 0], np.int32))
    assert not np.array_equal(O[:2], O3[:2])


def pin_single_visible_key(orc):
    """One visible key: the output is that key's value row, exactly."""
    rng = _rng(5)
    B, H, Lq, Lk, d = 2, 3, 4, 6, 8
    Q, K, V = _qkv(rng, B, H, Lq, Lk, d)
    O = orc.sdpa(Q, K, V, mask_kind=MASK_KEY_PADDING, key_lengths=np.array([1, 1], np.int32))
    for i in range(Lq):
        assert np.array_equal(O[:, :, i], V[:, :, 0]), "len 1 is not V row 0"
    Q, K, V = _qkv(rng, B, H, 5, 5, d)
    O = orc.sdpa(Q, K, V, mask_kind=MASK_CAUSAL)
    assert np.array_equal(O[:, :, 0], V[:, :, 0]), "causal row 0 is not V row 0"


def pin_zero_query_is_mean(orc):
    """q = 0: all scores equal, so the output is the mean of the visible values."""
    rng = _rng(6)
    B, H, L, d = 2, 2, 7, 8
    _, K, V = _qkv(rng, B, H, L, L, d)
    Q = np.zeros((B, H, L, d))
    O = orc.sdpa(Q, K, V)
    _allclose(O, np.broadcast_to(V.mean(axis=2, keepdims=True), O.shape), 1e-13, "uniform")
    O = orc.sdpa(Q, K, V, mask_kind=MASK_CAUSAL)
    prefix = np.cumsum(V, axis=2) / np.arange(1, L + 1)[None, None, :, None]
    _allclose(O, prefix, 1e-13, "causal uniform")
    lens = np.array([3, 6], np.int32)
    O = orc.sdpa(Q, K, V, mask_kind=MASK_KEY_PADDING, key_lengths=lens)
    for b, n in enumerate(lens):
        _allclose(O[b], np.broadcast_to(V[b, :, :n].mean(axis=1, keepdims=True), O[b].shape),
                  1e-13, "padding uniform")


def pin_two_keys_logistic(orc):
    """Two keys: the weights are (sigma(s0 - s1), sigma(s1 - s0)), sigma the
    logistic function, with s_j = <q, k_j> / sqrt(d)."""
    rng = _rng(7)
    d = 16
    Q, K, V = _qkv(rng, 1, 6, 3, 2, d)
    O, W = orc.sdpa(Q, K, V, return_weights=True)
    for h in range(6):
        for i in range(3):
            s0 = math.fsum(Q[0, h, i] * K[0, h, 0]) / math.sqrt(d)
            s1 = math.fsum(Q[0, h, i] * K[0, h, 1]) / math.sqrt(d)
            w0 = 1.0 / (1.0 + math.exp(s1 - s0))
            assert abs(W[0, h, i, 0] - w0) <= 1e-14, "two-key weight"
            assert abs(W[0, h, i, 1] - (1.0 - w0)) <= 1e-14
            exp_o = w0 * V[0, h, 0] + (1.0 - w0) * V[0, h, 1]
            _allclose(O[0, h, i], exp_o, 1e-14, "two-key output")


def pin_one_hot_margin(orc):
    """A key whose score beats every other by a margin g gets all but
    (n-1)e^-g of the weight, so the output is that key's value row."""
    rng = _rng(8)
    d, Lk = 32, 10
    for target in (0, 4, 9):
        q = rng.standard_normal(d)
        q /= np.linalg.norm(q)
        K = rng.standard_normal((Lk, d)) * 0.01
        gap = 30.0
        K[target] = q * gap * math.sqrt(d)          # scaled score ~= gap
        V = rng.standard_normal((Lk, d))
        O = orc.sdpa(q[None, None, None], K[None, None], V[None, None])
        bound = (Lk - 1) * math.exp(-gap + 2.0) * np.max(np.abs(V)) * 2
        _allclose(O[0, 0, 0], V[target], bound, "one-hot")


def pin_score_variance(orc):
    """For i.i.d. N(0,1) q, k the raw score has variance d_k and the scaled
    one variance 1.  With two keys the weight w0 = sigma(s0 - s1) exposes the
    score difference, whose variance is 2 (scaled) or 2 d_k (unscaled)."""
    rng = _rng(9)
    N = 20000
    for d in (64, 128):
        Q, K, V = _qkv(rng, 1, N, 1, 2, d)
        for scale, target in ((0.0, 2.0), (1.0, 2.0 * d)):
            _, W = orc.sdpa(Q, K, V, scale=scale, return_weights=True)
            diff = np.log(W[0, :, 0, 0]) - np.log(W[0, :, 0, 1])
            var = float(np.var(diff))
            rel_sd = math.sqrt((2.0 + 6.0 / d) / N)
            assert abs(var / target - 1.0) <= 5 * rel_sd, \
                f"d={d} scale={scale}: var {var:.4f} vs {target}"


def pin_kv_permutation_and_shift(orc):
    rng = _rng(10)
    B, H, Lq, Lk, d = 2, 2, 5, 9, 8
    Q, K, V = _qkv(rng, B, H, Lq, Lk, d)
    O = orc.sdpa(Q, K, V)
    perm = rng.permutation(Lk)
    _allclose(orc.sdpa(Q, K[:, :, perm], V[:, :, perm]), O, 1e-13, "kv permutation")
    w = rng.standard_normal(d) * 3
    _allclose(orc.sdpa(Q, K + w, V), O, 1e-12, "key shift")


def pin_torch_sdpa(orc):
    """Library cross-check: torch's CPU float64 scaled_dot_product_attention."""
    import torch
    import torch.nn.functional as F
    rng = _rng(11)
    cases = [(2, 3, 17, 17, 16, MASK_NONE), (2, 2, 13, 13, 32, MASK_CAUSAL),
             (3, 2, 11, 20, 8, MASK_KEY_PADDING), (1, 2, 19, 19, 64, MASK_CAUSAL | MASK_KEY_PADDING),
             (2, 1, 5, 33, 128, MASK_NONE)]
    for B, H, Lq, Lk, d, mk in cases:
        Q, K, V = _qkv(rng, B, H, Lq, Lk, d)
        lens = rng.integers(1, Lk + 1, size=B).astype(np.int32) if mk & MASK_KEY_PADDING else None
        if mk & MASK_KEY_PADDING and mk & MASK_CAUSAL:
            lens = np.maximum(lens, 1)
        add = np.zeros((B, 1, Lq, Lk))
        if mk & MASK_CAUSAL:
            add += np.triu(np.full((Lq, Lk), -np.inf), 1)[None, None]
        if mk & MASK_KEY_PADDING:
            for b in range(B):
                add[b, :, :, lens[b]:] = -np.inf
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q), torch.from_numpy(K),
                                             torch.from_numpy(V),
                                             attn_mask=torch.from_numpy(add)).numpy()
        got = orc.sdpa(Q, K, V, mask_kind=mk, key_lengths=lens)
        _allclose(got, ref, 1e-12, f"torch sdpa {B,H,Lq,Lk,d,mk}")
    # explicit scale
    Q, K, V = _qkv(rng, 1, 2, 6, 6, 16)
    ref = F.scaled_dot_product_attention(torch.from_numpy(Q), torch.from_numpy(K),
                                         torch.from_numpy(V), scale=0.3).numpy()
    _allclose(orc.sdpa(Q, K, V, scale=0.3), ref, 1e-12, "explicit scale")


def pin_sdpa_rows_match_full(orc):
    rng = _rng(12)
    B, H, L, d = 2, 3, 21, 16
    Q, K, V = _qkv(rng, B, H, L, L, d)
    for mk, lens in ((MASK_CAUSAL, None), (MASK_KEY_PADDING, np.array([4, 21], np.int32))):
        full = orc.sdpa(Q, K, V, mask_kind=mk, key_lengths=lens)
        rows = np.array([0, 5, 20, 21, 40, 62, 125], dtype=np.int64)
        got = orc.sdpa_rows(Q, K, V, rows, mask_kind=mk, key_lengths=lens)
        assert np.array_equal(got, full.reshape(-1, d)[rows]), "row sample differs"


def pin_printed_mask_as_float_mask(orc):
    """The printed 4x4 mask given as an additive float mask is the causal mask:
    the outputs are identical to mask_kind = causal, bit for bit."""
    mask = read_mask_fixture()
    rng = _rng(13)
    Q, K, V = _qkv(rng, 2, 3, 4, 4, 8)
    a = orc.sdpa(Q, K, V, add_mask=mask)
    b = orc.sdpa(Q, K, V, mask_kind=MASK_CAUSAL)
    assert np.array_equal(a, b), "float form of the printed mask differs from causal"


def pin_float_mask_torch(orc):
    """Library cross-check: a float mask with finite values and -inf entries,
    per head and broadcast, against torch's float64 SDPA attn_mask."""
    import torch
    import torch.nn.functional as F
    rng = _rng(14)
    for B, H, Lq, Lk, d, per in ((2, 3, 9, 13, 16, "head"), (1, 2, 7, 7, 32, "bcast"),
                                 (3, 1, 5, 20, 8, "batch")):
        Q, K, V = _qkv(rng, B, H, Lq, Lk, d)
        shape = {"head": (B, H, Lq, Lk), "bcast": (Lq, Lk), "batch": (B, 1, Lq, Lk)}[per]
        m = rng.standard_normal(shape) * 3.0
        m[rng.random(shape) < 0.3] = -np.inf
        m[..., 0] = 0.0                      # every row keeps key 0 visible
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V),
            attn_mask=torch.from_numpy(np.broadcast_to(m, (B, H, Lq, Lk)).copy())).numpy()
        _allclose(orc.sdpa(Q, K, V, add_mask=m), ref, 1e-12, f"float mask {per}")


def pin_float_mask_row_shift(orc):
    """Adding one constant to a whole mask row changes nothing (softmax shift
    invariance); adding it to one entry does."""
    rng = _rng(15)
    Q, K, V = _qkv(rng, 1, 2, 6, 9, 8)
    m = rng.standard_normal((6, 9))
    base = orc.sdpa(Q, K, V, add_mask=m)
    _allclose(orc.sdpa(Q, K, V, add_mask=m + rng.standard_normal((6, 1)) * 4), base,
              1e-12, "row shift")
    m2 = m.copy()
    m2[2, 3] += 2.0
    assert not np.allclose(orc.sdpa(Q, K, V, add_mask=m2)[0, :, 2], base[0, :, 2])


# ----------------------------------------------------------------- MHA pins

def _mha_inputs(rng, B, Lq, Lk, D, cross=True):
    xq = rng.standard_normal((B, Lq, D))
    xkv = rng.standard_normal((B, Lk, D)) if cross else xq
    Ws = [rng.standard_normal((D, D)) / math.sqrt(D) for _ in range(4)]
    return xq, xkv, Ws


def _torch_mha(xq, xkv, Ws, h, causal=False, lens=None):
    import torch
    import torch.nn.functional as F
    Wq, Wk, Wv, Wo = (torch.from_numpy(np.ascontiguousarray(w.T)) for w in Ws)
    D = xq.shape[-1]
    q = torch.from_numpy(xq).transpose(0, 1)
    kv = torch.from_numpy(xkv).transpose(0, 1)
    Lq, Lk = xq.shape[1], xkv.shape[1]
    attn_mask = None
    if causal:
        attn_mask = torch.triu(torch.full((Lq, Lk), float("-inf"), dtype=torch.float64), 1)
    kpm = None
    if lens is not None:
        kpm = torch.arange(Lk)[None, :] >= torch.from_numpy(np.asarray(lens))[:, None]
    out, _ = F.multi_head_attention_forward(
        q, kv, kv, D, h, None, None, None, None, False, 0.0, Wo, None,
        training=False, key_padding_mask=kpm, need_weights=False, attn_mask=attn_mask,
        use_separate_proj_weight=True, q_proj_weight=Wq, k_proj_weight=Wk,
        v_proj_weight=Wv)
    return out.transpose(0, 1).numpy()


def pin_mha_torch(orc):
    """Library cross-check: torch.nn.functional.multi_head_attention_forward,
    float64, separate projection weights (transposed: torch computes x W^T),
    no biases."""
    rng = _rng(20)
    cases = [(2, 9, 9, 32, 4, MASK_NONE, False), (1, 12, 12, 48, 3, MASK_CAUSAL, False),
             (2, 7, 13, 32, 2, MASK_KEY_PADDING, True), (3, 5, 11, 64, 8, MASK_NONE, True)]
    for B, Lq, Lk, D, h, mk, cross in cases:
        xq, xkv, Ws = _mha_inputs(rng, B, Lq, Lk, D, cross)
        lens = rng.integers(1, Lk + 1, size=B).astype(np.int32) if mk & MASK_KEY_PADDING else None
        ref = _torch_mha(xq, xkv, Ws, h, causal=bool(mk & MASK_CAUSAL), lens=lens)
        got = orc.mha(xq, xkv, *Ws, h=h, mask_kind=mk, key_lengths=lens)
        _allclose(got, ref, 1e-11, f"torch mha {B,Lq,Lk,D,h,mk}")


def pin_mha_single_head_identity(orc):
    """h = 1 and every W = I: the layer is SDPA(x, x, x) with scale 1/sqrt(D)."""
    rng = _rng(21)
    B, L, D = 2, 6, 16
    x = rng.standard_normal((B, L, D))
    I = np.eye(D)
    got = orc.mha(x, x, I, I, I, I, h=1)
    ref = orc.sdpa(x[:, None], x[:, None], x[:, None], scale=1.0 / math.sqrt(D))[:, 0]
    _allclose(got, ref, 1e-13, "single head identity")


def pin_mha_head_blocks(orc):
    """out = sum_i head_i @ Wo[rows of block i], head_i = SDPA on column block i."""
    rng = _rng(22)
    B, Lq, Lk, D, h = 2, 5, 7, 24, 3
    d = D // h
    xq, xkv, (Wq, Wk, Wv, Wo) = _mha_inputs(rng, B, Lq, Lk, D)
    got = orc.mha(xq, xkv, Wq, Wk, Wv, Wo, h=h)
    acc = np.zeros((B, Lq, D))
    for i in range(h):
        blk = slice(i * d, (i + 1) * d)
        head = orc.sdpa((xq @ Wq[:, blk])[:, None], (xkv @ Wk[:, blk])[:, None],
                        (xkv @ Wv[:, blk])[:, None])[:, 0]
        acc += head @ Wo[blk, :]
    _allclose(got, acc, 1e-12, "head block decomposition")


def pin_mha_permutation_equivariance(orc):
    rng = _rng(23)
    B, L, D, h = 2, 8, 32, 4
    x, _, Ws = _mha_inputs(rng, B, L, L, D, cross=False)
    out = orc.mha(x, x, *Ws, h=h)
    perm = rng.permutation(L)
    xp = x[:, perm]
    _allclose(orc.mha(xp, xp, *Ws, h=h), out[:, perm], 1e-12, "permutation equivariance")


def pin_mha_linearity(orc):
    rng = _rng(24)
    B, Lq, Lk, D, h = 1, 4, 6, 16, 2
    xq, xkv, (Wq, Wk, Wv, Wo) = _mha_inputs(rng, B, Lq, Lk, D)
    Wo2 = rng.standard_normal((D, D))
    Wv2 = rng.standard_normal((D, D))
    a = orc.mha(xq, xkv, Wq, Wk, Wv, Wo + Wo2, h=h)
    b = orc.mha(xq, xkv, Wq, Wk, Wv, Wo, h=h) + orc.mha(xq, xkv, Wq, Wk, Wv, Wo2, h=h)
    _allclose(a, b, 1e-12, "linear in Wo")
    a = orc.mha(xq, xkv, Wq, Wk, Wv + Wv2, Wo, h=h)
    b = orc.mha(xq, xkv, Wq, Wk, Wv, Wo, h=h) + orc.mha(xq, xkv, Wq, Wk, Wv2, Wo, h=h)
    _allclose(a, b, 1e-12, "linear in Wv")


# --------------------------------------------------------- encoder layer

def read_params_fixture():
    vals = {}
    with open(os.path.join(GOLDEN, "encoder_layer_params.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def _encoder_params(rng, D, F, scale=1.0):
    p = {}
    for n in ("Wq", "Wk", "Wv", "Wo"):
        p[n] = rng.standard_normal((D, D)) / math.sqrt(D)
    for n in ("bq", "bk", "bv", "bo", "b2", "ln1_beta", "ln2_beta"):
        p[n] = rng.standard_normal(D) * 0.1 * scale
    p["b1"] = rng.standard_normal(F) * 0.1 * scale
    p["W1"] = rng.standard_normal((D, F)) / math.sqrt(D)
    p["W2"] = rng.standard_normal((F, D)) / math.sqrt(F)
    p["ln1_gamma"] = 1.0 + rng.standard_normal(D) * 0.1 * scale
    p["ln2_gamma"] = 1.0 + rng.standard_normal(D) * 0.1 * scale
    return p


def pin_encoder_param_count(orc):
    """The printed parameter count of the base encoder layer, and the FFN's
    two-thirds share of it."""
    g = read_params_fixture()
    D, F = g["d_model"], g["d_ff"]
    assert orc.encoder_num_params(D, F) == g["params"]
    ffn = D * F + F + F * D + D
    assert abs(ffn / g["params"] - 2.0 / 3.0) < 0.005
    # and the arrays the layer consumes add up to the same count
    rng = _rng(30)
    p = _encoder_params(rng, D, F)
    assert sum(a.size for a in p.values()) == g["params"]


def _torch_encoder(x, p, h, causal=False, lens=None):
    import torch
    D = x.shape[-1]
    F = p["W1"].shape[1]
    layer = torch.nn.TransformerEncoderLayer(D, h, F, dropout=0.0, activation="relu",
                                             batch_first=True, norm_first=False,
                                             dtype=torch.float64)
    layer.eval()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    with torch.no_grad():
        layer.self_attn.in_proj_weight.copy_(t(np.concatenate([p["Wq"].T, p["Wk"].T, p["Wv"].T])))
        layer.self_attn.in_proj_bias.copy_(t(np.concatenate([p["bq"], p["bk"], p["bv"]])))
        layer.self_attn.out_proj.weight.copy_(t(p["Wo"].T))
        layer.self_attn.out_proj.bias.copy_(t(p["bo"]))
        layer.linear1.weight.copy_(t(p["W1"].T))
        layer.linear1.bias.copy_(t(p["b1"]))
        layer.linear2.weight.copy_(t(p["W2"].T))
        layer.linear2.bias.copy_(t(p["b2"]))
        layer.norm1.weight.copy_(t(p["ln1_gamma"]))
        layer.norm1.bias.copy_(t(p["ln1_beta"]))
        layer.norm2.weight.copy_(t(p["ln2_gamma"]))
        layer.norm2.bias.copy_(t(p["ln2_beta"]))
        L = x.shape[1]
        mask = torch.triu(torch.full((L, L), float("-inf"), dtype=torch.float64), 1) if causal else None
        kpm = None
        if lens is not None:
            kpm = torch.arange(L)[None, :] >= torch.from_numpy(np.asarray(lens))[:, None]
        return layer(t(x), src_mask=mask, src_key_padding_mask=kpm).numpy()


def pin_encoder_torch(orc):
    """Library cross-check: torch.nn.TransformerEncoderLayer (post-norm, ReLU,
    no dropout) in float64 with the same weights (transposed: torch applies
    x W^T)."""
    rng = _rng(31)
    for B, L, D, h, F, mk in ((2, 7, 32, 4, 64, MASK_NONE), (1, 9, 48, 3, 96, MASK_CAUSAL),
                              (3, 6, 16, 2, 40, MASK_KEY_PADDING)):
        x = rng.standard_normal((B, L, D))
        p = _encoder_params(rng, D, F)
        lens = np.array([6, 2, 4], np.int32) if mk == MASK_KEY_PADDING else None
        ref = _torch_encoder(x, p, h, causal=mk == MASK_CAUSAL, lens=lens)
        got = orc.encoder_layer(x, p, h, mask_kind=mk, key_lengths=lens)
        _allclose(got, ref, 1e-10, f"torch encoder layer {B, L, D, h, F, mk}")


def pin_encoder_layernorm_rows(orc):
    """With gamma = 1 and beta = 0 every output row has mean 0 and variance 1
    (up to eps), and the layer is permutation-equivariant over positions."""
    rng = _rng(32)
    B, L, D, h, F = 2, 8, 32, 4, 64
    x = rng.standard_normal((B, L, D)) * 3
    p = _encoder_params(rng, D, F)
    p["ln2_gamma"] = np.ones(D)
    p["ln2_beta"] = np.zeros(D)
    y = orc.encoder_layer(x, p, h, eps=0.0)
    _allclose(y.mean(-1), np.zeros((B, L)), 1e-12, "row means")
    _allclose(y.var(-1), np.ones((B, L)), 1e-10, "row variances")
    perm = rng.permutation(L)
    _allclose(orc.encoder_layer(x[:, perm], p, h), orc.encoder_layer(x, p, h)[:, perm], 1e-11,
              "permutation equivariance")


# ------------------------------------------------------- decode-shape pins

def pin_decode_equals_full_causal_rows(orc):
    """Attending from the last Lq positions of each sequence against a cache
    of capacity Lmax holding len_b tokens (garbage beyond) reproduces, bit for
    bit, rows len_b - Lq .. len_b - 1 of the full causal pass; Lq = 1 is key
    padding alone; Lq = len_b = Lmax is the causal mask."""
    rng = _rng(40)
    B, H, n, d, Lmax = 3, 2, 37, 16, 45
    Qf, Kf, Vf = _qkv(rng, B, H, n, n, d)
    full = orc.sdpa(Qf, Kf, Vf, mask_kind=MASK_CAUSAL)
    lens = np.array([37, 20, 5], np.int32)
    Kc = rng.standard_normal((B, H, Lmax, d)) * 7
    Vc = rng.standard_normal((B, H, Lmax, d)) * 7
    for b in range(B):
        Kc[b, :, : lens[b]] = Kf[b, :, : lens[b]]
        Vc[b, :, : lens[b]] = Vf[b, :, : lens[b]]
    mk = MASK_CAUSAL_BOTTOM_RIGHT | MASK_KEY_PADDING
    for Lq in (1, 4, 5):
        Q = np.stack([Qf[b, :, lens[b] - Lq: lens[b]] for b in range(B)])
        O = orc.sdpa(Q, Kc, Vc, mask_kind=mk, key_lengths=lens)
        assert orc.last_bad_rows == 0
        for b in range(B):
            assert np.array_equal(O[b], full[b, :, lens[b] - Lq: lens[b]]), \
                f"decode rows differ from the causal pass (Lq {Lq}, b {b})"
        if Lq == 1:
            Op = orc.sdpa(Q, Kc, Vc, mask_kind=MASK_KEY_PADDING, key_lengths=lens)
            assert np.array_equal(O, Op), "Lq = 1 is not key padding alone"
    O = orc.sdpa(Qf, Kf, Vf, mask_kind=MASK_CAUSAL_BOTTOM_RIGHT)
    assert np.array_equal(O, full), "square bottom-right is not the causal mask"


def pin_decode_torch_lower_right(orc):
    """Library cross-check: torch float64 SDPA with the ``causal_lower_right``
    bias (Lq <= Lk, no padding)."""
    import torch
    import torch.nn.functional as F
    from torch.nn.attention.bias import causal_lower_right
    rng = _rng(41)
    for B, H, Lq, Lk, d in ((2, 3, 1, 50, 16), (1, 2, 7, 19, 8), (2, 1, 16, 200, 32)):
        Q, K, V = _qkv(rng, B, H, Lq, Lk, d)
        t = torch.from_numpy
        ref = F.scaled_dot_product_attention(t(Q), t(K), t(V),
                                             attn_mask=causal_lower_right(Lq, Lk)).numpy()
        _allclose(orc.sdpa(Q, K, V, mask_kind=MASK_CAUSAL_BOTTOM_RIGHT), ref, 1e-12,
                  f"torch lower-right causal {B, H, Lq, Lk, d}")


# ----------------------------------------------------------- backward pass

def _torch_sdpa_grads(Q, K, V, dO, mask=None, scale=None):
    import torch
    import torch.nn.functional as F
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).requires_grad_(True)
    q, k, v = t(Q), t(K), t(V)
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    o.backward(torch.from_numpy(dO))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def pin_backward_torch(orc):
    """Library cross-check: torch float64 autograd, every mask kind."""
    import torch
    from torch.nn.attention.bias import causal_lower_right
    rng = _rng(60)
    B, H, Lq, Lk, d = 2, 3, 6, 9, 8
    Q, K, V = _qkv(rng, B, H, Lq, Lk, d)
    dO = rng.standard_normal(Q.shape)
    for name, mk, lens, mask in (
            ("none", MASK_NONE, None, None),
            ("padding", MASK_KEY_PADDING, np.array([9, 3], np.int32),
             torch.from_numpy(np.arange(Lk)[None, None, None, :] <
                              np.array([9, 3])[:, None, None, None])),
            ("bottom-right", MASK_CAUSAL_BOTTOM_RIGHT, None, causal_lower_right(Lq, Lk))):
        got = orc.sdpa_backward(Q, K, V, dO, mask_kind=mk, key_lengths=lens)
        ref = _torch_sdpa_grads(Q, K, V, dO, mask=mask)
        for gname, a, b in zip(("dQ", "dK", "dV"), got, ref):
            _allclose(a, b, 1e-12, f"torch {gname} {name}")
    Qs, Ks, Vs = _qkv(rng, 1, 2, 7, 7, 8)
    dOs = rng.standard_normal(Qs.shape)
    got = orc.sdpa_backward(Qs, Ks, Vs, dOs, scale=0.7, mask_kind=MASK_CAUSAL)
    causal = torch.from_numpy(np.tril(np.ones((7, 7), dtype=bool)))
    ref = _torch_sdpa_grads(Qs, Ks, Vs, dOs, mask=causal, scale=0.7)
    for gname, a, b in zip(("dQ", "dK", "dV"), got, ref):
        _allclose(a, b, 1e-12, f"torch {gname} causal, scale 0.7")


def pin_backward_finite_differences(orc):
    """dL/dx for L = sum(dO * O) against central differences of the oracle's
    own forward, entry by entry on a tiny head."""
    rng = _rng(61)
    Q, K, V = _qkv(rng, 1, 1, 3, 4, 3)
    dO = rng.standard_normal(Q.shape)
    dQ, dK, dV = orc.sdpa_backward(Q, K, V, dO, mask_kind=MASK_CAUSAL_BOTTOM_RIGHT)
    loss = lambda q, k, v: float(np.sum(dO * orc.sdpa(q, k, v,
                                                      mask_kind=MASK_CAUSAL_BOTTOM_RIGHT)))
    eps = 1e-6
    for which, grad in ((0, dQ), (1, dK), (2, dV)):
        for idx in np.ndindex(grad.shape):
            args_p = [Q.copy(), K.copy(), V.copy()]
            args_m = [Q.copy(), K.copy(), V.copy()]
            args_p[which][idx] += eps
            args_m[which][idx] -= eps
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-8, (which, idx, fd, grad[idx])


def pin_backward_softmax_structure(orc):
    """Each row of dS sums to zero: the key gradients of a head sum to zero,
    shifting every key by one vector leaves dQ unchanged, and with every key
    visible the value gradients sum to the sum of dO.  Blocked keys (beyond a
    length, or later than a causal query) get exactly zero gradient."""
    rng = _rng(62)
    B, H, Lq, Lk, d = 2, 2, 5, 8, 6
    Q, K, V = _qkv(rng, B, H, Lq, Lk, d)
    dO = rng.standard_normal(Q.shape)
    dQ, dK, dV = orc.sdpa_backward(Q, K, V, dO)
    _allclose(dK.sum(axis=2), np.zeros((B, H, d)), 1e-12, "sum of dK")
    _allclose(dV.sum(axis=2), dO.sum(axis=2), 1e-12, "sum of dV = sum of dO")
    shift = rng.standard_normal(d)
    _allclose(orc.sdpa_backward(Q, K + shift, V, dO)[0], dQ, 1e-11, "dQ under a key shift")
    lens = np.array([3, 8], np.int32)
    _, dKp, dVp = orc.sdpa_backward(Q, K, V, dO, mask_kind=MASK_KEY_PADDING, key_lengths=lens)
    assert np.all(dKp[0, :, 3:] == 0.0) and np.all(dVp[0, :, 3:] == 0.0)
    Qc, Kc, Vc = _qkv(rng, 1, 1, 6, 6, 4)
    dOc = rng.standard_normal(Qc.shape)
    dOc[:, :, 4:] = 0.0       # only queries 0..3 carry gradient
    _, dKc, dVc = orc.sdpa_backward(Qc, Kc, Vc, dOc, mask_kind=MASK_CAUSAL)
    assert np.all(dKc[:, :, 4:] == 0.0) and np.all(dVc[:, :, 4:] == 0.0)


def pin_backward_saturation(orc):
    """A row whose top score leads by a margin g is nearly one-hot, and the
    gradient reaching its other keys shrinks like e^-g (the saturation that
    scaling by 1/sqrt(dk) is there to avoid)."""
    d, Lk = 4, 6
    prev, prev_gap = None, None
    for gap in (4.0, 8.0, 16.0):
        Q = np.zeros((1, 1, 1, d))
        Q[..., 0] = 1.0
        K = np.zeros((1, 1, Lk, d))
        K[..., 0, 0] = gap      # key 0 leads by gap in the scaled score
        V = _rng(63).standard_normal((1, 1, Lk, d))
        dO = np.ones((1, 1, 1, d))
        _, dK, _ = orc.sdpa_backward(Q, K, V, dO, scale=1.0)
        inactive = float(np.abs(dK[0, 0, 1:]).max())
        assert inactive <= 4.0 * Lk * math.exp(-gap) * (np.abs(V).max() * d + 1.0)
        if prev is not None:
            # decays like e^-gap (up to the normaliser of the softmax)
            assert inactive < 1.5 * prev * math.exp(-(gap - prev_gap))
        prev, prev_gap = inactive, gap


# ------------------------------------------------------ positional encoding

def pin_pe_position_zero(orc):
    """At position 0 every sine column is 0 and every cosine column is 1."""
    for D in (8, 64, 512, 7):
        pe = orc.sinusoidal_pe(1, D)[0]
        assert np.all(pe[0::2] == 0.0) and np.all(pe[1::2] == 1.0), D


def pin_pe_pairs_rotate(orc):
    """Each (sin, cos) pair lies on the unit circle, and shifting the position
    by k turns every pair by the angle it has at position k: a fixed
    rotation per pair, whatever the start position."""
    D = 64
    pe = orc.sinusoidal_pe(300, D)
    s, c = pe[:, 0::2], pe[:, 1::2]
    _allclose(s * s + c * c, np.ones_like(s), 1e-14, "unit circle")
    for k in (1, 7, 100):
        sk, ck = s[k], c[k]          # position k from position 0 = (0, 1)
        pred_s = s[:-k] * ck + c[:-k] * sk
        pred_c = c[:-k] * ck - s[:-k] * sk
        _allclose(pred_s, s[k:], 1e-11, f"shift {k} (sin)")
        _allclose(pred_c, c[k:], 1e-11, f"shift {k} (cos)")


def pin_pe_frequencies(orc):
    """Pair 0 turns 1 rad per position; each next pair turns slower by the
    same factor, down to 1/10000 rad per position (10000^(-2/D) per pair)."""
    for D in (16, 512):
        pe = orc.sinusoidal_pe(2, D)
        w = np.arctan2(pe[1, 0::2], pe[1, 1::2])   # angle turned in one position
        assert abs(w[0] - 1.0) < 1e-15
        ratios = w[1:] / w[:-1]
        _allclose(ratios, np.full_like(ratios, 10000.0 ** (-2.0 / D)), 1e-12, f"ratio D={D}")
        assert abs(math.log(w[-1] / w[0]) / math.log(1e-4) - (D - 2) / D) < 1e-12


def pin_embed_torch_and_offset(orc):
    """x = embedding * sqrt(D) + PE: the lookup against torch's embedding in
    float64, and a window starting at position k equals columns k.. of the
    whole sequence (the position offset)."""
    import torch
    rng = _rng(50)
    vocab, D, B, L = 37, 16, 2, 9
    table = rng.standard_normal((vocab, D))
    ids = rng.integers(0, vocab, size=(B, L)).astype(np.int32)
    x = orc.embed_pe(ids, table)
    emb = torch.nn.functional.embedding(torch.from_numpy(ids.astype(np.int64)),
                                        torch.from_numpy(table)).numpy()
    _allclose(x - orc.sinusoidal_pe(L, D)[None], emb * math.sqrt(D), 1e-12, "torch embedding")
    for k in (1, 4):
        assert np.array_equal(orc.embed_pe(ids[:, k:].copy(), table, pos_offset=k), x[:, k:])
    _allclose(orc.embed_pe(ids, table, scale=1.0) - orc.sinusoidal_pe(L, D)[None], emb, 1e-12,
              "explicit scale 1")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
