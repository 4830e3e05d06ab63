"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and rounds them to the storage type; it
holds none of the attention arithmetic.  Both the CUDA path (through the tests
and the benchmark) and the CPU oracle are fed from it, so both see exactly the
same input values.

Generator: numpy's PCG64 bit generator (O'Neill, "PCG: A Family of Simple Fast
Space-Efficient Statistically Good Algorithms for Random Number Generation")
with numpy's ziggurat normal sampler, seeded with ``0x5EED0000 + workload id``.
Both are platform independent, so x86 and Arm hosts draw the same values.
Normal draws are made in float32 and then rounded to the storage type: bf16 by
round-to-nearest-even on the bit pattern, fp32 as drawn.  The arrays returned
are float32 holding values that are exactly representable in the storage
type, so upcasting them to float64 for the oracle is exact.

Draw order per workload: Q, K, V (or x, Wq, Wk, Wv, Wo), then key lengths,
then outlier dimensions.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KEY_PADDING = 2
MASK_CAUSAL_BOTTOM_RIGHT = 4

SEED_BASE = 0x5EED0000


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 out."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


class Draws:
    """One seeded stream of draws."""

    def __init__(self, seed: int):
        self.rng = np.random.Generator(np.random.PCG64(int(seed)))

    def normal(self, shape, std: float = 1.0, dtype: str = "bf16") -> np.ndarray:
        x = self.rng.standard_normal(size=shape, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if dtype == "bf16":
            return round_to_bf16(x)
        if dtype == "f32":
            return x
        raise ValueError(dtype)

    def integers(self, lo: int, hi_inclusive: int, size) -> np.ndarray:
        return self.rng.integers(lo, hi_inclusive + 1, size=size, dtype=np.int64).astype(np.int32)

    def choice(self, n: int, k: int) -> np.ndarray:
        return np.sort(self.rng.choice(n, size=k, replace=False))


@dataclass
class Workload:
    """Shapes and input recipe of one attention workload."""
    wid: int
    name: str
    kind: str                  # "sdpa" or "mha"
    dtype: str                 # "bf16" or "f32"
    B: int
    H: int
    Lq: int
    Lk: int
    d: int
    mask: int = MASK_NONE
    len_range: tuple | None = None      # key lengths, inclusive
    outliers: tuple | None = None       # (dims per head, factor) on Q and K
    w_std: float | None = None          # projection weight std (mha)
    notes: dict = field(default_factory=dict)

    @property
    def D(self) -> int:
        return self.H * self.d

    @property
    def seed(self) -> int:
        return SEED_BASE + self.wid

    def flops(self, key_lengths=None) -> float:
        """Algorithmic SDPA flops: 4*d per unmasked (query, key) pair."""
        B, H, Lq, Lk, d = self.B, self.H, self.Lq, self.Lk, self.d
        if self.mask & MASK_CAUSAL:
            return 2.0 * B * H * d * Lq * (Lq + 1)
        if self.mask & MASK_CAUSAL_BOTTOM_RIGHT:
            # query i of Lq sees len_b - Lq + i + 1 keys
            lens = (np.full(B, Lk) if key_lengths is None
                    else np.asarray(key_lengths, dtype=np.float64))
            pairs = float(np.sum(Lq * (lens - Lq) + Lq * (Lq + 1) / 2.0))
            return 4.0 * H * d * pairs
        if self.mask & MASK_KEY_PADDING:
            assert key_lengths is not None
            return 4.0 * H * Lq * d * float(np.sum(key_lengths))
        return 4.0 * B * H * Lq * Lk * d

    def sdpa_bytes(self, key_lengths=None) -> float:
        """Minimum HBM bytes of one attention forward (bf16): Q read and O
        written once, and every key and value row that some query may see
        read once (rows at or past len_b are never read under key padding)."""
        kv_rows = (float(np.sum(key_lengths)) if self.mask & MASK_KEY_PADDING
                   and key_lengths is not None else float(self.B * self.Lk))
        return 2.0 * self.H * self.d * (2.0 * self.B * self.Lq + 2.0 * kv_rows)

    def decode_bytes(self, key_lengths=None) -> float:
        """Algorithmic HBM bytes of one decode pass (bf16): every held key and
        value row read once, the queries read and the outputs written once."""
        lens = np.full(self.B, self.Lk) if key_lengths is None else np.asarray(key_lengths)
        return 2.0 * self.H * self.d * (2.0 * float(np.sum(lens)) + 2.0 * self.B * self.Lq)


WORKLOADS = {
    1: Workload(1, "mha self-attention base shape (B1 L128 D512 h8 fp32)", "mha", "f32",
                B=1, H=8, Lq=128, Lk=128, d=64, w_std=1.0 / np.sqrt(512.0)),
    2: Workload(2, "encoder self-attention, key padding (B32 L512 H8 d64 bf16)", "sdpa",
                "bf16", B=32, H=8, Lq=512, Lk=512, d=64, mask=MASK_KEY_PADDING,
                len_range=(256, 512)),
    3: Workload(3, "decoder causal self-attention (B16 L2048 H16 d64 bf16)", "sdpa",
                "bf16", B=16, H=16, Lq=2048, Lk=2048, d=64, mask=MASK_CAUSAL),
    4: Workload(4, "encoder-decoder cross-attention (B64 Lq256 Lk1024 H8 d64 bf16)",
                "sdpa", "bf16", B=64, H=8, Lq=256, Lk=1024, d=64),
    5: Workload(5, "long-context causal (B1 L32768 H32 d128 bf16, outlier dims)", "sdpa",
                "bf16", B=1, H=32, Lq=32768, Lk=32768, d=128, mask=MASK_CAUSAL,
                outliers=(4, 8.0)),
    # decoding against a cache: the newest Lq positions of each sequence attend
    # to its len_b cached keys (bottom-right causal); lengths vary per item
    6: Workload(6, "decode, one new token (B8 H32 d128, cache 32768, lengths U[16384, 32768] bf16)",
                "decode", "bf16", B=8, H=32, Lq=1, Lk=32768, d=128,
                mask=MASK_CAUSAL_BOTTOM_RIGHT | MASK_KEY_PADDING, len_range=(16384, 32768)),
    7: Workload(7, "decode, 16 new tokens (B8 H32 d128, cache 32768, lengths U[16384, 32768] bf16)",
                "decode", "bf16", B=8, H=32, Lq=16, Lk=32768, d=128,
                mask=MASK_CAUSAL_BOTTOM_RIGHT | MASK_KEY_PADDING, len_range=(16384, 32768)),
    8: Workload(8, "decode, base width (B64 H8 d64, cache 4096, lengths U[1024, 4096] bf16)",
                "decode", "bf16", B=64, H=8, Lq=1, Lk=4096, d=64,
                mask=MASK_CAUSAL_BOTTOM_RIGHT | MASK_KEY_PADDING, len_range=(1024, 4096)),
}


def sdpa_inputs(w: Workload, seed: int | None = None, **override):
    """Q [B,H,Lq,d], K, V [B,H,Lk,d] (float32 arrays of storage-type values),
    key lengths [B] int32 or None, and the outlier dims [H, n] or None.

    ``override`` replaces shape fields (B, H, Lq, Lk, d) for reduced cases
    drawn with the same recipe."""
    B = override.get("B", w.B)
    H = override.get("H", w.H)
    Lq = override.get("Lq", w.Lq)
    Lk = override.get("Lk", w.Lk)
    d = override.get("d", w.d)
    g = Draws(w.seed if seed is None else seed)
    Q = g.normal((B, H, Lq, d), dtype=w.dtype)
    K = g.normal((B, H, Lk, d), dtype=w.dtype)
    V = g.normal((B, H, Lk, d), dtype=w.dtype)
    lengths = None
    if w.mask & MASK_KEY_PADDING:
        lo, hi = override.get("len_range", w.len_range)
        lengths = g.integers(max(1, min(lo, Lk)), min(hi, Lk), B)
    dims = None
    if w.outliers is not None:
        n, factor = w.outliers
        dims = np.stack([g.choice(d, n) for _ in range(H)])
        f = np.float32(factor)   # a power of two: the scaling is exact in bf16
        for h in range(H):
            Q[:, h, :, dims[h]] *= f
            K[:, h, :, dims[h]] *= f
    return Q, K, V, lengths, dims


def mha_inputs(w: Workload, seed: int | None = None, **override):
    """x [B,Lq,D] ~ N(0,1), Wq, Wk, Wv, Wo [D,D] ~ N(0, w_std^2)."""
    B = override.get("B", w.B)
    Lq = override.get("Lq", w.Lq)
    D = override.get("D", w.D)
    std = override.get("w_std", w.w_std if w.w_std is not None else 1.0 / np.sqrt(D))
    g = Draws(w.seed if seed is None else seed)
    x = g.normal((B, Lq, D), dtype=w.dtype)
    Ws = [g.normal((D, D), std=std, dtype=w.dtype) for _ in range(4)]
    return (x, *Ws)


def sample_rows(B: int, H: int, Lq: int, per_head: int, seed: int,
                must=(0, 1, 127, 128, 129)) -> np.ndarray:
    """Flat row ids (b*H+h)*Lq+i: for every (b,h) the rows in ``must``, the
    last row, every 4096-boundary row, then seeded random rows up to
    ``per_head`` rows per head."""
    g = Draws(seed)
    out = []
    fixed = set(i for i in must if i < Lq) | {Lq - 1}
    fixed |= set(range(4096, Lq, 4096)) | set(i - 1 for i in range(4096, Lq, 4096))
    fixed = sorted(fixed)
    for bh in range(B * H):
        rest = max(0, per_head - len(fixed))
        pool = np.setdiff1d(np.arange(Lq), np.array(fixed))
        extra = g.rng.choice(pool, size=min(rest, pool.size), replace=False) if rest else []
        rows = np.sort(np.concatenate([np.array(fixed), np.asarray(extra, dtype=np.int64)]))
        out.append(bh * Lq + rows)
    return np.concatenate(out).astype(np.int64)
