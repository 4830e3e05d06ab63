"""Plain fp64 CPU oracle for multi-head scaled dot-product attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports, links or loads anything from this package, and this package imports
nothing from the CUDA library.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double, no blocking or
fusion); this module only compiles it with gcc and marshals numpy arrays into
it.  What each function computes, and the passage of the pages it follows, is
stated in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KEY_PADDING = 2
MASK_CAUSAL_BOTTOM_RIGHT = 4

_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile ``src`` into a shared library at ``out`` (OpenMP if gcc has it)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", *extra_flags, src, "-o", out, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    return out


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    lp = ctypes.POINTER(ctypes.c_int64)
    c_int, c_double = ctypes.c_int, ctypes.c_double
    c_i64 = ctypes.c_int64
    lib.oracle_sdpa.argtypes = [dp, dp, dp, dp, dp, c_int, c_int, c_int, c_int,
                                c_int, c_double, c_int, ip, dp, c_i64, c_i64, c_int]
    lib.oracle_sdpa.restype = c_int
    lib.oracle_sdpa_rows.argtypes = [dp, dp, dp, dp, lp, c_int, c_int, c_int,
                                     c_int, c_int, c_int, c_double, c_int, ip,
                                     dp, c_i64, c_i64, c_int]
    lib.oracle_sdpa_rows.restype = c_int
    lib.oracle_mha.argtypes = [dp, dp, dp, dp, dp, dp, dp, c_int, c_int, c_int,
                               c_int, c_int, c_int, ip, c_int]
    lib.oracle_mha.restype = c_int
    lib.oracle_encoder_layer.argtypes = [dp] * 17 + [c_double, dp, c_int, c_int, c_int, c_int,
                                                     c_int, c_int, ip, c_int]
    lib.oracle_encoder_layer.restype = c_int
    lib.oracle_encoder_layer_num_params.argtypes = [c_int, c_int]
    lib.oracle_encoder_layer_num_params.restype = ctypes.c_long
    lib.oracle_sdpa_backward.argtypes = [dp] * 7 + [c_int] * 5 + [c_double, c_int, ip, c_int]
    lib.oracle_sdpa_backward.restype = c_int
    lib.oracle_sinusoidal_pe.argtypes = [dp, c_int, c_int, c_int]
    lib.oracle_sinusoidal_pe.restype = None
    lib.oracle_embed_pe.argtypes = [ip, dp, c_int, dp, c_int, c_int, c_int, c_int, c_double]
    lib.oracle_embed_pe.restype = c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = c_int
    return lib


def load_library(path: str | None = None):
    """Load (building first if needed) the oracle shared library.

    With ``path`` given, that library is loaded as is; it must export the same
    functions (the mutation tests use this to load deliberately broken
    copies)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _d(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray, ctype=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _add_mask(add_mask, B: int, H: int, Lq: int, Lk: int):
    """Additive float mask broadcastable to [B, H, Lq, Lk] -> (array, its
    pointer, batch stride, head stride) in elements; strides 0 broadcast."""
    if add_mask is None:
        return None, None, 0, 0
    a = np.asarray(add_mask, dtype=np.float64)
    while a.ndim < 4:
        a = a[None]
    if a.shape[2:] != (Lq, Lk) or a.shape[0] not in (1, B) or a.shape[1] not in (1, H):
        raise ValueError("additive mask must broadcast to [B, H, Lq, Lk]")
    a = np.ascontiguousarray(a)
    sb = a.shape[1] * Lq * Lk if a.shape[0] == B and B > 1 else 0
    sh = Lq * Lk if a.shape[1] == H and H > 1 else 0
    return a, _ptr(a), sb, sh


def _lengths(mask_kind: int, key_lengths, B: int):
    if mask_kind & MASK_KEY_PADDING:
        kl = np.ascontiguousarray(np.asarray(key_lengths, dtype=np.int32))
        if kl.shape != (B,):
            raise ValueError("key_lengths must have shape [B]")
        return kl, _ptr(kl, ctypes.c_int32)
    return None, None


class Oracle:
    """Thin marshalling wrapper; ``lib`` may be a mutated copy in tests."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load_library()

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def sdpa(self, Q, K, V, scale: float = 0.0, mask_kind: int = MASK_NONE,
             key_lengths=None, return_weights: bool = False, nthreads: int = 0,
             add_mask=None):
        """Q [B,H,Lq,d], K/V [B,H,Lk,d] -> O [B,H,Lq,d] (and weights [B,H,Lq,Lk]).

        ``add_mask``: optional float mask broadcastable to [B,H,Lq,Lk], added
        to the scaled scores."""
        Q, K, V = _d(Q), _d(K), _d(V)
        B, H, Lq, d = Q.shape
        Lk = K.shape[2]
        if K.shape != (B, H, Lk, d) or V.shape != (B, H, Lk, d):
            raise ValueError("shape mismatch")
        O = np.empty((B, H, Lq, d))
        W = np.empty((B, H, Lq, Lk)) if return_weights else None
        kl, klp = _lengths(mask_kind, key_lengths, B)
        am, amp, sb, sh = _add_mask(add_mask, B, H, Lq, Lk)
        bad = self.lib.oracle_sdpa(_ptr(Q), _ptr(K), _ptr(V), _ptr(O),
                                   _ptr(W) if W is not None else None, B, H, Lq,
                                   Lk, d, float(scale), int(mask_kind), klp, amp,
                                   sb, sh, int(nthreads))
        self.last_bad_rows = int(bad)
        return (O, W) if return_weights else O

    def sdpa_rows(self, Q, K, V, rows, scale: float = 0.0,
                  mask_kind: int = MASK_NONE, key_lengths=None,
                  nthreads: int = 0, add_mask=None):
        """Rows ``rows`` (flat (b*H+h)*Lq+i) of the attention output -> [n, d]."""
        Q, K, V = _d(Q), _d(K), _d(V)
        B, H, Lq, d = Q.shape
        Lk = K.shape[2]
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        out = np.empty((r.size, d))
        kl, klp = _lengths(mask_kind, key_lengths, B)
        am, amp, sb, sh = _add_mask(add_mask, B, H, Lq, Lk)
        bad = self.lib.oracle_sdpa_rows(_ptr(Q), _ptr(K), _ptr(V), _ptr(out),
                                        _ptr(r, ctypes.c_int64), int(r.size), B,
                                        H, Lq, Lk, d, float(scale),
                                        int(mask_kind), klp, amp, sb, sh,
                                        int(nthreads))
        self.last_bad_rows = int(bad)
        return out

    def mha(self, x_q, x_kv, Wq, Wk, Wv, Wo, h: int, mask_kind: int = MASK_NONE,
            key_lengths=None, nthreads: int = 0):
        """x_q [B,Lq,D], x_kv [B,Lk,D], W* [D,D] -> out [B,Lq,D]."""
        x_q, x_kv = _d(x_q), _d(x_kv)
        Wq, Wk, Wv, Wo = _d(Wq), _d(Wk), _d(Wv), _d(Wo)
        B, Lq, D = x_q.shape
        Lk = x_kv.shape[1]
        out = np.empty((B, Lq, D))
        kl, klp = _lengths(mask_kind, key_lengths, B)
        bad = self.lib.oracle_mha(_ptr(x_q), _ptr(x_kv), _ptr(Wq), _ptr(Wk),
                                  _ptr(Wv), _ptr(Wo), _ptr(out), B, Lq, Lk, D,
                                  int(h), int(mask_kind), klp, int(nthreads))
        if bad < 0:
            raise ValueError("d_model must be divisible by the number of heads")
        self.last_bad_rows = int(bad)
        return out


ENCODER_PARAM_NAMES = ("Wq", "Wk", "Wv", "Wo", "bq", "bk", "bv", "bo", "ln1_gamma",
                       "ln1_beta", "W1", "b1", "W2", "b2", "ln2_gamma", "ln2_beta")


def _encoder_layer(self, x, params: dict, h: int, eps: float = 1e-5,
                   mask_kind: int = MASK_NONE, key_lengths=None, nthreads: int = 0):
    """Post-norm encoder layer: x [B,L,D] and the parameters (names in
    ENCODER_PARAM_NAMES; W* [D,D], W1 [D,F], W2 [F,D], vectors 1-D) -> [B,L,D]."""
    x = _d(x)
    B, L, D = x.shape
    arrs = [_d(params[n]) for n in ENCODER_PARAM_NAMES]
    F = arrs[10].shape[1]
    out = np.empty((B, L, D))
    kl, klp = _lengths(mask_kind, key_lengths, B)
    # parameter pointers in ENCODER_PARAM_NAMES order = the C argument order
    bad = self.lib.oracle_encoder_layer(_ptr(x), *[_ptr(a) for a in arrs], float(eps),
                                        _ptr(out), B, L, D, int(h), F, int(mask_kind), klp,
                                        int(nthreads))
    if bad < 0:
        raise ValueError("d_model must be divisible by the number of heads")
    self.last_bad_rows = int(bad)
    return out


def _encoder_num_params(self, D: int, F: int) -> int:
    return int(self.lib.oracle_encoder_layer_num_params(D, F))


def _sinusoidal_pe(self, n_pos: int, D: int, first_pos: int = 0):
    """PE rows first_pos .. first_pos + n_pos - 1 -> [n_pos, D]."""
    pe = np.empty((n_pos, D))
    self.lib.oracle_sinusoidal_pe(_ptr(pe), int(first_pos), int(n_pos), int(D))
    return pe


def _embed_pe(self, ids, table, pos_offset: int = 0, scale: float = 0.0):
    """ids [B, L] int32, table [vocab, D] -> x [B, L, D] = table[ids] * scale
    + PE(pos_offset + l) (scale 0 selects sqrt(D))."""
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    table = _d(table)
    B, L = ids.shape
    vocab, D = table.shape
    x = np.empty((B, L, D))
    bad = self.lib.oracle_embed_pe(_ptr(ids, ctypes.c_int32), _ptr(table), vocab, _ptr(x), B, L,
                                   D, int(pos_offset), float(scale))
    self.last_bad_rows = int(bad)
    return x


def _sdpa_backward(self, Q, K, V, dO, scale: float = 0.0, mask_kind: int = MASK_NONE,
                   key_lengths=None, nthreads: int = 0):
    """Gradients (dQ, dK, dV) of sum(dO * sdpa(Q, K, V)) for Q [B,H,Lq,d],
    K/V [B,H,Lk,d], dO [B,H,Lq,d]."""
    Q, K, V, dO = _d(Q), _d(K), _d(V), _d(dO)
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    if K.shape != (B, H, Lk, d) or V.shape != (B, H, Lk, d) or dO.shape != Q.shape:
        raise ValueError("shape mismatch")
    dQ, dK, dV = np.empty_like(Q), np.empty_like(K), np.empty_like(V)
    kl, klp = _lengths(mask_kind, key_lengths, B)
    bad = self.lib.oracle_sdpa_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ), _ptr(dK),
                                        _ptr(dV), B, H, Lq, Lk, d, float(scale), int(mask_kind),
                                        klp, int(nthreads))
    self.last_bad_rows = int(bad)
    return dQ, dK, dV


Oracle.sdpa_backward = _sdpa_backward
Oracle.sinusoidal_pe = _sinusoidal_pe
Oracle.embed_pe = _embed_pe
Oracle.encoder_layer = _encoder_layer
Oracle.encoder_num_params = _encoder_num_params

_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def sdpa(*a, **k):
    return default().sdpa(*a, **k)


def sdpa_rows(*a, **k):
    return default().sdpa_rows(*a, **k)


def mha(*a, **k):
    return default().mha(*a, **k)


def encoder_layer(*a, **k):
    return default().encoder_layer(*a, **k)


def sinusoidal_pe(*a, **k):
    return default().sinusoidal_pe(*a, **k)


def embed_pe(*a, **k):
    return default().embed_pe(*a, **k)


def sdpa_backward(*a, **k):
    return default().sdpa_backward(*a, **k)
