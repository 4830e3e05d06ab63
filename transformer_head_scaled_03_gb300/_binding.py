"""ctypes binding of libmha_gb300.so (include/mha.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, and status codes become exceptions.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
or PyTorch fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MHA_OK = 0
MHA_ERR_INVALID_ARG = 1
MHA_ERR_UNSUPPORTED = 2
MHA_ERR_CUDA = 3
MHA_ERR_OOM = 4
MHA_ERR_TIMEOUT = 5
MHA_ERR_DEVICE = 6

MHA_F32 = 0
MHA_BF16 = 1

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KEY_PADDING = 2
MASK_CAUSAL_BOTTOM_RIGHT = 4

LIB_PATH = _build.LIB

_lock = threading.Lock()
_lib = None


ENCODER_PARAM_NAMES = ("Wq", "Wk", "Wv", "Wo", "bq", "bk", "bv", "bo", "ln1_gamma",
                       "ln1_beta", "W1", "b1", "W2", "b2", "ln2_gamma", "ln2_beta")


class EncoderParams(ctypes.Structure):
    """mha_encoder_params of include/mha.h (device pointers)."""
    _fields_ = [(n, ctypes.c_void_p) for n in ENCODER_PARAM_NAMES]


class MhaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def _declare(lib):
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.sdpa_forward.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp,
                                 i32, i32, vp]
    lib.sdpa_forward.restype = i32
    lib.sdpa_decode.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, i32, i32,
                                vp]
    lib.sdpa_decode.restype = i32
    lib.sdpa_forward_lse.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp,
                                     i32, vp]
    lib.sdpa_forward_lse.restype = i32
    lib.sdpa_backward_workspace_bytes.argtypes = [i32, i32, i32]
    lib.sdpa_backward_workspace_bytes.restype = ctypes.c_size_t
    lib.sdpa_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                  f32, i32, vp, i32, vp, ctypes.c_size_t, vp]
    lib.sdpa_backward.restype = i32
    lib.sdpa_forward_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.sdpa_forward_host_workspace_bytes.restype = ctypes.c_size_t
    lib.sdpa_forward_host.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, i32,
                                      i32, vp, ctypes.c_size_t, vp]
    lib.sdpa_forward_host.restype = i32
    lib.sinusoidal_pe.argtypes = [vp, i32, i32, i32, vp]
    lib.sinusoidal_pe.restype = i32
    lib.embed_pe_forward.argtypes = [vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, f32, i32, vp]
    lib.embed_pe_forward.restype = i32
    lib.sdpa_decode_splits.argtypes = [i32, i32, i32, i32]
    lib.sdpa_decode_splits.restype = i32
    i64 = ctypes.c_int64
    lib.sdpa_forward_float_mask.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32,
                                            vp, vp, i64, i64, i32, i32, vp]
    lib.sdpa_forward_float_mask.restype = i32
    lib.encoder_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32]
    lib.encoder_create.restype = i32
    lib.encoder_forward.argtypes = [vp, vp, ctypes.POINTER(EncoderParams), i32, i32, i32, vp,
                                    f32, vp, i32, vp]
    lib.encoder_forward.restype = i32
    lib.encoder_destroy.argtypes = [vp]
    lib.encoder_destroy.restype = i32
    lib.mha_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32]
    lib.mha_create.restype = i32
    lib.mha_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.mha_forward.restype = i32
    lib.mha_check.argtypes = [vp]
    lib.mha_check.restype = i32
    lib.mha_destroy.argtypes = [vp]
    lib.mha_destroy.restype = i32
    lib.mha_status_string.argtypes = [i32]
    lib.mha_status_string.restype = ctypes.c_char_p
    lib.mha_set_wait_limit_ms.argtypes = [i32]
    lib.mha_set_wait_limit_ms.restype = i32
    lib.mha_selftest_wait_timeout.argtypes = [i32, vp]
    lib.mha_selftest_wait_timeout.restype = i32
    return lib


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {LIB_PATH} is missing; build it with "
                    "transformer_head_scaled_03_gb300.build.build()")
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def status_string(status: int) -> str:
    return lib().mha_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != MHA_OK:
        raise MhaError(status, what)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return MHA_BF16
    if t == torch.float32:
        return MHA_F32
    raise TypeError(f"unsupported dtype {t}")


def _dev_ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _mask_strides(add_mask, B, H, Lq, Lk):
    """Batch and head strides (elements, 0 = broadcast) of a float32 mask
    broadcastable to [B, H, Lq, Lk] whose [Lq, Lk] rows are contiguous."""
    if add_mask.dtype != torch.float32 or not add_mask.is_cuda:
        raise ValueError("add_mask must be a float32 CUDA tensor")
    m = add_mask
    while m.dim() < 4:
        m = m.unsqueeze(0)
    if m.dim() != 4 or tuple(m.shape[2:]) != (Lq, Lk) or m.shape[0] not in (1, B) \
            or m.shape[1] not in (1, H):
        raise ValueError("add_mask must broadcast to [B, H, Lq, Lk]")
    if Lk > 1 and m.stride(3) != 1 or Lq > 1 and m.stride(2) != Lk:
        raise ValueError("add_mask rows must be contiguous")
    sb = m.stride(0) if m.shape[0] > 1 else 0
    sh = m.stride(1) if m.shape[1] > 1 else 0
    return sb, sh


def sdpa_forward(Q, K, V, scale: float | None = None, mask_kind: int = MASK_NONE,
                 key_lengths=None, out_dtype: torch.dtype | None = None, out=None,
                 stream=None, add_mask=None):
    """O = softmax(Q K^T * scale + mask) V for Q [B,H,Lq,d], K/V [B,H,Lk,d].

    ``add_mask``: optional float32 tensor broadcastable to [B,H,Lq,Lk], added
    to the scaled scores (-inf blocks a key)."""
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    if K.shape != (B, H, Lk, d) or V.shape != (B, H, Lk, d):
        raise ValueError("Q/K/V shapes disagree")
    if K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise ValueError("Q/K/V dtypes disagree")
    odt = out_dtype or Q.dtype
    if out is None:
        out = torch.empty((B, H, Lq, d), dtype=odt, device=Q.device)
    elif out.shape != (B, H, Lq, d) or out.dtype != odt:
        raise ValueError("out has the wrong shape or dtype")
    if key_lengths is not None and key_lengths.dtype != torch.int32:
        raise ValueError("key_lengths must be int32")
    if add_mask is not None:
        sb, sh = _mask_strides(add_mask, B, H, Lq, Lk)
        st = lib().sdpa_forward_float_mask(
            _dev_ptr(Q), _dev_ptr(K), _dev_ptr(V), _dev_ptr(out), B, H, Lq, Lk, d,
            float(scale or 0.0), int(mask_kind), _dev_ptr(key_lengths),
            ctypes.c_void_p(add_mask.data_ptr()), sb, sh, _dtype_code(Q.dtype),
            _dtype_code(odt), _stream(stream))
        _check(st, "sdpa_forward_float_mask")
        return out
    st = lib().sdpa_forward(_dev_ptr(Q), _dev_ptr(K), _dev_ptr(V), _dev_ptr(out), B, H, Lq, Lk,
                            d, float(scale or 0.0), int(mask_kind), _dev_ptr(key_lengths),
                            _dtype_code(Q.dtype), _dtype_code(odt), _stream(stream))
    _check(st, "sdpa_forward")
    return out


def sdpa_decode(Q, K_cache, V_cache, kv_lengths=None, causal: bool = True,
                scale: float | None = None, out_dtype: torch.dtype | None = None,
                num_splits: int = 0, out=None, stream=None):
    """Decode-shape attention: Q [B,H,Lq<=16,d] (the newest Lq positions)
    against caches K/V [B,H,Lk,d] holding kv_lengths[b] tokens (all Lk when
    None); bottom-right causal unless ``causal`` is False."""
    B, H, Lq, d = Q.shape
    Lk = K_cache.shape[2]
    if K_cache.shape != (B, H, Lk, d) or V_cache.shape != (B, H, Lk, d):
        raise ValueError("Q/cache shapes disagree")
    if K_cache.dtype != Q.dtype or V_cache.dtype != Q.dtype:
        raise ValueError("Q/cache dtypes disagree")
    odt = out_dtype or Q.dtype
    if out is None:
        out = torch.empty((B, H, Lq, d), dtype=odt, device=Q.device)
    elif out.shape != (B, H, Lq, d) or out.dtype != odt:
        raise ValueError("out has the wrong shape or dtype")
    mask = MASK_CAUSAL_BOTTOM_RIGHT if causal else MASK_NONE
    if kv_lengths is not None:
        if kv_lengths.dtype != torch.int32:
            raise ValueError("kv_lengths must be int32")
        mask |= MASK_KEY_PADDING
    st = lib().sdpa_decode(_dev_ptr(Q), _dev_ptr(K_cache), _dev_ptr(V_cache), _dev_ptr(out), B, H,
                           Lq, Lk, d, float(scale or 0.0), mask, _dev_ptr(kv_lengths),
                           _dtype_code(odt), int(num_splits), _stream(stream))
    _check(st, "sdpa_decode")
    return out


def decode_splits(B: int, H: int, Lk: int, d: int) -> int:
    """The split count sdpa_decode picks by default."""
    return int(lib().sdpa_decode_splits(B, H, Lk, d))


def sdpa_forward_lse(Q, K, V, scale: float | None = None, mask_kind: int = MASK_NONE,
                     key_lengths=None, out=None, lse=None, stream=None):
    """bf16 forward that also returns the base-2 row log-sum-exp [B,H,Lq]."""
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    if Q.dtype != torch.bfloat16 or K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise ValueError("bf16 Q/K/V required")
    if out is None:
        out = torch.empty_like(Q)
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=Q.device)
    st = lib().sdpa_forward_lse(_dev_ptr(Q), _dev_ptr(K), _dev_ptr(V), _dev_ptr(out),
                                _dev_ptr(lse), B, H, Lq, Lk, d, float(scale or 0.0),
                                int(mask_kind), _dev_ptr(key_lengths), _dtype_code(out.dtype),
                                _stream(stream))
    _check(st, "sdpa_forward_lse")
    return out, lse


def sdpa_backward(Q, K, V, O, dO, lse, scale: float | None = None, mask_kind: int = MASK_NONE,
                  key_lengths=None, grad_dtype: torch.dtype = torch.bfloat16, workspace=None,
                  stream=None):
    """(dQ fp32, dK, dV) of scaled dot-product attention for upstream dO."""
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    dQ = torch.empty((B, H, Lq, d), dtype=torch.float32, device=Q.device)
    dK = torch.empty((B, H, Lk, d), dtype=grad_dtype, device=Q.device)
    dV = torch.empty((B, H, Lk, d), dtype=grad_dtype, device=Q.device)
    need = int(lib().sdpa_backward_workspace_bytes(B, H, Lq))
    if workspace is None:
        workspace = torch.empty(max(16, (need + 15) // 16 * 16), dtype=torch.uint8,
                                device=Q.device)
    st = lib().sdpa_backward(_dev_ptr(Q), _dev_ptr(K), _dev_ptr(V), _dev_ptr(O), _dev_ptr(dO),
                             _dev_ptr(lse), _dev_ptr(dQ), _dev_ptr(dK), _dev_ptr(dV), B, H, Lq, Lk,
                             d, float(scale or 0.0), int(mask_kind), _dev_ptr(key_lengths),
                             _dtype_code(grad_dtype), _dev_ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "sdpa_backward")
    return dQ, dK, dV


def sinusoidal_pe(n_pos: int, d_model: int, first_pos: int = 0, out=None, stream=None,
                  device=None):
    """The positional-encoding table, fp32 [n_pos, d_model] on the device."""
    if out is None:
        out = torch.empty((n_pos, d_model), dtype=torch.float32,
                          device=device if device is not None else "cuda")
    elif out.shape != (n_pos, d_model) or out.dtype != torch.float32:
        raise ValueError("out has the wrong shape or dtype")
    _check(lib().sinusoidal_pe(_dev_ptr(out), int(first_pos), int(n_pos), int(d_model),
                               _stream(stream)), "sinusoidal_pe")
    return out


def embed_pe(ids, table, pe, pos_offset: int = 0, scale: float | None = None, out=None,
             stream=None):
    """x [B, L, D] = table[ids] * scale (default sqrt(D)) + pe[pos_offset + l]."""
    B, L = ids.shape
    vocab, D = table.shape
    if ids.dtype != torch.int32:
        raise ValueError("ids must be int32")
    if pe.dtype != torch.float32 or pe.dim() != 2 or pe.shape[1] != D:
        raise ValueError("pe must be float32 [rows, D]")
    if out is None:
        out = torch.empty((B, L, D), dtype=table.dtype, device=table.device)
    elif out.shape != (B, L, D) or out.dtype != table.dtype:
        raise ValueError("out has the wrong shape or dtype")
    st = lib().embed_pe_forward(_dev_ptr(ids), _dev_ptr(table), vocab, _dev_ptr(pe), pe.shape[0],
                                _dev_ptr(out), B, L, D, int(pos_offset), float(scale or 0.0),
                                _dtype_code(table.dtype), _stream(stream))
    _check(st, "embed_pe_forward")
    return out


class MhaHandle:
    """Owner of an ``mha_create`` handle (destroyed with ``close``)."""

    def __init__(self, d_model: int, dtype: torch.dtype, max_batch: int, max_lq: int,
                 max_lk: int):
        h = ctypes.c_void_p()
        _check(lib().mha_create(ctypes.byref(h), d_model, _dtype_code(dtype), max_batch, max_lq,
                                max_lk), "mha_create")
        self._h = h
        self.d_model, self.dtype = d_model, dtype

    @property
    def raw(self):
        if self._h is None:
            raise RuntimeError("handle destroyed")
        return self._h

    def close(self):
        if self._h is not None:
            _check(lib().mha_destroy(self._h), "mha_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mha_create(d_model: int, dtype: torch.dtype, max_batch: int, max_lq: int,
               max_lk: int) -> MhaHandle:
    return MhaHandle(d_model, dtype, max_batch, max_lq, max_lk)


def mha_forward(handle: MhaHandle, x_q, x_kv, Wq, Wk, Wv, Wo, h: int,
                mask_kind: int = MASK_NONE, key_lengths=None, out=None, stream=None):
    """out = Concat(head_1..head_h) Wo, head_i = Attention(x_q Wq_i, x_kv Wk_i, x_kv Wv_i)."""
    B, Lq, D = x_q.shape
    Lk = x_kv.shape[1]
    if x_kv.shape != (B, Lk, D):
        raise ValueError("x_kv shape")
    for W in (Wq, Wk, Wv, Wo):
        if W.shape != (D, D) or W.dtype != x_q.dtype:
            raise ValueError("weights must be [D, D] of the activations' dtype")
    if out is None:
        out = torch.empty((B, Lq, D), dtype=x_q.dtype, device=x_q.device)
    st = lib().mha_forward(handle.raw, _dev_ptr(x_q), _dev_ptr(x_kv), _dev_ptr(Wq),
                           _dev_ptr(Wk), _dev_ptr(Wv), _dev_ptr(Wo), B, Lq, Lk, int(h),
                           int(mask_kind), _dev_ptr(key_lengths), _dev_ptr(out),
                           _stream(stream))
    _check(st, "mha_forward")
    return out


class EncoderLayer:
    """One post-norm encoder layer on the library (encoder_create /
    encoder_forward / encoder_destroy).  ``params`` maps the names in
    ENCODER_PARAM_NAMES to device tensors of the layer's dtype."""

    def __init__(self, d_model: int, heads: int, d_ff: int, dtype: torch.dtype,
                 max_batch: int, max_len: int):
        h = ctypes.c_void_p()
        _check(lib().encoder_create(ctypes.byref(h), d_model, heads, d_ff, _dtype_code(dtype),
                                    max_batch, max_len), "encoder_create")
        self._h = h
        self.d_model, self.heads, self.d_ff, self.dtype = d_model, heads, d_ff, dtype

    def forward(self, x, params: dict, mask_kind: int = MASK_NONE, key_lengths=None,
                ln_eps: float = 1e-5, out=None, stream=None, out_dtype=None):
        """``out_dtype``: the layer's dtype (default), or torch.float32 for a
        bf16 layer to keep the final LayerNorm's output unrounded."""
        if self._h is None:
            raise RuntimeError("encoder destroyed")
        B, L, D = x.shape
        if D != self.d_model or x.dtype != self.dtype:
            raise ValueError("x does not match the layer")
        shapes = {"W1": (D, self.d_ff), "b1": (self.d_ff,), "W2": (self.d_ff, D)}
        for n in ENCODER_PARAM_NAMES:
            t = params[n]
            want = shapes.get(n, (D, D) if n.startswith("W") else (D,))
            if tuple(t.shape) != want or t.dtype != self.dtype:
                raise ValueError(f"parameter {n} must be {want} {self.dtype}")
        p = EncoderParams(*[_dev_ptr(params[n]) for n in ENCODER_PARAM_NAMES])
        odt = self.dtype if out_dtype is None else out_dtype
        if out is None:
            out = torch.empty(x.shape, dtype=odt, device=x.device)
        if out.dtype != odt or tuple(out.shape) != tuple(x.shape):
            raise ValueError("out does not match the output dtype and shape")
        st = lib().encoder_forward(self._h, _dev_ptr(x), ctypes.byref(p), B, L, int(mask_kind),
                                   _dev_ptr(key_lengths), float(ln_eps), _dev_ptr(out),
                                   _dtype_code(odt), _stream(stream))
        _check(st, "encoder_forward")
        return out

    def close(self):
        if self._h is not None:
            _check(lib().encoder_destroy(self._h), "encoder_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mha_check(handle: MhaHandle | None = None) -> int:
    """Synchronise and return (then clear) the device error status code."""
    return int(lib().mha_check(handle.raw if handle is not None else None))


def mha_destroy(handle: MhaHandle):
    handle.close()


def selftest_wait_timeout(limit_ms: int = 100, stream=None):
    """Launch the bounded-wait self-test (see include/mha.h); mha_check() then
    reports MHA_ERR_TIMEOUT."""
    _check(lib().mha_selftest_wait_timeout(int(limit_ms), _stream(stream)),
           "mha_selftest_wait_timeout")


def set_wait_limit_ms(ms: int) -> int:
    return int(lib().mha_set_wait_limit_ms(int(ms)))


def sdpa_forward_host(Qh, Kh, Vh, scale=None, mask_kind=MASK_NONE, lengths_h=None,
                      out_dtype=None, device="cuda", bufs=None, stream=None):
    """End-to-end call from host (pinned) tensors through the library's
    sdpa_forward_host: copies in, attention and copies out overlap chunk by
    chunk on the device.  Returns the pinned output; it is complete once
    ``stream`` (the current stream by default) has been synchronised.

    ``bufs`` (a dict) keeps the device workspace and the pinned output
    between calls."""
    bufs = {} if bufs is None else bufs
    B, H, Lq, d = Qh.shape
    Lk = Kh.shape[2]
    odt = out_dtype or Qh.dtype
    need = int(lib().sdpa_forward_host_workspace_bytes(B, H, Lq, Lk, d, _dtype_code(Qh.dtype),
                                                       _dtype_code(odt)))
    ws = bufs.get("ws")
    if ws is None or ws.numel() < need:
        ws = bufs["ws"] = torch.empty(max(256, need), dtype=torch.uint8, device=device)
    Oh = bufs.get("Oh")
    if Oh is None or Oh.shape != Qh.shape or Oh.dtype != odt:
        Oh = bufs["Oh"] = torch.empty(Qh.shape, dtype=odt, pin_memory=True)
    lp = ctypes.c_void_p(lengths_h.data_ptr()) if lengths_h is not None else None
    st = lib().sdpa_forward_host(ctypes.c_void_p(Qh.data_ptr()), ctypes.c_void_p(Kh.data_ptr()),
                                 ctypes.c_void_p(Vh.data_ptr()), ctypes.c_void_p(Oh.data_ptr()),
                                 B, H, Lq, Lk, d, float(scale or 0.0), int(mask_kind), lp,
                                 _dtype_code(Qh.dtype), _dtype_code(odt), _dev_ptr(ws),
                                 ws.numel(), _stream(stream))
    _check(st, "sdpa_forward_host")
    return Oh
