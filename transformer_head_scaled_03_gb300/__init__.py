"""GB300 (sm_103a) multi-head scaled dot-product attention.

The compute lives in ``libmha_gb300.so`` (C ABI in ``include/mha.h``):
a fused tcgen05/TMEM attention kernel for bf16, tcgen05 projection GEMMs
whose store layouts do the head split and the concat, and fp32 CUDA-core
kernels.  This package is the thin Python binding over that ABI
(``sdpa_forward``, ``mha_create``, ``mha_forward``, ``mha_check``,
``mha_destroy``), the in-tree build (``build``) and the seeded input
generators (``inputs``).  Attribute access loads the binding lazily, so
importing the package (e.g. for ``inputs``) needs neither torch nor a GPU.
"""
_BINDING_NAMES = {
    "sdpa_forward", "sdpa_forward_host", "sdpa_decode", "decode_splits", "sinusoidal_pe",
    "sdpa_forward_lse", "sdpa_backward",
    "embed_pe",
    "MASK_CAUSAL_BOTTOM_RIGHT", "mha_create", "mha_forward", "mha_check",
    "mha_destroy", "MhaHandle", "MhaError", "EncoderLayer", "EncoderParams",
    "ENCODER_PARAM_NAMES", "set_wait_limit_ms", "selftest_wait_timeout", "status_string", "lib",
    "MASK_NONE", "MASK_CAUSAL", "MASK_KEY_PADDING", "MHA_OK", "MHA_ERR_INVALID_ARG",
    "MHA_ERR_UNSUPPORTED", "MHA_ERR_CUDA", "MHA_ERR_OOM", "MHA_ERR_TIMEOUT",
    "MHA_ERR_DEVICE", "MHA_F32", "MHA_BF16", "LIB_PATH",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)
