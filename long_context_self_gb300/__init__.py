"""GB300 (sm_103a) hot path for MagicDec-style long-context self-speculative decoding.

The compute lives in ``libmagicdec.so`` (CUDA kernels behind the C ABI of
``include/magicdec.h``); :mod:`long_context_self_gb300.binding` is the thin
ctypes binding with the same entry-point names, and
:mod:`long_context_self_gb300.synth` draws the seeded synthetic workloads.
Importing the package does not load the library; the first call does, and
raises if the library was not built.
"""
from .binding import (  # noqa: F401
    EXPORTED,
    KVShape,
    MagicdecError,
    kv_shape,
    lib,
    magicdec_attn_workspace_size,
    magicdec_device_error,
    magicdec_draft_attn,
    magicdec_gather_kv,
    magicdec_snapkv_select,
    magicdec_snapkv_workspace_size,
    magicdec_spec_accept,
    magicdec_spec_accept_workspace_size,
    magicdec_streaming_select,
    magicdec_verify_attn,
    magicdec_verify_attn_noalloc,
    status_string,
)
