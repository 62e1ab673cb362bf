"""The C-ABI library loads, exports every entry point include/magicdec.h declares, and
rejects bad arguments on the host before anything is enqueued.  CPU only: no call here
reaches a kernel (every call fails validation first) and no GPU is needed."""
import ctypes
import os
import re

import pytest

from long_context_self_gb300 import binding
from long_context_self_gb300 import build as lbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "magicdec.h")


@pytest.fixture(scope="module")
def lib():
    lbuild.build()
    return binding.lib()


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(magicdec_[a-z_]+)\s*\(", text)))


def test_header_declares_the_path(lib):
    names = declared_entry_points()
    for required in ("magicdec_streaming_select", "magicdec_snapkv_select", "magicdec_gather_kv",
                     "magicdec_draft_attn", "magicdec_verify_attn", "magicdec_spec_accept"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name
        assert name in binding.EXPORTED, f"binding lacks {name}"


def test_library_exports_only_the_abi(lib):
    out = os.popen(f"nm -D --defined-only {binding._LIB_PATH}").read()
    syms = {line.split()[-1] for line in out.splitlines() if " T " in line}
    extra = {s for s in syms if not s.startswith("magicdec_")}
    assert not extra, f"unexpected exported text symbols: {sorted(extra)[:10]}"


def test_status_strings(lib):
    assert binding.status_string(0) == "ok"
    assert "null" in binding.status_string(-1)
    assert "workspace" in binding.status_string(-4)


P = ctypes.c_void_p
FAKE = P(0x10000)           # a 16-byte aligned non-null address never dereferenced: validation fails first
MISALIGNED = P(0x10008)


def shape(B=2, H_q=8, H_kv=2, d=128, L=64):
    return binding.KVShape(B, H_q, H_kv, d, L)


def test_null_and_shape_errors_are_reported_before_launch(lib):
    NULL = P(0)
    assert lib.magicdec_verify_attn(shape(), 4, NULL, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, NULL) == -1
    assert lib.magicdec_verify_attn(shape(d=96), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, NULL) == -2
    assert lib.magicdec_verify_attn(shape(H_q=6, H_kv=4), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, NULL) == -2
    assert lib.magicdec_verify_attn(shape(), 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, NULL) == -2
    # more than 32 query rows per KV head: a valid shape with no kernel
    assert lib.magicdec_verify_attn(shape(H_q=16, H_kv=2), 5, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, NULL) == -5
    assert lib.magicdec_verify_attn(shape(), 4, MISALIGNED, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, NULL) == -3
    assert lib.magicdec_draft_attn(shape(), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, NULL) == -4
    assert lib.magicdec_gather_kv(shape(), FAKE, FAKE, FAKE, 10, 5, FAKE, FAKE, NULL) == -2
    assert lib.magicdec_gather_kv(shape(), FAKE, FAKE, NULL, 4, 5, FAKE, FAKE, NULL) == -1
    assert lib.magicdec_streaming_select(FAKE, 0, 8, 16, 496, FAKE, FAKE, NULL) == -2
    assert lib.magicdec_streaming_select(FAKE, 4, 8, 0, 0, FAKE, FAKE, NULL) == -2
    assert lib.magicdec_streaming_select(NULL, 4, 8, 16, 496, FAKE, FAKE, NULL) == -1
    assert lib.magicdec_streaming_select(FAKE, 4, 8, 2**31 - 1, 1, FAKE, FAKE, NULL) == -2   # width past INT_MAX
    # one block row per (KV head, sequence): more than 65535 of either has no launch shape
    assert lib.magicdec_streaming_select(FAKE, 70000, 8, 16, 496, FAKE, FAKE, NULL) == -5
    assert lib.magicdec_streaming_select(FAKE, 4, 70000, 16, 496, FAKE, FAKE, NULL) == -5
    # a width of exactly INT_MAX passes the shape check (its grid and indices are 64-bit); the
    # batch bound still refuses before anything is launched
    assert lib.magicdec_streaming_select(FAKE, 70000, 8, 2**31 - 2, 1, FAKE, FAKE, NULL) == -5
    assert lib.magicdec_device_error(NULL) == -1
    # the no-allocation verification entry point validates like the workspace one
    assert lib.magicdec_verify_attn_noalloc(shape(), 4, NULL, FAKE, FAKE, FAKE, FAKE, NULL) == -1
    assert lib.magicdec_verify_attn_noalloc(shape(d=96), 4, FAKE, FAKE, FAKE, FAKE, FAKE, NULL) == -2
    assert lib.magicdec_verify_attn_noalloc(shape(), 0, FAKE, FAKE, FAKE, FAKE, FAKE, NULL) == -2
    assert lib.magicdec_verify_attn_noalloc(shape(H_q=16, H_kv=2), 5, FAKE, FAKE, FAKE, FAKE, FAKE, NULL) == -5
    assert lib.magicdec_verify_attn_noalloc(shape(), 4, FAKE, FAKE, MISALIGNED, FAKE, FAKE, NULL) == -3
    assert lib.magicdec_snapkv_select(shape(), FAKE, FAKE, FAKE, 32, 7, 16, FAKE, FAKE, FAKE, 1 << 40, NULL) == -2
    assert lib.magicdec_snapkv_select(shape(), FAKE, FAKE, FAKE, 32, 6, 64, FAKE, FAKE, FAKE, 1 << 40, NULL) == -2
    assert lib.magicdec_snapkv_select(shape(), FAKE, FAKE, FAKE, 32, 7, 64, FAKE, FAKE, FAKE, 16, NULL) == -4
    assert lib.magicdec_snapkv_select(shape(), FAKE, FAKE, FAKE, 32, 11, 64, FAKE, FAKE, FAKE, 1 << 40, NULL) == -5
    assert lib.magicdec_snapkv_select_budgets(shape(), FAKE, FAKE, FAKE, 32, 7, NULL, 64, FAKE, FAKE, FAKE, 1 << 40,
                                              NULL) == -1
    assert lib.magicdec_snapkv_select_budgets(shape(), FAKE, FAKE, FAKE, 32, 7, FAKE, 16, FAKE, FAKE, FAKE, 1 << 40,
                                              NULL) == -2
    assert lib.magicdec_spec_accept(4, 3, 100, FAKE, NULL, FAKE, FAKE, FAKE, 0, FAKE, FAKE, NULL, FAKE,
                                    1 << 30, NULL) == -1
    assert lib.magicdec_spec_accept(0, 3, 100, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, NULL, FAKE,
                                    1 << 30, NULL) == -2
    assert lib.magicdec_spec_accept(4, 3, 100, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, NULL, FAKE,
                                    8, NULL) == -4
    big = 1 << 40
    assert lib.magicdec_pq_encode(shape(), FAKE, 16, 256, NULL, FAKE, NULL) == -1
    assert lib.magicdec_pq_encode(shape(), FAKE, 8, 256, FAKE, FAKE, NULL) == -2        # M must be d/8
    assert lib.magicdec_pq_encode(shape(), FAKE, 16, 257, FAKE, FAKE, NULL) == -2
    assert lib.magicdec_pq_update(shape(), FAKE, NULL, 16, 256, FAKE, FAKE, NULL) == -1
    assert lib.magicdec_pq_draft_attn(shape(), FAKE, FAKE, FAKE, FAKE, 16, 256, FAKE, FAKE, 0, FAKE, NULL, FAKE,
                                      big, NULL) == -2
    assert lib.magicdec_pq_draft_attn(shape(), FAKE, FAKE, FAKE, FAKE, 16, 256, FAKE, FAKE, 64, FAKE, NULL, FAKE,
                                      64, NULL) == -4
    assert lib.magicdec_pq_draft_attn(shape(), MISALIGNED, FAKE, FAKE, FAKE, 16, 256, FAKE, FAKE, 64, FAKE, NULL,
                                      FAKE, big, NULL) == -3
    I32 = P(0x20000)
    assert lib.magicdec_draft_cache_update(shape(), FAKE, FAKE, I32, I32, I32, I32, NULL, 0, 64, FAKE, FAKE, I32,
                                           NULL) == -1
    assert lib.magicdec_draft_cache_update(shape(), FAKE, FAKE, I32, I32, I32, I32, NULL, 80, 64, FAKE, FAKE, I32,
                                           NULL) == -2
    assert lib.magicdec_draft_cache_update(shape(), FAKE, FAKE, I32, I32, I32, I32, NULL, -1, 64, FAKE, FAKE, I32,
                                           NULL) == -2
    assert lib.magicdec_draft_cache_update(shape(), FAKE, FAKE, I32, I32, I32, I32, NULL, 16, 64, MISALIGNED, FAKE,
                                           I32, NULL) == -3
    assert lib.magicdec_step_lengths(4, 3, 100, NULL, NULL, I32, I32, NULL) == -1
    assert lib.magicdec_step_lengths(4, 3, 100, I32, NULL, I32, NULL, NULL) == -1
    assert lib.magicdec_step_lengths(0, 3, 100, I32, NULL, I32, I32, NULL) == -2
    assert lib.magicdec_step_lengths(4, -1, 100, I32, NULL, I32, I32, NULL) == -2
    assert lib.magicdec_step_lengths(4, 3, 0, I32, NULL, I32, I32, NULL) == -2
    assert lib.magicdec_topk_draft_attn(shape(), NULL, FAKE, FAKE, FAKE, 16, FAKE, NULL, FAKE, big, NULL) == -1
    assert lib.magicdec_topk_draft_attn(shape(), FAKE, FAKE, FAKE, FAKE, 0, FAKE, NULL, FAKE, big, NULL) == -2
    assert lib.magicdec_topk_draft_attn(shape(d=96), FAKE, FAKE, FAKE, FAKE, 16, FAKE, NULL, FAKE, big, NULL) == -2
    assert lib.magicdec_topk_draft_attn(shape(), FAKE, MISALIGNED, FAKE, FAKE, 16, FAKE, NULL, FAKE, big, NULL) == -3
    assert lib.magicdec_topk_draft_attn(shape(), FAKE, FAKE, FAKE, FAKE, 16, FAKE, NULL, FAKE, 64, NULL) == -4
    # more than 8 query heads per KV head, or a budget past 8192: valid shapes with no kernel
    assert lib.magicdec_topk_draft_attn(shape(H_q=32, H_kv=2), FAKE, FAKE, FAKE, FAKE, 16, FAKE, NULL, FAKE, big,
                                        NULL) == -5
    assert lib.magicdec_topk_draft_attn(shape(), FAKE, FAKE, FAKE, FAKE, 8193, FAKE, NULL, FAKE, big, NULL) == -5


def test_workspace_sizes_are_positive_and_monotone(lib):
    a = lib.magicdec_snapkv_workspace_size(shape(L=1000), 32)
    b = lib.magicdec_snapkv_workspace_size(shape(L=4000), 32)
    assert 0 < a < b
    assert lib.magicdec_snapkv_workspace_size(shape(d=80), 32) == 0
    assert lib.magicdec_topk_attn_workspace_size(shape(B=2, H_q=8, L=61)) == 2 * 8 * 64 * 4
    assert lib.magicdec_topk_attn_workspace_size(shape(d=80)) == 0
    s1 = lib.magicdec_spec_accept_workspace_size(4, 3, 128256)
    s2 = lib.magicdec_spec_accept_workspace_size(8, 3, 128256)
    assert 0 < s1 < s2


def test_binding_raises_without_cuda_tensors(lib):
    import torch
    with pytest.raises((ValueError, TypeError)):
        binding.magicdec_streaming_select(torch.zeros(4, dtype=torch.int32), 8, 16, 496)


def test_binding_refuses_mismatched_shapes_before_any_launch(lib):
    """The binding checks every tensor's shape against the others (the kernels would otherwise
    index out of bounds); the check runs before the library is called, so it needs no GPU data."""
    import torch

    # shapes are checked after dtype/device; on a CPU-only host the device check raises first,
    # so exercise the shape helper directly with a stand-in that passes the device check
    t = torch.zeros(3, dtype=torch.int32)
    orig = binding._need
    try:
        binding._need = lambda *a, **k: None
        with pytest.raises(ValueError, match="must have shape"):
            binding._need_shape(t, "seq_len", torch.int32, None, (4,))
        binding._need_shape(t, "seq_len", torch.int32, None, (3,))
    finally:
        binding._need = orig
