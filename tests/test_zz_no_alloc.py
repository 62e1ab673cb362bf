"""magicdec_verify_attn_noalloc -- verification attention for callers that cannot
allocate device memory (a plug-in handed only its input and output buffers, an engine
with a fixed memory plan, a process whose device memory another allocator owns).  Its
scratch is an array inside the library instead of a caller workspace.

Checked through the C ABI against magicdec_verify_attn on the same inputs, within the
attention tolerance the parity tests use, on two calls in a row (different inputs, so
the second call also shows the shared scratch was left ready).  Collected last so that
a stop at the first failure has already run every other test."""
import pytest
import torch

from parity_util import bf16_out_to_f64, check_attention

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _inputs(seed, B, H_q, H_kv, d, L_cap, n_q):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, n_q, H_q, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    return q.to(DEV), k.to(DEV), v.to(DEV)


def test_noalloc_verify_matches_workspace_entry_point_on_two_calls():
    from long_context_self_gb300 import binding as mb
    from long_context_self_gb300 import build
    build.build()
    B, H_q, H_kv, d, n_q = 6, 32, 8, 128, 4
    # the third case has pairs of >= 64 tiles (dynamic tails)
    cases = [(101, 2500, [2500, 1, 0, 64, 1777, 2049]), (102, 2500, [300, 2500, 2499, 65, 128, 4]),
             (103, 5000, [5000, 4500, 17, 4096, 0, 4999])]
    for seed, L_cap, lens in cases:
        q, k, v = _inputs(seed, B, H_q, H_kv, d, L_cap, n_q)
        sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
        ref = mb.magicdec_verify_attn(q, k, v, sl)
        got = mb.magicdec_verify_attn_noalloc(q, k, v, sl)
        torch.cuda.synchronize()
        check_attention(bf16_out_to_f64(got), bf16_out_to_f64(ref), "verify_attn_noalloc")
    assert mb.magicdec_device_error() == 0
