"""magicdec_verify_attn_noalloc -- verification attention for callers that cannot
allocate device memory (a plug-in handed only its input and output buffers, an engine
with a fixed memory plan, a process whose device memory another allocator owns).  Its
scratch is an array inside the library instead of a caller workspace.

Checked through the C ABI against magicdec_verify_attn on the same inputs, within the
attention tolerance the parity tests use, on two calls in a row (different inputs, so
the second call also shows the shared scratch was left ready), and against the CPU
oracle.  Every verification kernel runs through it: the all-heads kernels (d = 128,
8 KV heads, 16 and 20 query rows per KV head) and the per-pair kernel (40 query heads
over 8 KV heads with 5 speculated rows, and d = 64), which splits long pairs across CTAs and merges them through
the array's counters.  Collected last so that a stop at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import bf16_out_to_f64, check_attention, to_u16

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _inputs(seed, B, H_q, H_kv, d, L_cap, n_q):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, n_q, H_q, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    return q, k, v


# (H_q, H_kv, d, n_q): all-heads kernels at 16 and 20 rows per KV head; per-pair kernel at
# 25 rows per KV head; per-pair at d = 64
SHAPES = [(32, 8, 128, 4), (32, 8, 128, 5), (40, 8, 128, 5), (32, 8, 64, 4)]


@pytest.mark.parametrize("H_q,H_kv,d,n_q", SHAPES)
def test_noalloc_verify_matches_workspace_entry_point_on_two_calls(H_q, H_kv, d, n_q):
    from long_context_self_gb300 import binding as mb
    from long_context_self_gb300 import build
    build.build()
    B = 6
    # ragged lengths: empty, one row, a block shorter than n_q, full; the 5000-row case
    # splits its long pairs over several CTAs, whose partials merge through the shared array
    cases = [(101, 2500, [2500, 1, 0, 64, 1777, 2049]), (102, 2500, [300, 2500, 2499, 65, 128, 4]),
             (103, 5000, [5000, 4500, 17, 4096, 0, 4999])]
    for seed, L_cap, lens in cases:
        q, k, v = _inputs(seed, B, H_q, H_kv, d, L_cap, n_q)
        qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
        sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
        ref = mb.magicdec_verify_attn(qd, kd, vd, sl)
        got = mb.magicdec_verify_attn_noalloc(qd, kd, vd, sl)
        torch.cuda.synchronize()
        check_attention(bf16_out_to_f64(got), bf16_out_to_f64(ref), "verify_attn_noalloc vs verify_attn")
        ora = oracle.verify_attn(to_u16(q), to_u16(k), to_u16(v), np.array(lens, np.int32), n_q)
        check_attention(bf16_out_to_f64(got), ora, "verify_attn_noalloc vs oracle")
    assert mb.magicdec_device_error() == 0
