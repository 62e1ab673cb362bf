"""Workspaces whose contents no call may depend on, filled with NaN bytes.

The workspace contract is: zero-filled once before first use, then every call leaves
it ready for the next.  What must be zero is the attention workspace's counter head
(one merge counter per (sequence, KV head) pair and 64 scheduler words); everything
after it -- the split partials of the attention kernels, the SnapKV partial
statistics, scores and pooled rows, the Top-K score rows and the acceptance records --
is written before it is read within a call.  Here every such byte starts as 0xFF (a
NaN in fp32, and in bf16), so a merge that reads a partial no CTA of this call wrote,
or a reduction over an unwritten record, shows up as a NaN or a wrong value against
the CPU oracle.  The shapes split sequences over many CTAs (partials and merges on
every pair)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_self_gb300 import binding as mb
from long_context_self_gb300 import synth
from parity_util import (bf16_out_to_f64, check_accept, check_attention, check_topk, check_topk_attn,
                         oracle_accept, to_u16)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
# The attention workspace's head that must start at zero: 65536 pair counters and 64
# scheduler words, int32 (the library's fixed counter region).
ATTN_COUNTER_BYTES = (65536 + 64) * 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_self_gb300 import build
    build.build()
    mb.lib()
    yield
    assert mb.magicdec_device_error() == 0


def poisoned(nbytes, zero_head=0):
    ws = torch.full((max(int(nbytes), 256),), 0xFF, dtype=torch.uint8, device=DEV)
    if zero_head:
        ws[:zero_head].zero_()
    return ws


def rand_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("H_q,H_kv,d,n_q", [(32, 8, 128, 4), (32, 8, 128, 5), (40, 8, 128, 5), (16, 2, 64, 4)])
def test_verify_with_poisoned_partials(H_q, H_kv, d, n_q):
    """Every verification kernel (all-heads at d = 128 / 8 KV heads / 16 and 20 rows;
    per-pair otherwise)."""
    B, L_cap = 4, 5000
    lens = np.array([5000, 3, 4100, 2500], np.int32)
    q, k, v = rand_bf16((B, n_q, H_q, d), 61), rand_bf16((B, L_cap, H_kv, d), 62), rand_bf16((B, L_cap, H_kv, d), 63)
    shape = mb.kv_shape(B, H_q, H_kv, d, L_cap)
    ws = poisoned(mb.magicdec_attn_workspace_size(shape, n_q), ATTN_COUNTER_BYTES)
    sl = torch.from_numpy(lens).to(DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    ref = oracle.verify_attn(to_u16(q), to_u16(k), to_u16(v), lens, n_q)
    for _ in range(2):          # the second call runs over the first call's leftovers
        out = mb.magicdec_verify_attn(qd, kd, vd, sl, ws=ws)
        torch.cuda.synchronize()
        check_attention(bf16_out_to_f64(out), ref, "verify over a poisoned workspace")
    assert torch.all(ws[:ATTN_COUNTER_BYTES] == 0), "counter head not left zero"


def test_draft_with_poisoned_partials():
    B, H_q, H_kv, d, cap = 3, 32, 8, 128, 4096
    lens = np.array([4096, 700, 1], np.int32)
    q = rand_bf16((B, 1, H_q, d), 71)
    kc, vc = rand_bf16((B, H_kv, cap, d), 72), rand_bf16((B, H_kv, cap, d), 73)
    shape = mb.kv_shape(B, H_q, H_kv, d, cap)
    ws = poisoned(mb.magicdec_attn_workspace_size(shape, 1), ATTN_COUNTER_BYTES)
    out = mb.magicdec_draft_attn(q.to(DEV), kc.to(DEV), vc.to(DEV), torch.from_numpy(lens).to(DEV), ws=ws)
    torch.cuda.synchronize()
    check_attention(bf16_out_to_f64(out), oracle.draft_attn(to_u16(q), to_u16(kc), to_u16(vc), lens),
                    "draft over a poisoned workspace")


def test_snapkv_select_with_poisoned_workspace():
    B, H_q, H_kv, d, L_cap, w, pool, budget = 2, 32, 8, 128, 3000, 32, 7, 512
    wl = synth.Workload("case", B=B, H_q=H_q, H_kv=H_kv, d=d, L=L_cap, gamma=1, V=8, snap_window=w,
                        snap_pool=pool, snap_budget=budget, heavy_frac=0.005, seed=21)
    k, _, dirs = synth.kv_cache(wl, "cpu")
    q_win = synth.window_queries(wl, "cpu", heavy_dirs=dirs)
    sl = np.array([3000, 2222], np.int32)
    ws = poisoned(mb.magicdec_snapkv_workspace_size(mb.kv_shape(B, H_q, H_kv, d, L_cap), w))
    idx, n_sel = mb.magicdec_snapkv_select(q_win.to(DEV), k.to(DEV), torch.from_numpy(sl).to(DEV), w, pool, budget,
                                           ws=ws)
    torch.cuda.synchronize()
    idx_o, n_sel_o, pooled = oracle.snapkv_select(to_u16(q_win), to_u16(k), sl, pool, budget)
    check_topk(idx.cpu().numpy(), n_sel.cpu().numpy(), idx_o, n_sel_o, pooled, sl, w, budget)


def test_topk_draft_with_poisoned_workspace():
    B, H_q, H_kv, d, L_cap, top_k = 2, 32, 8, 128, 3000, 256
    q, k, v = rand_bf16((B, 1, H_q, d), 81), rand_bf16((B, L_cap, H_kv, d), 82), rand_bf16((B, L_cap, H_kv, d), 83)
    lens = np.array([3000, 1000], np.int32)
    ws = poisoned(mb.magicdec_topk_attn_workspace_size(mb.kv_shape(B, H_q, H_kv, d, L_cap)))
    idx = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_topk_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(lens).to(DEV), top_k,
                                      idx=idx, ws=ws)
    torch.cuda.synchronize()
    out_o, idx_o, scores = oracle.topk_attn(to_u16(q), to_u16(k), to_u16(v), lens, top_k, want_scores=True)
    check_topk_attn(bf16_out_to_f64(out), idx.cpu().numpy(), out_o, idx_o, scores, lens, top_k,
                    "topk over a poisoned workspace", qkv=(to_u16(q), to_u16(k), to_u16(v)))


@pytest.mark.parametrize("greedy", [False, True])
def test_spec_accept_with_poisoned_workspace(greedy):
    w = synth.WORKLOADS["llama8b_b128_l32k"]
    B = 16
    target, draft, tok, u_acc, u_res = synth.logits(w, "cpu", B=B, seed=37)
    ws = poisoned(mb.magicdec_spec_accept_workspace_size(B, w.gamma, w.V))
    got = mb.magicdec_spec_accept(target.to(DEV), draft.to(DEV), tok.to(DEV), u_acc.to(DEV), u_res.to(DEV), greedy,
                                  ws=ws)
    torch.cuda.synchronize()
    t, d, x, ua, ur = (a.numpy() for a in (target, draft, tok, u_acc, u_res))
    check_accept(tuple(a.cpu().numpy() for a in got), oracle_accept(t, d, x, ua, ur, greedy), "accept, poisoned",
                 inputs=(t, d, ur), greedy=greedy)
