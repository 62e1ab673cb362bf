"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

Each workload runs the whole call at full size on the GPU (B up to 128, L up to
100000, V up to 152064); the oracle recomputes sampled outputs one (sequence, KV head)
pair or one sequence at a time from host copies of exactly the bytes the GPU read:
  * verification attention: every query row of sampled pairs;
  * StreamingLLM selection + gather + draft attention: sampled sequences;
  * SnapKV selection: sampled pairs (band rule at the k-th pooled score);
  * Top-K attention draft: every query head of sampled sequences (band rule at the
    top_k-th score);
  * draft-cache update: the StreamingLLM ring of sampled sequences, byte for byte;
  * PQCache-style selection: the encode of sampled sequences (margin rule) and PQ draft
    attention with host-drawn codes (band rule);
  * speculative accept: every sequence of the batch (sampling mode) or a sample (greedy).
"""
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_self_gb300 import build
    build.build()
    mb.lib()
    yield
    torch.cuda.empty_cache()
    assert mb.magicdec_device_error() == 0


def sample_pairs(w, n, seed):
    rng = np.random.default_rng(seed)
    bs = rng.choice(w.B, size=min(n, w.B), replace=False)
    return [(int(b), int(rng.integers(w.H_kv))) for b in bs]


def check_verify_pairs(w, q, k, v, sl, out, pairs):
    G = w.G
    for b, h in pairs:
        L = int(sl[b])
        qo = to_u16(q[b:b + 1, :, h * G:(h + 1) * G])
        ko = to_u16(k[b:b + 1, :L, h:h + 1])
        vo = to_u16(v[b:b + 1, :L, h:h + 1])
        ref = oracle.verify_attn(qo, ko, vo, np.array([L], np.int32), w.n_q)
        got = bf16_out_to_f64(out[b:b + 1, :, h * G:(h + 1) * G])
        check_attention(got, ref, f"{w.name} verify b={b} h={h}")


@pytest.mark.parametrize("name", ["llama8b_b32_l32k", "llama8b_b64_l32k_snapkv", "llama8b_b128_l32k",
                                  "qwen32b_b16_l100k"])
def test_fullsize_verify_attn_sampled(name):
    w = synth.WORKLOADS[name]
    k, v, _ = synth.kv_cache(w, DEV)
    q = synth.queries(w, w.n_q, DEV, seed=w.seed * 7 + 2)
    sl = torch.full((w.B,), w.L, dtype=torch.int32, device=DEV)
    out = mb.magicdec_verify_attn(q, k, v, sl)
    torch.cuda.synchronize()
    check_verify_pairs(w, q, k, v, sl.cpu().numpy(), out, sample_pairs(w, 3, w.seed))
    del k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["llama8b_b32_l32k", "llama8b_b128_l32k"])
def test_fullsize_streaming_draft_sampled(name):
    w = synth.WORKLOADS[name]
    k, v, _ = synth.kv_cache(w, DEV)
    qd = synth.queries(w, 1, DEV, seed=w.seed * 7 + 1)
    sl = torch.full((w.B,), w.L, dtype=torch.int32, device=DEV)
    idx, n_sel = mb.magicdec_streaming_select(sl, w.H_kv, w.n_sink, w.n_recent)
    kc, vc = mb.magicdec_gather_kv(k, v, idx, w.stream_budget)
    out = mb.magicdec_draft_attn(qd, kc, vc, n_sel)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w.seed + 5)
    for b in rng.choice(w.B, size=3, replace=False):
        b = int(b)
        L = int(sl[b])
        idx_o, n_sel_o = oracle.streaming_select(np.array([L], np.int32), w.H_kv, w.n_sink, w.n_recent)
        assert np.array_equal(idx[b:b + 1].cpu().numpy(), idx_o)
        assert int(n_sel[b]) == int(n_sel_o[0])
        # the gather reads only the selected rows: rebuild them on the host from the same cache bytes
        kc_o, vc_o = oracle.gather_kv(to_u16(k[b:b + 1]), to_u16(v[b:b + 1]), idx_o, w.stream_budget)
        assert np.array_equal(to_u16(kc[b:b + 1]), kc_o)
        assert np.array_equal(to_u16(vc[b:b + 1]), vc_o)
        ref = oracle.draft_attn(to_u16(qd[b:b + 1]), kc_o, vc_o, n_sel_o)
        check_attention(bf16_out_to_f64(out[b:b + 1]), ref, f"{name} draft b={b}")
    del k, v, kc, vc
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["llama8b_b64_l32k_snapkv", "llama8b_b128_l32k", "qwen32b_b16_l100k"])
def test_fullsize_snapkv_select_sampled(name):
    w = synth.WORKLOADS[name]
    k, v, dirs = synth.kv_cache(w, DEV)
    del v
    q_win = synth.window_queries(w, DEV, heavy_dirs=dirs)
    sl = torch.full((w.B,), w.L, dtype=torch.int32, device=DEV)
    idx, n_sel = mb.magicdec_snapkv_select(q_win, k, sl, w.snap_window, w.snap_pool, w.snap_budget)
    torch.cuda.synchronize()
    G = w.G
    band = 0
    for b, h in sample_pairs(w, 2, w.seed + 9):
        L = int(sl[b])
        qo = to_u16(q_win[b:b + 1, :, h * G:(h + 1) * G])
        ko = to_u16(k[b:b + 1, :L, h:h + 1])
        sl_o = np.array([L], np.int32)
        idx_o, n_sel_o, pooled = oracle.snapkv_select(qo, ko, sl_o, w.snap_pool, w.snap_budget)
        band += check_topk(idx[b:b + 1, h:h + 1].cpu().numpy(), n_sel[b:b + 1].cpu().numpy(), idx_o, n_sel_o,
                           pooled, sl_o, w.snap_window, w.snap_budget)
    assert band <= 4 * w.snap_pool + 8
    del k
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,top_k", [("llama8b_b128_l32k", 512), ("qwen32b_b16_l100k", 4096)])
def test_fullsize_topk_draft_sampled(name, top_k):
    w = synth.WORKLOADS[name]
    k, v, _ = synth.kv_cache(w, DEV)
    qd = synth.queries(w, 1, DEV, seed=w.seed * 7 + 3)
    sl = torch.full((w.B,), w.L, dtype=torch.int32, device=DEV)
    idx = torch.empty((w.B, w.H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_topk_draft_attn(qd, k, v, sl, top_k, idx=idx)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w.seed + 11)
    swapped = 0
    for b in rng.choice(w.B, size=2, replace=False):
        b = int(b)
        L = int(sl[b])
        sl_o = np.array([L], np.int32)
        qkv = (to_u16(qd[b:b + 1]), to_u16(k[b:b + 1, :L]), to_u16(v[b:b + 1, :L]))
        ref, idx_o, scores = oracle.topk_attn(*qkv, sl_o, top_k, want_scores=True)
        sw, _ = check_topk_attn(bf16_out_to_f64(out[b:b + 1]), idx[b:b + 1].cpu().numpy(), ref, idx_o, scores, sl_o,
                                top_k, f"{name} topk b={b}", qkv=qkv)
        swapped += sw
    assert swapped <= 2
    del k, v
    torch.cuda.empty_cache()


def test_fullsize_pq_sampled():
    """B=128, L=32000, M=16, C=256: the encode of sampled sequences equals the oracle's (margin rule),
    and PQ draft attention with host-drawn codes matches the oracle on sampled sequences (band rule)."""
    w = synth.WORKLOADS["llama8b_b128_l32k"]
    k, v, _ = synth.kv_cache(w, DEV)
    M, C, top_k = w.d // 8, 256, 512
    gen = torch.Generator(device="cpu").manual_seed(91)
    pick = torch.randint(0, w.L, (w.B, w.H_kv, C), generator=gen).to(DEV)
    bidx = torch.arange(w.B, device=DEV)[:, None, None]
    hidx = torch.arange(w.H_kv, device=DEV)[None, :, None]
    cb = k[bidx, pick, hidx].float().reshape(w.B, w.H_kv, C, M, 8).permute(0, 1, 3, 2, 4).contiguous()
    codes = mb.magicdec_pq_encode(k, cb)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w.seed + 17)
    for b in rng.choice(w.B, size=2, replace=False):
        b = int(b)
        cbo = cb[b:b + 1].cpu().numpy()
        ko = to_u16(k[b:b + 1])
        codes_o, gap = oracle.pq_encode(ko, cbo, want_gap=True)
        kf = bf16_out_to_f64(k[b:b + 1]).reshape(1, w.L, w.H_kv, M, 8).transpose(0, 2, 1, 3, 4)
        kn = (kf ** 2).sum(-1)
        cn = (cbo.astype(np.float64) ** 2).sum(-1)
        cbest = np.take_along_axis(cn[:, :, None], codes_o[..., None].astype(np.int64), axis=-1)[..., 0]
        margin = gap <= 1e-5 * (kn + cbest)
        g = codes[b:b + 1].cpu().numpy()
        assert np.array_equal(g[~margin], codes_o[~margin])
        # 256 centroids in 8 dimensions: the two nearest are often close, so a fraction of a
        # percent of the decisions sits inside the margin
        assert margin.mean() < 2e-2
    rand_codes = torch.randint(0, C, (w.B, w.H_kv, w.L, M), generator=gen, dtype=torch.uint8)
    qd = synth.queries(w, 1, DEV, seed=w.seed * 7 + 5)
    sl = torch.full((w.B,), w.L, dtype=torch.int32, device=DEV)
    idx = torch.empty((w.B, w.H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_pq_draft_attn(qd, k, v, sl, cb, rand_codes.to(DEV), top_k, idx=idx)
    torch.cuda.synchronize()
    for b in rng.choice(w.B, size=2, replace=False):
        b = int(b)
        sl_o = np.array([w.L], np.int32)
        qkv = (to_u16(qd[b:b + 1]), to_u16(k[b:b + 1]), to_u16(v[b:b + 1]))
        ref, idx_o, approx = oracle.pq_attn(*qkv, sl_o, cb[b:b + 1].cpu().numpy(), rand_codes[b:b + 1].numpy(), top_k,
                                            want_approx=True)
        sw, _ = check_topk_attn(bf16_out_to_f64(out[b:b + 1]), idx[b:b + 1].cpu().numpy(), ref, idx_o, approx, sl_o,
                                top_k, f"pq b={b}", qkv=qkv)
        assert sw <= 2
    del k, v, cb, codes, rand_codes
    torch.cuda.empty_cache()


def test_fullsize_draft_cache_ring_sampled():
    """The StreamingLLM ring built from an empty cache at B=128, L=32000, then one draft/verify
    cycle (3 appends, refresh to n_acc = 1): sampled sequences equal the oracle byte for byte."""
    w = synth.WORKLOADS["llama8b_b128_l32k"]
    k, v, _ = synth.kv_cache(w, DEV)
    cap = w.stream_budget
    kc = torch.zeros((w.B, w.H_kv, cap, w.d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    i32 = lambda x: torch.full((w.B,), int(x), dtype=torch.int32, device=DEV)
    L0 = w.L - 8
    org = i32(w.n_sink)
    mb.magicdec_draft_cache_update(k, v, kc, vc, i32(0), i32(0), i32(L0), org, None, w.n_recent)
    for g in range(3):
        mb.magicdec_draft_cache_update(k, v, kc, vc, i32(L0 + g), i32(L0 + g), i32(L0 + g + 1), org, None, w.n_recent)
    dl = mb.magicdec_draft_cache_update(k, v, kc, vc, i32(L0), i32(L0 + 3), i32(L0 + 2), org, None, w.n_recent)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w.seed + 13)
    for b in rng.choice(w.B, size=2, replace=False):
        b = int(b)
        ko, vo = to_u16(k[b:b + 1]), to_u16(v[b:b + 1])
        kc_o = np.zeros((1, w.H_kv, cap, w.d), np.uint16)
        vc_o = np.zeros_like(kc_o)
        one = lambda x: np.array([x], np.int32)
        oo = one(w.n_sink)
        oracle.draft_cache_update(ko, vo, kc_o, vc_o, one(0), one(0), one(L0), oo, None, w.n_recent)
        for g in range(3):
            oracle.draft_cache_update(ko, vo, kc_o, vc_o, one(L0 + g), one(L0 + g), one(L0 + g + 1), oo, None,
                                      w.n_recent)
        dl_o, _ = oracle.draft_cache_update(ko, vo, kc_o, vc_o, one(L0), one(L0 + 3), one(L0 + 2), oo, None,
                                            w.n_recent)
        assert int(dl[b]) == int(dl_o[0]) == cap
        assert np.array_equal(to_u16(kc[b:b + 1]), kc_o)
        assert np.array_equal(to_u16(vc[b:b + 1]), vc_o)
    del k, v, kc, vc
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,greedy", [("llama8b_b128_l32k", False), ("llama8b_b128_l32k", True),
                                         ("llama8b_b64_l32k_snapkv", False), ("qwen32b_b16_l100k", False)])
def test_fullsize_spec_accept(name, greedy):
    w = synth.WORKLOADS[name]
    target, draft, tok, u_acc, u_res = synth.logits(w, DEV)
    got = mb.magicdec_spec_accept(target, draft, tok, u_acc, u_res, greedy)
    torch.cuda.synchronize()
    t, d, x, ua, ur = (a.cpu().numpy() for a in (target, draft, tok, u_acc, u_res))
    ref = oracle_accept(t, d, x, ua, ur, greedy)
    n_amb = check_accept(tuple(a.cpu().numpy() for a in got), ref, name, inputs=(t, d, ur), greedy=greedy)
    assert n_amb <= max(2, w.B // 8)
