"""GPU path (through the C ABI) against the CPU oracle, element by element, on seeded
inputs small enough for the oracle to finish in seconds but spanning several 64-row
tiles, several CTAs per sequence, ragged tails and the degenerate cases."""
import os

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
    assert mb.magicdec_device_error() == 0


def rand_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


# ---------------------------------------------------------------- verification
VERIFY_CASES = [
    # B, H_q, H_kv, d, L_cap, n_q, lengths
    (2, 4, 1, 64, 256, 3, [256, 200]),                                 # the tiny workload
    (5, 32, 8, 128, 1500, 4, [1500, 1, 0, 64, 65]),                    # Llama-3.1-8B heads, edge lengths
    (3, 40, 8, 128, 700, 5, [700, 333, 129]),                          # Qwen-like G=5, 25 rows
    (3, 32, 8, 128, 900, 5, [900, 5, 640]),                            # 20 rows
    (2, 4, 4, 128, 300, 4, [300, 257]),                                # MHA: H_kv == H_q
    (2, 16, 2, 64, 400, 4, [400, 390]),                                # d=64, 32 rows
    (7, 32, 8, 128, 4100, 4, [4100, 4000, 3999, 128, 2050, 17, 4033]),  # many tiles and splits
    # pairs of >= 64 tiles hand a dynamic tail to the pool
    (2, 32, 8, 128, 6000, 4, [6000, 5000]),                            # tails on every pair
    (2, 40, 8, 128, 4500, 5, [4500, 4096]),                            # tails with 25 rows (two row tiles)
    (2, 16, 2, 64, 5000, 4, [5000, 4200]),                             # tails with d=64, 32 rows
    (1, 8, 1, 128, 9000, 4, [9000]),                                   # one pair over every CTA, plus its tail
    (3, 4, 1, 128, 20000, 2, [20000, 3, 19999]),                       # a few long pairs, one short
    # d = 128 with eight KV heads and <= 16 rows per KV head: the all-heads kernel
    (3, 32, 8, 128, 2000, 3, [2000, 1999, 700]),                       # 12 rows per KV head
    (2, 16, 8, 128, 1000, 4, [1000, 513]),                             # G = 2, 8 rows
    (2, 8, 8, 128, 700, 16, [700, 650]),                               # G = 1, 16 speculated tokens
    (4, 32, 8, 128, 64, 4, [64, 1, 0, 9]),                             # fewer tiles than CTAs
    (1, 32, 8, 128, 9000, 4, [9000]),                                  # one sequence over every CTA
    (2, 32, 8, 128, 3000, 1, [3000, 17]),                              # one query token
    # ... and 17 to 32 rows per KV head: 17-24 through the swapped-operand all-heads kernel
    # (three 8-row n-tiles), 25-32 through the per-pair kernel's two row tiles
    (2, 64, 8, 128, 1000, 4, [1000, 333]),                             # G = 8: exactly 32 rows
    (2, 8, 8, 128, 800, 17, [800, 17]),                                # G = 1, 17 rows (one in tile 2)
    (5, 40, 8, 128, 3000, 5, [3000, 5, 0, 2999, 1]),                   # the Qwen-like shape, edge lengths
    (1, 32, 8, 128, 9000, 5, [9000]),                                  # 20 rows, one sequence over every CTA
]


@pytest.mark.parametrize("B,H_q,H_kv,d,L_cap,n_q,lens", VERIFY_CASES)
def test_verify_attn_matches_oracle(B, H_q, H_kv, d, L_cap, n_q, lens):
    q = rand_bf16((B, n_q, H_q, d), 1)
    k = rand_bf16((B, L_cap, H_kv, d), 2)
    v = rand_bf16((B, L_cap, H_kv, d), 3)
    k[:, ::97] *= 4                                                    # a few dominant keys
    sl = torch.tensor(lens, dtype=torch.int32)
    out = mb.magicdec_verify_attn(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.verify_attn(to_u16(q), to_u16(k), to_u16(v), sl.numpy(), n_q)
    check_attention(bf16_out_to_f64(out), ref, "verify")


def test_verify_attn_is_deterministic_and_split_invariant(monkeypatch):
    B, H_q, H_kv, d, L_cap, n_q = 6, 32, 8, 128, 3000, 4
    q, k, v = rand_bf16((B, n_q, H_q, d), 4).to(DEV), rand_bf16((B, L_cap, H_kv, d), 5).to(DEV), \
        rand_bf16((B, L_cap, H_kv, d), 6).to(DEV)
    sl = torch.tensor([3000, 2999, 1500, 64, 700, 2222], dtype=torch.int32, device=DEV)
    a = mb.magicdec_verify_attn(q, k, v, sl)
    b = mb.magicdec_verify_attn(q, k, v, sl)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    monkeypatch.setenv("MAGICDEC_ATTN_CTAS_PER_SM", "2")
    monkeypatch.setenv("MAGICDEC_ATTN_STAGES", "2")
    c = mb.magicdec_verify_attn(q, k, v, sl)
    torch.cuda.synchronize()
    check_attention(bf16_out_to_f64(c), bf16_out_to_f64(a).astype(np.float64), "split invariance")


@pytest.mark.parametrize("n_q", [2, 4])
def test_verify_attn_all_heads_stage_depth_does_not_change_bits(monkeypatch, n_q):
    """The all-heads kernel runs five stages unless MAGICDEC_ATTN_STAGES asks otherwise;
    six (where shared memory has room) and three give the same bits, since the ring's
    depth changes only when a tile arrives, not the order of the arithmetic."""
    B, H_q, H_kv, d, L_cap = 5, 32, 8, 128, 2000
    q, k, v = rand_bf16((B, n_q, H_q, d), 61), rand_bf16((B, L_cap, H_kv, d), 62), rand_bf16((B, L_cap, H_kv, d), 63)
    sl = torch.tensor([2000, 1999, 64, 1, 1234], dtype=torch.int32)
    qd, kd, vd, sld = q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV)
    base = mb.magicdec_verify_attn(qd, kd, vd, sld)
    for st in ("6", "3"):
        monkeypatch.setenv("MAGICDEC_ATTN_STAGES", st)
        other = mb.magicdec_verify_attn(qd, kd, vd, sld)
        torch.cuda.synchronize()
        assert torch.equal(base, other), st
    ref = oracle.verify_attn(to_u16(q), to_u16(k), to_u16(v), sl.numpy(), n_q)
    check_attention(bf16_out_to_f64(base), ref, "verify, all-heads stage depths")


def test_verify_attn_dynamic_tails_deterministic_and_match_static_schedule(monkeypatch):
    """With dynamic tails (per-pair kernel, pairs of >= 64 tiles, at least two pairs per
    CTA) which CTA takes a tail varies from call to call, but the chunk boundaries and
    the merge order do not: repeated calls agree bit for bit, the static schedule (tails
    off) agrees within the tolerance, and sampled sequences match the oracle."""
    monkeypatch.setenv("MAGICDEC_ATTN_HEADS", "0")
    monkeypatch.setenv("MAGICDEC_ATTN_TAILS", "1")                     # opt-in
    B, H_q, H_kv, d, L_cap, n_q = 40, 40, 8, 128, 4200, 4          # 320 pairs, 20 rows per KV head
    g = torch.Generator().manual_seed(17)
    lens = torch.randint(3000, L_cap + 1, (B,), generator=g)
    lens[::7] = L_cap
    lens[3] = 5
    sl = lens.to(torch.int32)
    q, k, v = rand_bf16((B, n_q, H_q, d), 14), rand_bf16((B, L_cap, H_kv, d), 15), rand_bf16((B, L_cap, H_kv, d), 16)
    qd, kd, vd, sld = q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV)
    runs = [mb.magicdec_verify_attn(qd, kd, vd, sld) for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(runs[0], r) for r in runs[1:])
    monkeypatch.setenv("MAGICDEC_ATTN_TAILS", "0")
    static = mb.magicdec_verify_attn(qd, kd, vd, sld)
    torch.cuda.synchronize()
    check_attention(bf16_out_to_f64(runs[0]), bf16_out_to_f64(static).astype(np.float64), "tails vs static")
    pick = [0, 3, 7, 22, 39]
    ref = oracle.verify_attn(to_u16(q[pick]), to_u16(k[pick]), to_u16(v[pick]), sl[pick].numpy(), n_q)
    check_attention(bf16_out_to_f64(runs[0][pick]), ref, "verify with tails")


@pytest.mark.parametrize("heads,H_q,n_q", [("1", 32, 4), ("0", 32, 4), ("1", 32, 5)])
def test_verify_attn_repeated_calls_identical_with_two_waves_of_ctas(monkeypatch, heads, H_q, n_q):
    """Two CTAs per SM (a grid that runs in two waves) and two pipeline stages: short
    sequence runs reuse the query slot and the stages right after releasing them, the
    case where a refill issued without a proxy fence overwrote rows a warp was still
    reading (a 64-position sequence split over three CTAs).  The schedule is fixed, so
    every call must give the same bits, and match the oracle.  16 rows per KV head in
    both kernels; 20 in the swapped-operand all-heads kernel."""
    monkeypatch.setenv("MAGICDEC_ATTN_HEADS", heads)
    monkeypatch.setenv("MAGICDEC_ATTN_CTAS_PER_SM", "2")
    monkeypatch.setenv("MAGICDEC_ATTN_STAGES", "2")
    B, H_kv, d, L_cap = 6, 8, 128, 3000
    q, k, v = rand_bf16((B, n_q, H_q, d), 4), rand_bf16((B, L_cap, H_kv, d), 5), rand_bf16((B, L_cap, H_kv, d), 6)
    sl = torch.tensor([3000, 2999, 1500, 64, 700, 2222], dtype=torch.int32)
    qd, kd, vd, sld = q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV)
    first = mb.magicdec_verify_attn(qd, kd, vd, sld)
    for _ in range(30):
        again = mb.magicdec_verify_attn(qd, kd, vd, sld)
        torch.cuda.synchronize()
        assert torch.equal(first, again)
    ref = oracle.verify_attn(to_u16(q), to_u16(k), to_u16(v), sl.numpy(), n_q)
    check_attention(bf16_out_to_f64(first), ref, "verify, two waves of CTAs")


@pytest.mark.parametrize("H_q,n_q", [(32, 4), (32, 5)])
def test_verify_attn_per_pair_and_all_heads_kernels_agree(monkeypatch, H_q, n_q):
    """The Llama-3.1-8B verification shapes (16 and 20 rows per KV head) run the all-heads
    kernels; the per-pair kernel (MAGICDEC_ATTN_HEADS=0) on the same inputs matches the
    oracle too, and the two agree within the attention tolerance."""
    B, H_kv, d, L_cap = 5, 8, 128, 2600
    q = rand_bf16((B, n_q, H_q, d), 21)
    k = rand_bf16((B, L_cap, H_kv, d), 22)
    v = rand_bf16((B, L_cap, H_kv, d), 23)
    k[:, ::53] *= 4
    sl = torch.tensor([2600, 2, 1300, 0, 2599], dtype=torch.int32)
    ref = oracle.verify_attn(to_u16(q), to_u16(k), to_u16(v), sl.numpy(), n_q)
    qd, kd, vd, sld = q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV)
    heads = mb.magicdec_verify_attn(qd, kd, vd, sld)
    monkeypatch.setenv("MAGICDEC_ATTN_HEADS", "0")
    pair = mb.magicdec_verify_attn(qd, kd, vd, sld)
    torch.cuda.synchronize()
    check_attention(bf16_out_to_f64(heads), ref, "verify, all-heads kernel")
    check_attention(bf16_out_to_f64(pair), ref, "verify, per-pair kernel")
    check_attention(bf16_out_to_f64(heads), bf16_out_to_f64(pair).astype(np.float64), "all-heads vs per-pair")


# ----------------------------------------------------------------------- draft
DRAFT_CASES = [
    (4, 32, 8, 128, 600, [512, 600, 1, 0]),
    (2, 4, 1, 64, 64, [64, 30]),
    (3, 40, 8, 128, 4096, [4096, 4000, 1234]),
]


@pytest.mark.parametrize("B,H_q,H_kv,d,cap,lens", DRAFT_CASES)
def test_draft_attn_matches_oracle(B, H_q, H_kv, d, cap, lens):
    q = rand_bf16((B, 1, H_q, d), 7)
    kc = rand_bf16((B, H_kv, cap, d), 8)
    vc = rand_bf16((B, H_kv, cap, d), 9)
    dl = torch.tensor(lens, dtype=torch.int32)
    out = mb.magicdec_draft_attn(q.to(DEV), kc.to(DEV), vc.to(DEV), dl.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.draft_attn(to_u16(q), to_u16(kc), to_u16(vc), dl.numpy())
    check_attention(bf16_out_to_f64(out), ref, "draft")
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[b]) == 0


def test_draft_attn_ignores_row_order():
    """Attention over a set: permuting the gathered rows leaves the output unchanged."""
    B, H_q, H_kv, d, cap = 2, 32, 8, 128, 512
    q, kc, vc = rand_bf16((B, 1, H_q, d), 10), rand_bf16((B, H_kv, cap, d), 11), rand_bf16((B, H_kv, cap, d), 12)
    perm = torch.randperm(cap, generator=torch.Generator().manual_seed(13))
    dl = torch.full((B,), cap, dtype=torch.int32)
    a = mb.magicdec_draft_attn(q.to(DEV), kc.to(DEV), vc.to(DEV), dl.to(DEV))
    b = mb.magicdec_draft_attn(q.to(DEV), kc[:, :, perm].contiguous().to(DEV), vc[:, :, perm].contiguous().to(DEV),
                               dl.to(DEV))
    torch.cuda.synchronize()
    check_attention(bf16_out_to_f64(b), bf16_out_to_f64(a), "permutation")


# ------------------------------------------------------ StreamingLLM and gather
@pytest.mark.parametrize("n_sink,n_recent", [(4, 60), (16, 496), (0, 32), (7, 0)])
def test_streaming_select_bit_exact(n_sink, n_recent):
    lens = np.array([0, 1, 5, n_sink + n_recent - 1, n_sink + n_recent, n_sink + n_recent + 3, 32000, 100000],
                    np.int32)
    idx, n_sel = mb.magicdec_streaming_select(torch.from_numpy(lens).to(DEV), 8, n_sink, n_recent)
    torch.cuda.synchronize()
    idx_o, n_sel_o = oracle.streaming_select(lens, 8, n_sink, n_recent)
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    assert np.array_equal(n_sel.cpu().numpy(), n_sel_o)


def test_gather_bit_exact_with_padding():
    B, L, H, d, cap = 3, 700, 8, 128, 600
    k, v = rand_bf16((B, L, H, d), 14), rand_bf16((B, L, H, d), 15)
    lens = np.array([700, 300, 20], np.int32)
    idx_o, _ = oracle.streaming_select(lens, H, 16, 496)
    kc_g, vc_g = mb.magicdec_gather_kv(k.to(DEV), v.to(DEV), torch.from_numpy(idx_o).to(DEV), cap)
    torch.cuda.synchronize()
    kc_o, vc_o = oracle.gather_kv(to_u16(k), to_u16(v), idx_o, cap)
    assert np.array_equal(to_u16(kc_g), kc_o)
    assert np.array_equal(to_u16(vc_g), vc_o)


def test_streaming_draft_pipeline_tiny():
    """Select -> gather -> draft attention on the tiny workload, against the oracle chain."""
    w = synth.WORKLOADS["tiny"]
    k, v, _ = synth.kv_cache(w, "cpu")
    q = synth.queries(w, 1, "cpu", seed=99)
    lens = np.array([w.L, w.L - 40], np.int32)
    sl = torch.from_numpy(lens).to(DEV)
    idx, n_sel = mb.magicdec_streaming_select(sl, w.H_kv, w.n_sink, w.n_recent)
    kc, vc = mb.magicdec_gather_kv(k.to(DEV), v.to(DEV), idx, w.stream_budget)
    out = mb.magicdec_draft_attn(q.to(DEV), kc, vc, n_sel)
    torch.cuda.synchronize()
    idx_o, n_sel_o = oracle.streaming_select(lens, w.H_kv, w.n_sink, w.n_recent)
    kc_o, vc_o = oracle.gather_kv(to_u16(k), to_u16(v), idx_o, w.stream_budget)
    ref = oracle.draft_attn(to_u16(q), kc_o, vc_o, n_sel_o)
    check_attention(bf16_out_to_f64(out), ref, "streaming draft")


# ---------------------------------------------------------------------- SnapKV
SNAP_CASES = [
    # B, H_q, H_kv, d, L_cap, w, pool, budget, lens, heavy
    (2, 4, 1, 64, 256, 16, 7, 64, [256, 200], False),                  # the tiny workload
    (2, 4, 1, 64, 256, 16, 7, 64, [64, 30], False),                    # L <= budget keeps everything
    (2, 32, 8, 128, 3000, 32, 7, 512, [3000, 2500], True),             # heavy hitters, 128 window rows
    (2, 40, 8, 128, 2100, 32, 7, 256, [2100, 1800], True),             # G=5: 160 window rows
    (1, 32, 8, 128, 1100, 32, 7, 32, [1100], True),                    # budget == window
]


@pytest.mark.parametrize("B,H_q,H_kv,d,L_cap,w,pool,budget,lens,heavy", SNAP_CASES)
def test_snapkv_select_matches_oracle(B, H_q, H_kv, d, L_cap, w, pool, budget, lens, heavy):
    wl = synth.Workload("case", B=B, H_q=H_q, H_kv=H_kv, d=d, L=L_cap, gamma=1, V=8, snap_window=w,
                        snap_pool=pool, snap_budget=budget, heavy_frac=0.005 if heavy else 0.0, seed=21)
    k, _, dirs = synth.kv_cache(wl, "cpu")
    q_win = synth.window_queries(wl, "cpu", heavy_dirs=dirs)
    sl = np.array(lens, np.int32)
    idx, n_sel = mb.magicdec_snapkv_select(q_win.to(DEV), k.to(DEV), torch.from_numpy(sl).to(DEV), w, pool, budget)
    torch.cuda.synchronize()
    idx_o, n_sel_o, pooled = oracle.snapkv_select(to_u16(q_win), to_u16(k), sl, pool, budget)
    band = check_topk(idx.cpu().numpy(), n_sel.cpu().numpy(), idx_o, n_sel_o, pooled, sl, w, budget)
    # max-pooling copies each local maximum to up to `pool` neighbours, so a
    # plateau or two at the threshold per (sequence, KV head) is expected
    assert band <= 2 * pool * B * H_kv + 8, f"too many band positions: {band}"


# ------------------------------------------------------------ PQCache-style
PQ_MARGIN = 1e-5      # relative to |k_m|^2 + |c|^2: fp32 dot-product distances vs the oracle's fp64


def _pq_codebook(rng, B, H_kv, M, C, scale=1.0):
    return (scale * rng.standard_normal((B, H_kv, M, C, 8))).astype(np.float32)


@pytest.mark.parametrize("tc", ["1", "0"])          # tensor-core encoder; the FMA encoder
@pytest.mark.parametrize("B,H_kv,L,C", [(2, 8, 3000, 64), (2, 2, 1500, 256), (1, 8, 700, 7), (2, 4, 999, 200)])
def test_pq_encode_matches_oracle(B, H_kv, L, C, tc, monkeypatch):
    monkeypatch.setenv("MAGICDEC_PQ_TC", tc)
    rng = np.random.default_rng(71)
    d, M = 128, 16
    k = rand_bf16((B, L, H_kv, d), 72)
    cb = _pq_codebook(rng, B, H_kv, M, C)
    codes = mb.magicdec_pq_encode(k.to(DEV), torch.from_numpy(cb).to(DEV))
    torch.cuda.synchronize()
    codes_o, gap = oracle.pq_encode(to_u16(k), cb, want_gap=True)
    g = codes.cpu().numpy()
    kf = bf16_out_to_f64(k).reshape(B, L, H_kv, M, 8).transpose(0, 2, 1, 3, 4)      # [B,H_kv,L,M,8]
    kn = (kf ** 2).sum(-1)
    cn = (cb.astype(np.float64) ** 2).sum(-1)                                       # [B,H_kv,M,C]
    cbest = np.take_along_axis(cn[:, :, None, :, :], codes_o[..., None].astype(np.int64), axis=-1)[..., 0]
    margin = gap <= PQ_MARGIN * (kn + cbest)
    assert np.array_equal(g[~margin], codes_o[~margin])
    assert margin.mean() < 1e-3, f"{margin.sum()} margin codes"


def test_pq_update_matches_oracle_exactly():
    rng = np.random.default_rng(73)
    B, H_kv, d, L, M, C = 2, 8, 128, 2500, 16, 64
    k = rand_bf16((B, L, H_kv, d), 74)
    cb = _pq_codebook(rng, B, H_kv, M, C)
    codes, _ = oracle.pq_encode(to_u16(k), cb)
    codes[0, 0, :, 3] = 5                  # crowd one centroid, empty another
    codes[codes == 9] = 10
    sl = np.array([L, 1777], np.int32)
    cb_g = torch.from_numpy(cb.copy()).to(DEV)
    mb.magicdec_pq_update(k.to(DEV), torch.from_numpy(sl).to(DEV), torch.from_numpy(codes).to(DEV), cb_g)
    torch.cuda.synchronize()
    cb_o = oracle.pq_update(to_u16(k), sl, codes, cb)
    np.testing.assert_array_equal(cb_g.cpu().numpy(), cb_o)


@pytest.mark.parametrize("B,H_q,H_kv,L,C,top_k,lens", [
    (3, 32, 8, 3000, 64, 256, [3000, 2000, 100]),
    (2, 40, 8, 2100, 256, 512, [2100, 1500]),
    (2, 16, 2, 1200, 32, 64, [1200, 0]),
])
def test_pq_draft_attn_matches_oracle(B, H_q, H_kv, L, C, top_k, lens):
    rng = np.random.default_rng(75)
    d, M = 128, 16
    q = rand_bf16((B, 1, H_q, d), 76)
    k = rand_bf16((B, L, H_kv, d), 77)
    v = rand_bf16((B, L, H_kv, d), 78)
    k[:, ::61] *= 3
    cb = _pq_codebook(rng, B, H_kv, M, C)
    sl = np.array(lens, np.int32)
    codes, _ = oracle.pq_encode(to_u16(k), cb)
    cb = oracle.pq_update(to_u16(k), np.full(B, L, np.int32), codes, cb)
    codes, _ = oracle.pq_encode(to_u16(k), cb)
    idx = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_pq_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(sl).to(DEV),
                                    torch.from_numpy(cb).to(DEV), torch.from_numpy(codes).to(DEV), top_k, idx=idx)
    torch.cuda.synchronize()
    ref, idx_o, approx = oracle.pq_attn(to_u16(q), to_u16(k), to_u16(v), sl, cb, codes, top_k, want_approx=True)
    swapped, _ = check_topk_attn(bf16_out_to_f64(out), idx.cpu().numpy(), ref, idx_o, approx, sl, top_k, "pq",
                                 qkv=(to_u16(q), to_u16(k), to_u16(v)))
    assert swapped <= max(1, B * H_q // 50)
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.count_nonzero(out[b]) == 0


def test_pq_head_dim_64():
    """d = 64 (M = 8 subspaces, 8-byte code rows): encode under the margin rule, an exact update,
    and PQ attention under the band rule."""
    rng = np.random.default_rng(80)
    B, H_q, H_kv, d, L, M, C, top_k = 2, 16, 4, 64, 1800, 8, 64, 128
    q = rand_bf16((B, 1, H_q, d), 81)
    k = rand_bf16((B, L, H_kv, d), 82)
    v = rand_bf16((B, L, H_kv, d), 83)
    cb = _pq_codebook(rng, B, H_kv, M, C)
    codes_g = mb.magicdec_pq_encode(k.to(DEV), torch.from_numpy(cb).to(DEV))
    torch.cuda.synchronize()
    codes_o, gap = oracle.pq_encode(to_u16(k), cb, want_gap=True)
    kf = bf16_out_to_f64(k).reshape(B, L, H_kv, M, 8).transpose(0, 2, 1, 3, 4)
    kn = (kf ** 2).sum(-1)
    cn = (cb.astype(np.float64) ** 2).sum(-1)
    cbest = np.take_along_axis(cn[:, :, None, :, :], codes_o[..., None].astype(np.int64), axis=-1)[..., 0]
    margin = gap <= PQ_MARGIN * (kn + cbest)
    assert np.array_equal(codes_g.cpu().numpy()[~margin], codes_o[~margin])
    sl = np.array([L, 1100], np.int32)
    cb_g = torch.from_numpy(cb.copy()).to(DEV)
    mb.magicdec_pq_update(k.to(DEV), torch.from_numpy(sl).to(DEV), torch.from_numpy(codes_o).to(DEV), cb_g)
    torch.cuda.synchronize()
    cb2 = oracle.pq_update(to_u16(k), sl, codes_o, cb)
    np.testing.assert_array_equal(cb_g.cpu().numpy(), cb2)
    codes2, _ = oracle.pq_encode(to_u16(k), cb2)
    idx = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_pq_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(sl).to(DEV),
                                    torch.from_numpy(cb2).to(DEV), torch.from_numpy(codes2).to(DEV), top_k, idx=idx)
    torch.cuda.synchronize()
    ref, idx_o, approx = oracle.pq_attn(to_u16(q), to_u16(k), to_u16(v), sl, cb2, codes2, top_k, want_approx=True)
    swapped, _ = check_topk_attn(bf16_out_to_f64(out), idx.cpu().numpy(), ref, idx_o, approx, sl, top_k, "pq d64",
                                 qkv=(to_u16(q), to_u16(k), to_u16(v)))
    assert swapped <= 1


def test_pq_lloyd_pipeline_on_planted_clusters():
    """GPU encode + update twice from one member per planted cluster: codes equal the oracle's and the
    planted labels, codebooks equal the oracle's."""
    rng = np.random.default_rng(79)
    B, L, H_kv, d, M, C = 2, 2000, 4, 128, 16, 12
    proto = rng.standard_normal((B, H_kv, M, C, 8)) * 4.0
    label = rng.integers(0, C, size=(B, H_kv, L, M))
    label[:, :, :C] = np.arange(C)[None, None, :, None]
    sub = np.take_along_axis(proto[:, :, None], label[..., None, None].repeat(8, -1), axis=4)[..., 0, :]
    kf = (sub + 0.05 * rng.standard_normal(sub.shape)).transpose(0, 2, 1, 3, 4).reshape(B, L, H_kv, d)
    k = torch.from_numpy(np.ascontiguousarray(kf, dtype=np.float32)).to(torch.bfloat16)
    ku = to_u16(k)
    kb = bf16_out_to_f64(k).reshape(B, L, H_kv, M, 8)
    cb0 = kb[:, :C].transpose(0, 2, 3, 1, 4).astype(np.float32).copy()
    sl = np.full(B, L, np.int32)
    cb_g = torch.from_numpy(cb0.copy()).to(DEV)
    k_g, sl_g = k.to(DEV), torch.from_numpy(sl).to(DEV)
    cb_o = cb0
    for _ in range(2):
        codes_g = mb.magicdec_pq_encode(k_g, cb_g)
        mb.magicdec_pq_update(k_g, sl_g, codes_g, cb_g)
        codes_o, _ = oracle.pq_encode(ku, cb_o)
        cb_o = oracle.pq_update(ku, sl, codes_o, cb_o)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(codes_g.cpu().numpy(), codes_o)
    np.testing.assert_array_equal(codes_o, label)
    np.testing.assert_array_equal(cb_g.cpu().numpy(), cb_o)


# ------------------------------------------------------- draft-cache update
def _dc_step(k, v, kc, vc, kc_o, vc_o, lv, lo, ln, origin, base, ring):
    dev = torch.device(DEV)
    t = lambda a: torch.from_numpy(np.asarray(a, np.int32)).to(dev)
    dl = mb.magicdec_draft_cache_update(k, v, kc, vc, t(lv), t(lo), t(ln), t(origin),
                                        None if base is None else t(base), ring)
    dl_o, _ = oracle.draft_cache_update(to_u16(k), to_u16(v), kc_o, vc_o, lv, lo, ln, origin, base, ring)
    torch.cuda.synchronize()
    dl_g = dl.cpu().numpy()
    assert np.array_equal(dl_g, dl_o)
    kg, vg = to_u16(kc), to_u16(vc)
    for b in range(kc.shape[0]):
        assert np.array_equal(kg[b, :, : dl_o[b]], kc_o[b, :, : dl_o[b]]), b
        assert np.array_equal(vg[b, :, : dl_o[b]], vc_o[b, :, : dl_o[b]]), b
    return dl


def test_draft_cache_update_ring_walk_matches_oracle():
    """StreamingLLM 16+496 ring: build from empty, then draft appends and post-verification refreshes
    with random acceptance; every state equals the oracle's byte for byte, and draft attention over the
    ring equals the oracle's attention over the ascending StreamingLLM gather."""
    rng = np.random.default_rng(61)
    B, H_q, H_kv, d, L, S, W, gamma = 4, 32, 8, 128, 3000, 16, 496, 3
    k = rand_bf16((B, L, H_kv, d), 62).to(DEV)
    v = rand_bf16((B, L, H_kv, d), 63).to(DEV)
    cap = S + W
    kc = torch.zeros((B, H_kv, cap, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kc_o = np.zeros((B, H_kv, cap, d), np.uint16)
    vc_o = np.zeros_like(kc_o)
    origin = np.full(B, S, np.int32)
    length = np.array([5, 300, 512, 2500], np.int32)
    z = np.zeros(B, np.int32)
    _dc_step(k, v, kc, vc, kc_o, vc_o, z, z, length, origin, None, W)
    for _ in range(12):
        for i in range(gamma):
            _dc_step(k, v, kc, vc, kc_o, vc_o, length + i, length + i, length + i + 1, origin, None, W)
        new = length + rng.integers(0, gamma + 1, size=B).astype(np.int32) + 1
        dl = _dc_step(k, v, kc, vc, kc_o, vc_o, length, length + gamma, new, origin, None, W)
        length = new
    q = rand_bf16((B, 1, H_q, d), 64)
    out = mb.magicdec_draft_attn(q.to(DEV), kc, vc, dl)
    torch.cuda.synchronize()
    idx, n_sel = oracle.streaming_select(length, H_kv, S, W)
    kg_o, vg_o = oracle.gather_kv(to_u16(k), to_u16(v), idx, cap)
    ref = oracle.draft_attn(to_u16(q), kg_o, vg_o, n_sel)
    check_attention(bf16_out_to_f64(out), ref, "draft over the ring cache")


def test_draft_cache_update_linear_and_capacity():
    B, H_kv, d, L, L0, n_sel, cap = 3, 8, 64, 900, 600, 100, 160
    k = rand_bf16((B, L, H_kv, d), 65).to(DEV)
    v = rand_bf16((B, L, H_kv, d), 66).to(DEV)
    kc = torch.zeros((B, H_kv, cap, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kc_o = np.zeros((B, H_kv, cap, d), np.uint16)
    vc_o = np.zeros_like(kc_o)
    origin = np.full(B, L0, np.int32)
    base = np.array([n_sel, n_sel - 7, n_sel], np.int32)
    length = origin.copy()
    for grow in (3, 1, 20):
        _dc_step(k, v, kc, vc, kc_o, vc_o, length, length, length + grow, origin, base, 0)
        length = length + grow
    # roll back 10 then re-append 4 (lengths shrink: nothing to restore in the linear layout)
    _dc_step(k, v, kc, vc, kc_o, vc_o, length - 10, length, length - 6, origin, base, 0)
    length = length - 6
    assert mb.magicdec_device_error() == 0
    # past the capacity: rows skipped, draft_len clamped, error word 3 reported once
    over = np.full(B, L0 + cap, np.int32)
    _dc_step(k, v, kc, vc, kc_o, vc_o, length, length, over, origin, base, 0)
    assert mb.magicdec_device_error() == 3
    assert mb.magicdec_device_error() == 0


# ------------------------------------------------------------ Top-K attention
TOPK_CASES = [
    # B, H_q, H_kv, d, L_cap, top_k, lens
    (2, 4, 1, 64, 256, 48, [256, 200]),                                # the tiny workload's shape
    (4, 32, 8, 128, 3000, 512, [3000, 2999, 513, 0]),                  # Llama-3.1-8B heads, k+1, empty
    (3, 40, 8, 128, 2100, 256, [2100, 256, 100]),                      # G=5; len == k; len < k
    (2, 16, 2, 64, 1500, 1, [1500, 1]),                                # G=8, top-1
    (2, 8, 2, 128, 70000, 2048, [70000, 41000]),                       # long rows
    (1, 40, 8, 128, 20000, 4096, [20000]),                             # G=5, a 4096 budget
    (2, 4, 4, 128, 1500, 64, [1500, 900]),                             # MHA: G=1
    (2, 4, 2, 64, 1000, 100, [1000, 999]),                             # G=2, d=64
    (3, 64, 8, 128, 1700, 128, [1700, 15, 1009]),                      # G=8 over eight KV heads, ragged tiles
]


@pytest.mark.parametrize("B,H_q,H_kv,d,L_cap,top_k,lens", TOPK_CASES)
def test_topk_draft_attn_matches_oracle(B, H_q, H_kv, d, L_cap, top_k, lens):
    q = rand_bf16((B, 1, H_q, d), 41)
    k = rand_bf16((B, L_cap, H_kv, d), 42)
    v = rand_bf16((B, L_cap, H_kv, d), 43)
    k[:, ::97] *= 4                                                    # a few dominant keys
    sl = np.array(lens, np.int32)
    idx = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_topk_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(sl).to(DEV), top_k, idx=idx)
    torch.cuda.synchronize()
    ref, idx_o, scores = oracle.topk_attn(to_u16(q), to_u16(k), to_u16(v), sl, top_k, want_scores=True)
    swapped, band = check_topk_attn(bf16_out_to_f64(out), idx.cpu().numpy(), ref, idx_o, scores, sl, top_k,
                                    qkv=(to_u16(q), to_u16(k), to_u16(v)))
    assert swapped <= max(1, B * H_q // 50), f"{swapped} heads swapped a position inside the band"
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[b]) == 0


@pytest.mark.parametrize("stages", ["", "3"])
def test_topk_scores_all_heads_and_per_pair_kernels_agree(monkeypatch, stages):
    """At d = 128 with eight KV heads the scores come from the kernel that streams all
    heads of a sequence per stage; the per-pair kernel (MAGICDEC_TOPK_HEADS=0) runs the
    same mma sequence per (position, query head), so the kept positions are identical
    and the outputs equal, whatever the score pass's stage depth (MAGICDEC_TOPK_STAGES:
    the default and three per CTA)."""
    if stages:
        monkeypatch.setenv("MAGICDEC_TOPK_STAGES", stages)
    B, H_q, H_kv, d, L_cap, top_k = 3, 32, 8, 128, 2500, 256
    q = rand_bf16((B, 1, H_q, d), 51).to(DEV)
    k = rand_bf16((B, L_cap, H_kv, d), 52).to(DEV)
    v = rand_bf16((B, L_cap, H_kv, d), 53).to(DEV)
    sl = torch.tensor([2500, 1999, 300], dtype=torch.int32, device=DEV)
    idx_h = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    idx_p = torch.empty_like(idx_h)
    out_h = mb.magicdec_topk_draft_attn(q, k, v, sl, top_k, idx=idx_h)
    monkeypatch.setenv("MAGICDEC_TOPK_HEADS", "0")
    out_p = mb.magicdec_topk_draft_attn(q, k, v, sl, top_k, idx=idx_p)
    torch.cuda.synchronize()
    assert torch.equal(idx_h, idx_p)
    assert torch.equal(out_h, out_p)


def test_topk_draft_attn_ties_go_to_smaller_positions():
    """Thirty copies of one dominant key and top_k = 10: exactly the ten smallest copies are kept."""
    B, H_q, H_kv, d, L = 2, 8, 2, 128, 1000
    q = rand_bf16((B, 1, H_q, d), 44)
    k = rand_bf16((B, L, H_kv, d), 45)
    v = rand_bf16((B, L, H_kv, d), 46)
    pos = torch.randperm(L, generator=torch.Generator().manual_seed(47))[:30]
    for h in range(H_kv):
        k[:, pos, h, :] = (q[:, 0, h * (H_q // H_kv), :] * 4).unsqueeze(1)
    sl = np.array([L, L - 3], np.int32)
    idx = torch.empty((B, H_q, 10), dtype=torch.int32, device=DEV)
    out = mb.magicdec_topk_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(sl).to(DEV), 10, idx=idx)
    torch.cuda.synchronize()
    ref, idx_o, _ = oracle.topk_attn(to_u16(q), to_u16(k), to_u16(v), sl, 10)
    g = idx.cpu().numpy()
    for h in range(0, H_q, H_q // H_kv):     # the query head the copies were aligned with
        assert np.array_equal(g[:, h], idx_o[:, h]), h
    check_attention(bf16_out_to_f64(out)[:, 0, :: H_q // H_kv], ref[:, 0, :: H_q // H_kv], "topk ties")


def test_topk_draft_attn_all_scores_equal():
    """Every key identical: all scores tie, so the first top_k positions are kept and the output is
    the mean of their values (the candidate list overflows and the whole row is searched)."""
    B, H_q, H_kv, d, L, top_k = 2, 8, 2, 128, 6000, 100
    q = rand_bf16((B, 1, H_q, d), 48)
    k = rand_bf16((B, 1, H_kv, d), 49).expand(B, L, H_kv, d).contiguous()
    v = rand_bf16((B, L, H_kv, d), 50)
    sl = np.array([L, 4500], np.int32)
    idx = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_topk_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(sl).to(DEV), top_k, idx=idx)
    torch.cuda.synchronize()
    ref, idx_o, _ = oracle.topk_attn(to_u16(q), to_u16(k), to_u16(v), sl, top_k)
    assert np.array_equal(idx_o, np.broadcast_to(np.arange(top_k, dtype=np.int32), idx_o.shape))
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    check_attention(bf16_out_to_f64(out), ref, "topk all-equal")


def test_topk_long_row_all_scores_equal():
    """A row long enough for the sampled threshold (L >= 8192 and >= 8 top_k) with every score
    tied: the candidates overflow the slots, so the whole row is counted and searched, and the
    first top_k positions are kept."""
    B, H_q, H_kv, d, L, top_k = 1, 4, 1, 128, 9000, 100
    q = rand_bf16((B, 1, H_q, d), 51)
    k = rand_bf16((B, 1, H_kv, d), 52).expand(B, L, H_kv, d).contiguous()
    v = rand_bf16((B, L, H_kv, d), 53)
    sl = np.array([L], np.int32)
    idx = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_topk_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(sl).to(DEV), top_k, idx=idx)
    torch.cuda.synchronize()
    ref, idx_o, _ = oracle.topk_attn(to_u16(q), to_u16(k), to_u16(v), sl, top_k)
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    check_attention(bf16_out_to_f64(out), ref, "topk long all-equal")


def test_topk_sampled_threshold_miss_falls_back_to_the_whole_row():
    """The sampled threshold reads one 128-key block per warp at positions len * w / 16 (w < 16).
    Keys there are made the largest of the row (spread over several first-digit bins), so the
    sample's threshold keeps fewer than top_k candidates; the kernel must notice, count the
    whole row and still keep exactly the oracle's top_k."""
    B, H_q, H_kv, d, L, top_k = 1, 4, 1, 128, 32768, 4096
    q = rand_bf16((B, 1, H_q, d), 54)
    k = rand_bf16((B, L, H_kv, d), 55)
    v = rand_bf16((B, L, H_kv, d), 56)
    qd = q[0, 0, 0].float()
    unit = qd / qd.norm()
    for w in range(16):
        sb = (L * w // 16) & ~3
        scale = torch.linspace(2.0, 6.0, 128) * (1.0 + 0.01 * w)
        k[0, sb:sb + 128, 0, :] = (unit.unsqueeze(0) * scale.unsqueeze(1) * 3.0).to(torch.bfloat16)
    sl = np.array([L], np.int32)
    idx = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_topk_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(sl).to(DEV), top_k, idx=idx)
    torch.cuda.synchronize()
    ref, idx_o, scores = oracle.topk_attn(to_u16(q), to_u16(k), to_u16(v), sl, top_k, want_scores=True)
    g = idx.cpu().numpy()
    # head 0's sample-block keys are all kept (they are its 2048 largest scores)
    blocks = np.concatenate([np.arange((L * w // 16) & ~3, ((L * w // 16) & ~3) + 128) for w in range(16)])
    assert np.isin(blocks, g[0, 0]).all()
    check_topk_attn(bf16_out_to_f64(out), g, ref, idx_o, scores, sl, top_k, "topk sampled-threshold miss",
                    qkv=(to_u16(q), to_u16(k), to_u16(v)))


def test_snapkv_select_with_a_budget_per_sequence():
    """Heterogeneous budgets in one batch: each sequence equals the oracle run at its own budget
    (band rule), rows padded with -1 to the largest budget."""
    B, H_q, H_kv, d, L_cap, w, pool = 4, 32, 8, 128, 3000, 32, 7
    budgets = np.array([512, 96, 32, 700], np.int32)
    lens = np.array([3000, 2500, 2000, 600], np.int32)          # the last is shorter than its budget
    wl = synth.Workload("case", B=B, H_q=H_q, H_kv=H_kv, d=d, L=L_cap, gamma=1, V=8, snap_window=w,
                        snap_pool=pool, snap_budget=512, heavy_frac=0.005, seed=23)
    k, _, dirs = synth.kv_cache(wl, "cpu")
    q_win = synth.window_queries(wl, "cpu", heavy_dirs=dirs)
    max_budget = int(budgets.max())
    idx, n_sel = mb.magicdec_snapkv_select_budgets(q_win.to(DEV), k.to(DEV), torch.from_numpy(lens).to(DEV), w, pool,
                                                   torch.from_numpy(budgets).to(DEV), max_budget)
    torch.cuda.synchronize()
    g_idx, g_n = idx.cpu().numpy(), n_sel.cpu().numpy()
    for b in range(B):
        bud = int(budgets[b])
        idx_o, n_sel_o, pooled = oracle.snapkv_select(to_u16(q_win[b:b + 1]), to_u16(k[b:b + 1]), lens[b:b + 1],
                                                      pool, bud)
        check_topk(g_idx[b:b + 1, :, :bud], g_n[b:b + 1], idx_o, n_sel_o, pooled, lens[b:b + 1], w, bud)
        assert np.all(g_idx[b, :, bud:] == -1)


# ------------------------------------------------------------------ acceptance
ACCEPT_CASES = [
    ("tiny", 64, False), ("tiny", 64, True),
    ("llama8b_b128_l32k", 24, False), ("llama8b_b128_l32k", 24, True),
    ("qwen32b_b16_l100k", 8, False),
]


@pytest.mark.parametrize("name,B,greedy", ACCEPT_CASES)
def test_spec_accept_matches_oracle(name, B, greedy):
    w = synth.WORKLOADS[name]
    target, draft, tok, u_acc, u_res = synth.logits(w, "cpu", B=B, seed=31)
    if greedy:
        # make the chain non-trivial: half the draft tokens are the target argmax
        am = target[:, : w.gamma].argmax(-1).to(torch.int32)
        pick = torch.rand(tok.shape, generator=torch.Generator().manual_seed(5)) < 0.7
        tok = torch.where(pick, am, tok)
    got = mb.magicdec_spec_accept(target.to(DEV), draft.to(DEV), tok.to(DEV), u_acc.to(DEV), u_res.to(DEV), greedy)
    torch.cuda.synchronize()
    ref = oracle_accept(target.numpy(), draft.numpy(), tok.numpy(), u_acc.numpy(), u_res.numpy(), greedy)
    gpu = tuple(t.cpu().numpy() for t in got)
    n_amb = check_accept(gpu, ref, name, inputs=(target.numpy(), draft.numpy(), u_res.numpy()), greedy=greedy)
    assert n_amb <= max(2, B // 4)


def test_spec_accept_edge_tokens():
    """Out-of-range draft tokens are rejected; gamma = 0 only draws the bonus token."""
    B, V = 8, 40
    g = torch.Generator().manual_seed(3)
    target = torch.randn((B, 3, V), generator=g) * 2
    draft = target[:, :2] + torch.randn((B, 2, V), generator=g) * 0.5
    tok = torch.randint(0, V, (B, 2), generator=g, dtype=torch.int32)
    tok[0, 0] = -3
    tok[1, 0] = V + 5
    u_acc, u_res = torch.rand((B, 2), generator=g), torch.rand((B,), generator=g)
    got = mb.magicdec_spec_accept(target.to(DEV), draft.to(DEV), tok.to(DEV), u_acc.to(DEV), u_res.to(DEV), False)
    torch.cuda.synchronize()
    ref = oracle_accept(target.numpy(), draft.numpy(), tok.numpy(), u_acc.numpy(), u_res.numpy(), False)
    check_accept(tuple(t.cpu().numpy() for t in got), ref)
    assert got[0][0].item() == 0 and got[0][1].item() == 0
    t0 = target[:, :1].contiguous()
    got0 = mb.magicdec_spec_accept(t0.to(DEV), None, torch.zeros((B, 0), dtype=torch.int32, device=DEV),
                                   torch.zeros((B, 0), device=DEV), u_res.to(DEV), False)
    torch.cuda.synchronize()
    ref0 = oracle_accept(t0.numpy(), np.zeros((B, 0, V), np.float32), np.zeros((B, 0), np.int32),
                         np.zeros((B, 0), np.float32), u_res.numpy(), False)
    check_accept(tuple(t.cpu().numpy() for t in got0), ref0, "gamma=0")


@pytest.mark.parametrize("V", [10003, 4097, 1021])
@pytest.mark.parametrize("greedy", [False, True])
def test_spec_accept_vocabulary_not_a_multiple_of_4(V, greedy):
    """Scalar load paths of the statistics, chunk-sum and draw kernels (V % 4 != 0), several
    4096-logit chunks and a partial last statistics record."""
    B, gamma = 16, 3
    g = torch.Generator().manual_seed(V)
    target = torch.randn((B, gamma + 1, V), generator=g) * 2
    draft = target[:, :gamma] + torch.randn((B, gamma, V), generator=g) * 0.5
    tok = torch.distributions.Categorical(logits=draft).sample().to(torch.int32)
    if greedy:
        am = target[:, :gamma].argmax(-1).to(torch.int32)
        tok = torch.where(torch.rand(tok.shape, generator=g) < 0.7, am, tok)
    u_acc, u_res = torch.rand((B, gamma), generator=g), torch.rand((B,), generator=g)
    got = mb.magicdec_spec_accept(target.to(DEV), draft.to(DEV), tok.to(DEV), u_acc.to(DEV), u_res.to(DEV), greedy)
    torch.cuda.synchronize()
    t, d, x, ua, ur = (a.numpy() for a in (target, draft, tok, u_acc, u_res))
    ref = oracle_accept(t, d, x, ua, ur, greedy)
    n_amb = check_accept(tuple(a.cpu().numpy() for a in got), ref, f"V={V}", inputs=(t, d, ur), greedy=greedy)
    assert n_amb <= 2


def test_rows_past_the_length_never_reach_the_output():
    """Cache rows at or beyond a sequence's length may hold anything (here NaN): outputs
    must equal the oracle's, which never reads them."""
    B, H_q, H_kv, d, L_cap, n_q = 3, 32, 8, 128, 500, 4
    q, k, v = rand_bf16((B, n_q, H_q, d), 40), rand_bf16((B, L_cap, H_kv, d), 41), rand_bf16((B, L_cap, H_kv, d), 42)
    lens = [437, 64, 130]
    for b, L in enumerate(lens):
        k[b, L:] = float("nan")
        v[b, L:] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32)
    out = mb.magicdec_verify_attn(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV))
    kc, vc = k.transpose(1, 2).contiguous(), v.transpose(1, 2).contiguous()
    dout = mb.magicdec_draft_attn(q[:, -1:].contiguous().to(DEV), kc.to(DEV), vc.to(DEV), sl.to(DEV))
    torch.cuda.synchronize()
    check_attention(bf16_out_to_f64(out), oracle.verify_attn(to_u16(q), to_u16(k), to_u16(v), sl.numpy(), n_q),
                    "verify with NaN tail")
    check_attention(bf16_out_to_f64(dout), oracle.draft_attn(to_u16(q[:, -1:]), to_u16(kc), to_u16(vc), sl.numpy()),
                    "draft with NaN tail")
