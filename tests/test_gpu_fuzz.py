"""Randomised shapes and length mixes at d = 128 with eight KV heads: the all-heads
verification kernel (up to 16 rows per KV head) against the per-pair kernel and against
itself across repeated calls; verification at 17-32 rows per KV head (17-24 in the
swapped-operand all-heads kernel, 25-32 in the per-pair kernel's two row tiles) against the
oracle; the Top-K score pass against the per-pair score kernel; draft attention over
random compact caches, speculative accept over random vocabularies, SnapKV selection,
the Top-K draft and the gather against the oracle.  Seeded; each case is small (a few
MB), so the whole file runs in well under a minute."""
import os

import numpy as np
import pytest
import torch

from long_context_self_gb300 import binding as mb
from parity_util import bf16_out_to_f64, check_attention

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_self_gb300 import build
    build.build()
    mb.lib()
    yield
    assert mb.magicdec_device_error() == 0


def _lengths(rng, B, L_cap):
    kinds = rng.integers(0, 5, size=B)
    lens = []
    for k in kinds:
        if k == 0:
            lens.append(int(L_cap))                      # full
        elif k == 1:
            lens.append(int(rng.integers(0, 9)))         # empty or shorter than a tile
        elif k == 2:
            lens.append(int(rng.integers(1, L_cap + 1)))
        elif k == 3:
            lens.append(int(max(0, L_cap - rng.integers(0, 17))))
        else:
            lens.append(int(rng.integers(1, 65)))
    return [min(x, L_cap) for x in lens]


def _case(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 24))
    L_cap = int(rng.choice([8, 63, 200, 1000, 2500, 4100, 7000]))
    G = int(rng.choice([1, 2, 4]))
    n_q = int(rng.integers(1, 16 // G + 1)) if G < 4 else int(rng.integers(1, 5))
    n_q = min(n_q, 4)
    return rng, B, L_cap, G, n_q, _lengths(rng, B, L_cap)


@pytest.mark.parametrize("seed", range(40))
def test_verify_all_heads_fuzz(seed, monkeypatch):
    rng, B, L_cap, G, n_q, lens = _case(seed)
    H_kv, d = 8, 128
    H_q = G * H_kv
    g = torch.Generator().manual_seed(1000 + seed)
    q = torch.randn((B, n_q, H_q, d), generator=g).to(torch.bfloat16).to(DEV)
    k = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16).to(DEV)
    v = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16).to(DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    monkeypatch.setenv("MAGICDEC_ATTN_CTAS_PER_SM", str(int(rng.integers(1, 3))))
    monkeypatch.setenv("MAGICDEC_ATTN_STAGES", str(int(rng.choice([0, 2, 3]))))
    a = mb.magicdec_verify_attn(q, k, v, sl)
    b = mb.magicdec_verify_attn(q, k, v, sl)
    monkeypatch.setenv("MAGICDEC_ATTN_HEADS", "0")
    ref = mb.magicdec_verify_attn(q, k, v, sl)
    torch.cuda.synchronize()
    assert torch.equal(a, b), "all-heads verification is not reproducible"
    check_attention(bf16_out_to_f64(a), bf16_out_to_f64(ref).astype(np.float64),
                    f"all-heads vs per-pair, B={B} L={L_cap} G={G} n_q={n_q} lens={lens}")
    for i, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(a[i]) == 0


def _case_two_tiles(seed):
    """17 to 32 query rows per KV head (two 16-row tiles), the shapes of 4-5 speculated
    tokens over 4-8 query heads per KV head."""
    rng = np.random.default_rng(5000 + seed)
    B = int(rng.integers(1, 10))
    L_cap = int(rng.choice([8, 63, 200, 1000, 2500, 4100]))
    G = int(rng.choice([1, 2, 4, 5, 8]))
    n_q = int(rng.integers((17 + G - 1) // G, 32 // G + 1))
    return rng, B, L_cap, G, n_q, _lengths(rng, B, L_cap)


@pytest.mark.parametrize("seed", range(16))
def test_verify_two_row_tiles_fuzz(seed, monkeypatch):
    """d = 128 with eight KV heads and 17-32 rows per KV head (17-24: the swapped-operand
    all-heads kernel; 25-32: the per-pair kernel with two row tiles): equal to the oracle,
    reproducible across calls and across schedules (stage counts); the per-pair kernel on the
    same inputs equals the oracle too."""
    import oracle
    from parity_util import to_u16
    rng, B, L_cap, G, n_q, lens = _case_two_tiles(seed)
    assert 17 <= G * n_q <= 32
    H_kv, d = 8, 128
    H_q = G * H_kv
    g = torch.Generator().manual_seed(3000 + seed)
    q = torch.randn((B, n_q, H_q, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    a = mb.magicdec_verify_attn(qd, kd, vd, sl)
    b = mb.magicdec_verify_attn(qd, kd, vd, sl)
    monkeypatch.setenv("MAGICDEC_ATTN_STAGES", str(int(rng.choice([2, 3]))))
    c = mb.magicdec_verify_attn(qd, kd, vd, sl)
    monkeypatch.setenv("MAGICDEC_ATTN_HEADS", "0")
    monkeypatch.delenv("MAGICDEC_ATTN_STAGES")
    pp = mb.magicdec_verify_attn(qd, kd, vd, sl)
    torch.cuda.synchronize()
    assert torch.equal(a, b), "verification is not reproducible"
    ref = oracle.verify_attn(to_u16(q), to_u16(k), to_u16(v), np.array(lens, np.int32), n_q)
    what = f"17-32 rows, B={B} L={L_cap} G={G} n_q={n_q} lens={lens}"
    check_attention(bf16_out_to_f64(a), ref, what)
    check_attention(bf16_out_to_f64(c), ref, what + " (fewer stages)")
    check_attention(bf16_out_to_f64(pp), ref, what + " (per-pair kernel)")
    for i, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(a[i]) == 0


@pytest.mark.parametrize("seed", range(12))
def test_topk_scores_all_heads_fuzz(seed, monkeypatch):
    rng, B, L_cap, G, _, lens = _case(seed)
    H_kv, d = 8, 128
    H_q = G * H_kv
    top_k = int(rng.choice([1, 16, 100, 512]))
    g = torch.Generator().manual_seed(2000 + seed)
    q = torch.randn((B, 1, H_q, d), generator=g).to(torch.bfloat16).to(DEV)
    k = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16).to(DEV)
    v = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16).to(DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    idx_h = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    idx_p = torch.empty_like(idx_h)
    out_h = mb.magicdec_topk_draft_attn(q, k, v, sl, top_k, idx=idx_h)
    monkeypatch.setenv("MAGICDEC_TOPK_HEADS", "0")
    out_p = mb.magicdec_topk_draft_attn(q, k, v, sl, top_k, idx=idx_p)
    torch.cuda.synchronize()
    assert torch.equal(idx_h, idx_p)
    assert torch.equal(out_h, out_p)


def _draft_case(seed):
    """Draft attention over a compact cache [B, H_kv, cap, d]: random batch, head shape,
    capacity (one tile to several per pair) and lengths (empty, partial tile, full)."""
    rng = np.random.default_rng(9000 + seed)
    B = int(rng.integers(1, 20))
    H_kv = int(rng.choice([1, 2, 8]))
    G = int(rng.choice([1, 4, 5, 8]))
    d = int(rng.choice([64, 128]))
    cap = int(rng.choice([16, 64, 100, 512, 1000, 2048]))
    lens = [min(x, cap) for x in _lengths(rng, B, cap)]
    return B, G * H_kv, H_kv, d, cap, lens


@pytest.mark.parametrize("seed", range(16))
def test_draft_attn_fuzz(seed, monkeypatch):
    """The draft's per-pair kernel (head-major cache, L2 prefetch before the dependency
    wait, four stages or a random cap) against the oracle; empty rows are zero."""
    import oracle
    from parity_util import to_u16
    B, H_q, H_kv, d, cap, lens = _draft_case(seed)
    rng = np.random.default_rng(9500 + seed)
    monkeypatch.setenv("MAGICDEC_ATTN_STAGES", str(int(rng.choice([0, 2, 3]))))
    g = torch.Generator().manual_seed(4000 + seed)
    q = torch.randn((B, 1, H_q, d), generator=g).to(torch.bfloat16)
    kc = torch.randn((B, H_kv, cap, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, H_kv, cap, d), generator=g).to(torch.bfloat16)
    dl = torch.tensor(lens, dtype=torch.int32)
    out = mb.magicdec_draft_attn(q.to(DEV), kc.to(DEV), vc.to(DEV), dl.to(DEV))
    again = mb.magicdec_draft_attn(q.to(DEV), kc.to(DEV), vc.to(DEV), dl.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(out, again), "draft attention is not reproducible"
    ref = oracle.draft_attn(to_u16(q), to_u16(kc), to_u16(vc), dl.numpy())
    check_attention(bf16_out_to_f64(out), ref, f"draft B={B} H_q={H_q} H_kv={H_kv} d={d} cap={cap} lens={lens}")
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[b]) == 0


@pytest.mark.parametrize("seed", range(16))
def test_spec_accept_fuzz(seed):
    """Speculative accept on random batch, draft length, vocabulary (one statistics record
    to many, multiples of 4 or not), logit scale and draft noise, sampling or greedy; only
    the fp64 oracle's margins exclude a sequence."""
    from parity_util import check_accept, oracle_accept
    rng = np.random.default_rng(7000 + seed)
    B = int(rng.integers(1, 41))
    gamma = int(rng.integers(1, 9))
    V = int(rng.choice([5, 33, 1000, 4096, 4097, 8191, 20000, 50021]))
    sigma = float(rng.choice([0.5, 2.0, 4.0]))
    noise = float(rng.choice([0.1, 0.5, 1.5]))
    greedy = bool(rng.integers(0, 2))
    g = torch.Generator().manual_seed(7500 + seed)
    target = torch.randn((B, gamma + 1, V), generator=g) * sigma
    draft = target[:, :gamma] + torch.randn((B, gamma, V), generator=g) * noise
    tok = torch.distributions.Categorical(logits=draft).sample().to(torch.int32)
    if greedy:
        am = target[:, :gamma].argmax(-1).to(torch.int32)
        tok = torch.where(torch.rand(tok.shape, generator=g) < 0.7, am, tok)
    u_acc, u_res = torch.rand((B, gamma), generator=g), torch.rand((B,), generator=g)
    got = mb.magicdec_spec_accept(target.to(DEV), draft.to(DEV), tok.to(DEV), u_acc.to(DEV), u_res.to(DEV), greedy)
    torch.cuda.synchronize()
    t, d_, x, ua, ur = (a.numpy() for a in (target, draft, tok, u_acc, u_res))
    ref = oracle_accept(t, d_, x, ua, ur, greedy)
    what = f"accept B={B} gamma={gamma} V={V} sigma={sigma} noise={noise} greedy={greedy}"
    n_excl = check_accept(tuple(a.cpu().numpy() for a in got), ref, what, inputs=(t, d_, ur), greedy=greedy)
    assert n_excl <= max(2, B // 4), what


@pytest.mark.parametrize("seed", range(12))
def test_snapkv_select_fuzz(seed):
    """SnapKV selection (tensor-core window scores, max-pool, per-KV-head top-k) on random
    head shapes (G up to 8, w*G up to 256 window rows), head sizes, windows, pool widths,
    budgets and lengths (shorter than the budget, equal, longer), with and without planted
    heavy hitters, under the oracle's band rule."""
    import oracle
    from long_context_self_gb300 import synth
    from parity_util import check_topk, to_u16
    rng = np.random.default_rng(11000 + seed)
    B = int(rng.integers(1, 5))
    H_kv = int(rng.choice([1, 2, 8]))
    G = int(rng.choice([1, 2, 4, 5, 8]))
    d = int(rng.choice([64, 128]))
    w = int(rng.choice([w_ for w_ in (1, 4, 8, 16, 32) if w_ * G <= 256]))
    pool = int(rng.choice([1, 3, 5, 7, 9]))
    L_cap = int(rng.choice([100, 700, 3000, 9000]))
    budget = int(rng.integers(w, max(w + 1, L_cap // 2)))
    lens = []
    for _ in range(B):
        kind = int(rng.integers(0, 4))
        lens.append(L_cap if kind == 0 else int(rng.integers(0, budget + 1)) if kind == 1 else
                    budget if kind == 2 else int(rng.integers(budget + 1, L_cap + 1)))
    lens = [min(x, L_cap) for x in lens]
    heavy = bool(rng.integers(0, 2))
    wl = synth.Workload("fuzz", B=B, H_q=G * H_kv, H_kv=H_kv, d=d, L=L_cap, gamma=1, V=8, snap_window=w,
                        snap_pool=pool, snap_budget=budget, heavy_frac=0.005 if heavy else 0.0, seed=40 + seed)
    k, _, dirs = synth.kv_cache(wl, "cpu")
    q_win = synth.window_queries(wl, "cpu", heavy_dirs=dirs)
    sl = np.array(lens, np.int32)
    idx, n_sel = mb.magicdec_snapkv_select(q_win.to(DEV), k.to(DEV), torch.from_numpy(sl).to(DEV), w, pool, budget)
    torch.cuda.synchronize()
    idx_o, n_sel_o, pooled = oracle.snapkv_select(to_u16(q_win), to_u16(k), sl, pool, budget)
    band = check_topk(idx.cpu().numpy(), n_sel.cpu().numpy(), idx_o, n_sel_o, pooled, sl, w, budget)
    what = f"snapkv B={B} H_kv={H_kv} G={G} d={d} w={w} pool={pool} L={L_cap} budget={budget} lens={lens}"
    # The band must leave the comparison meaningful.  Positions tied exactly with the k-th
    # pooled score (planted heavy hitters share one key, so their pooled plateaus tie) may
    # all sit in it; beyond those, a plateau or two per (sequence, KV head), or 1 % of the
    # competing positions where the budget puts the threshold in the dense middle of the
    # score distribution.
    ties, compared = 0, 0
    for b, L in enumerate(lens):
        if L <= budget or budget == w:
            continue
        for h in range(H_kv):
            pl = pooled[b, h, :L - w]
            ties += int(np.count_nonzero(pl == np.sort(pl)[::-1][budget - w - 1]))
            compared += L - w
    assert band - ties <= max(2 * pool * B * H_kv + 8, 0.01 * compared), what


@pytest.mark.parametrize("seed", range(12))
def test_topk_draft_attn_fuzz(seed):
    """Top-K attention draft on random head shapes, head sizes, lengths (empty, shorter than
    top_k, long enough for the sampled threshold) and budgets, with a few dominant keys,
    against the oracle under the band rule."""
    import oracle
    from parity_util import check_topk_attn, to_u16
    rng = np.random.default_rng(13000 + seed)
    B = int(rng.integers(1, 6))
    H_kv = int(rng.choice([1, 2, 8]))
    G = int(rng.choice([1, 2, 4, 5, 8]))
    d = int(rng.choice([64, 128]))
    L_cap = int(rng.choice([64, 700, 3000, 9000, 20000]))
    top_k = int(rng.integers(1, min(L_cap, 4096) + 1))
    lens = _lengths(rng, B, L_cap)
    H_q = G * H_kv
    g = torch.Generator().manual_seed(13500 + seed)
    q = torch.randn((B, 1, H_q, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    k[:, ::int(rng.integers(50, 200))] *= 4
    sl = np.array(lens, np.int32)
    idx = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_topk_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(sl).to(DEV), top_k, idx=idx)
    torch.cuda.synchronize()
    ref, idx_o, scores = oracle.topk_attn(to_u16(q), to_u16(k), to_u16(v), sl, top_k, want_scores=True)
    what = f"topk B={B} H_q={H_q} H_kv={H_kv} d={d} L={L_cap} top_k={top_k} lens={lens}"
    check_topk_attn(bf16_out_to_f64(out), idx.cpu().numpy(), ref, idx_o, scores, sl, top_k, what,
                    qkv=(to_u16(q), to_u16(k), to_u16(v)))
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[b]) == 0


@pytest.mark.parametrize("seed", range(12))
def test_gather_kv_fuzz(seed):
    """Gather into the compact cache: random shapes, capacities, index lists (any order,
    repeats, -1 padding), bit for bit against the oracle."""
    import oracle
    from parity_util import to_u16
    rng = np.random.default_rng(15000 + seed)
    B = int(rng.integers(1, 6))
    H_kv = int(rng.choice([1, 2, 8]))
    d = int(rng.choice([64, 128]))
    L_cap = int(rng.choice([1, 17, 300, 4000]))
    n_idx = int(rng.integers(1, 700))
    cap = int(n_idx + rng.integers(0, 40))
    idx = rng.integers(0, L_cap, size=(B, H_kv, n_idx)).astype(np.int32)
    idx[rng.random(idx.shape) < 0.1] = -1
    g = torch.Generator().manual_seed(15500 + seed)
    k = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, L_cap, H_kv, d), generator=g).to(torch.bfloat16)
    kc, vc = mb.magicdec_gather_kv(k.to(DEV), v.to(DEV), torch.from_numpy(idx).to(DEV), cap)
    torch.cuda.synchronize()
    kc_o, vc_o = oracle.gather_kv(to_u16(k), to_u16(v), idx, cap)
    assert np.array_equal(to_u16(kc), kc_o)
    assert np.array_equal(to_u16(vc), vc_o)


@pytest.mark.parametrize("seed", range(10))
def test_pq_fuzz(seed, monkeypatch):
    """PQCache-style draft on random shapes: the encode (tensor-core or FMA) under the
    distance-margin rule, one Lloyd update bit for bit, and PQ attention over the oracle's
    codes under the band rule (G up to 8, d 64/128, C 2-256, budgets, ragged and empty
    lengths)."""
    import oracle
    from parity_util import check_topk_attn, to_u16
    rng = np.random.default_rng(17000 + seed)
    B = int(rng.integers(1, 4))
    H_kv = int(rng.choice([1, 2, 8]))
    G = int(rng.choice([1, 4, 5, 8]))
    d = int(rng.choice([64, 128]))
    M = d // 8
    C = int(rng.choice([2, 7, 32, 64, 200, 256]))
    L = int(rng.choice([100, 999, 3000]))
    top_k = int(rng.integers(1, min(L, 1024) + 1))
    lens = [x if x > 0 or rng.random() < 0.5 else 1 for x in _lengths(rng, B, L)]
    monkeypatch.setenv("MAGICDEC_PQ_TC", str(int(rng.integers(0, 2))))
    H_q = G * H_kv
    g = torch.Generator().manual_seed(17500 + seed)
    q = torch.randn((B, 1, H_q, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, L, H_kv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, L, H_kv, d), generator=g).to(torch.bfloat16)
    k[:, ::int(rng.integers(40, 120))] *= 3
    cb = rng.standard_normal((B, H_kv, M, C, 8)).astype(np.float32)
    what = f"pq B={B} H_q={H_q} H_kv={H_kv} d={d} C={C} L={L} top_k={top_k} lens={lens}"
    # encode under the margin rule
    codes_g = mb.magicdec_pq_encode(k.to(DEV), torch.from_numpy(cb).to(DEV))
    torch.cuda.synchronize()
    codes_o, gap = oracle.pq_encode(to_u16(k), cb, want_gap=True)
    kf = bf16_out_to_f64(k).reshape(B, L, H_kv, M, 8).transpose(0, 2, 1, 3, 4)
    kn = (kf ** 2).sum(-1)
    cn = (cb.astype(np.float64) ** 2).sum(-1)
    cbest = np.take_along_axis(cn[:, :, None, :, :], codes_o[..., None].astype(np.int64), axis=-1)[..., 0]
    margin = gap <= 1e-5 * (kn + cbest)
    assert np.array_equal(codes_g.cpu().numpy()[~margin], codes_o[~margin]), what
    # one Lloyd update over each sequence's own length, bit for bit
    sl = np.array(lens, np.int32)
    cb_g = torch.from_numpy(cb.copy()).to(DEV)
    mb.magicdec_pq_update(k.to(DEV), torch.from_numpy(sl).to(DEV), torch.from_numpy(codes_o).to(DEV), cb_g)
    torch.cuda.synchronize()
    cb2 = oracle.pq_update(to_u16(k), sl, codes_o, cb)
    np.testing.assert_array_equal(cb_g.cpu().numpy(), cb2, err_msg=what)
    # PQ attention over the oracle's codes for the updated codebook
    codes2, _ = oracle.pq_encode(to_u16(k), cb2)
    idx = torch.empty((B, H_q, top_k), dtype=torch.int32, device=DEV)
    out = mb.magicdec_pq_draft_attn(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(sl).to(DEV),
                                    torch.from_numpy(cb2).to(DEV), torch.from_numpy(codes2).to(DEV), top_k, idx=idx)
    torch.cuda.synchronize()
    ref, idx_o, approx = oracle.pq_attn(to_u16(q), to_u16(k), to_u16(v), sl, cb2, codes2, top_k, want_approx=True)
    # a small codebook (C = 2: at most 2^M distinct approximate scores) ties many positions
    # at the threshold, broken by rounding-level differences of the score sums: heads that
    # swap inside the band are checked over their own kept positions
    check_topk_attn(bf16_out_to_f64(out), idx.cpu().numpy(), ref, idx_o, approx, sl, top_k, what,
                    qkv=(to_u16(q), to_u16(k), to_u16(v)))
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.count_nonzero(out[b]) == 0
