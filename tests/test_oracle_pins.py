"""Pins for the CPU oracle against facts fixed outside it.

Each test ties one oracle function to something other than its own formula: a
library routine on a special case (torch's scaled-dot-product attention,
softmax, max-pool), a brute-force enumeration, a closed form from the paper
(Eq. 1 of "MagicDec: Breaking the Latency-Throughput Tradeoff for Long Context
Generation with Speculative Decoding", section 3.1), or an invariant that any
correct implementation satisfies.  CPU only.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle


def bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(u: np.ndarray) -> np.ndarray:
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def sdpa_reference(q, k, v, mask):
    """torch SDPA in fp64 on CPU with a boolean keep-mask; rows with nothing visible -> 0."""
    qt, kt, vt = (torch.from_numpy(a) for a in (q, k, v))
    m = torch.from_numpy(mask)
    empty = ~m.any(-1, keepdim=True)
    m_safe = m | empty
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m_safe)
    return torch.where(empty, torch.zeros_like(out), out).numpy()


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------
@pytest.mark.parametrize("B,H_q,H_kv,d,L_cap,n_q", [(3, 8, 2, 64, 40, 4), (2, 5, 1, 32, 17, 3), (2, 4, 4, 16, 9, 1)])
def test_verify_attn_matches_torch_sdpa(B, H_q, H_kv, d, L_cap, n_q):
    rng = np.random.default_rng(7)
    q = bf16_bits(rng.standard_normal((B, n_q, H_q, d)))
    k = bf16_bits(rng.standard_normal((B, L_cap, H_kv, d)))
    v = bf16_bits(rng.standard_normal((B, L_cap, H_kv, d)))
    seq_len = rng.integers(1, L_cap + 1, size=B).astype(np.int32)
    seq_len[0] = L_cap
    if B > 1:
        seq_len[1] = max(1, n_q - 2)      # shorter than the speculated block: leading rows see nothing
    got = oracle.verify_attn(q, k, v, seq_len, n_q)

    G = H_q // H_kv
    qf = bits_to_f64(q).transpose(0, 2, 1, 3)                       # [B,H_q,n_q,d]
    kf = np.repeat(bits_to_f64(k).transpose(0, 2, 1, 3), G, axis=1)  # repeat_kv -> [B,H_q,L,d]
    vf = np.repeat(bits_to_f64(v).transpose(0, 2, 1, 3), G, axis=1)
    mask = np.zeros((B, 1, n_q, L_cap), bool)
    for b in range(B):
        for i in range(n_q):
            mask[b, 0, i, : max(0, seq_len[b] - n_q + i + 1)] = True
    ref = sdpa_reference(qf, kf, vf, np.broadcast_to(mask, (B, H_q, n_q, L_cap)).copy())
    np.testing.assert_allclose(got, ref.transpose(0, 2, 1, 3), rtol=1e-11, atol=1e-12)


def test_draft_attn_matches_torch_sdpa():
    rng = np.random.default_rng(8)
    B, H_q, H_kv, d, cap = 3, 8, 2, 64, 24
    q = bf16_bits(rng.standard_normal((B, 1, H_q, d)))
    kc = bf16_bits(rng.standard_normal((B, H_kv, cap, d)))
    vc = bf16_bits(rng.standard_normal((B, H_kv, cap, d)))
    dl = np.array([cap, 5, 0], np.int32)
    got = oracle.draft_attn(q, kc, vc, dl)
    G = H_q // H_kv
    qf = bits_to_f64(q).transpose(0, 2, 1, 3)
    kf = np.repeat(bits_to_f64(kc), G, axis=1)
    vf = np.repeat(bits_to_f64(vc), G, axis=1)
    mask = np.zeros((B, H_q, 1, cap), bool)
    for b in range(B):
        mask[b, :, :, : dl[b]] = True
    ref = sdpa_reference(qf, kf, vf, mask)
    np.testing.assert_allclose(got, ref.transpose(0, 2, 1, 3), rtol=1e-11, atol=1e-12)
    assert np.all(got[2] == 0.0)


def test_attention_special_cases():
    rng = np.random.default_rng(9)
    d, cap = 32, 16
    q = bf16_bits(rng.standard_normal((3, 1, 1, d)))
    kc = bf16_bits(rng.standard_normal((3, 1, cap, d)))
    vc = bf16_bits(rng.standard_normal((3, 1, cap, d)))
    # (a) a single visible row returns that value row exactly
    # (b) identical keys give the plain mean of the values
    kc[1, 0, :, :] = kc[1, 0, 0, :]
    # (c) one key aligned with a huge query dominates: output equals its value row
    q[2, 0, 0, :] = bf16_bits(np.full(d, 8.0))
    kc[2, 0, :, :] = bf16_bits(np.zeros((cap, d)))
    kc[2, 0, 11, :] = bf16_bits(np.full(d, 8.0))
    dl = np.array([1, cap, cap], np.int32)
    out = oracle.draft_attn(q, kc, vc, dl)
    vf = bits_to_f64(vc)
    np.testing.assert_array_equal(out[0, 0, 0], vf[0, 0, 0])
    np.testing.assert_allclose(out[1, 0, 0], vf[1, 0].mean(0), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out[2, 0, 0], vf[2, 0, 11], rtol=1e-12, atol=1e-12)


def test_split_merge_invariance():
    """Attention over a set of keys equals the log-sum-exp weighted combine of attention over
    any partition of that set (the identity a split-KV merge relies on).  Each part's
    normaliser Z = sum_j exp(s_j) is read from the oracle itself: a probe cache holding the
    part's keys plus one all-zero key whose value row is e_0 (every other value row zero)
    gives out[0] = 1 / (1 + Z), because the zero key's logit is 0 whatever the scale.  The
    recombined output must equal the oracle's unsplit result."""
    rng = np.random.default_rng(11)
    B, H_q, H_kv, d, n = 2, 8, 2, 64, 37
    q = bf16_bits(rng.standard_normal((B, 1, H_q, d)))
    kc = bf16_bits(rng.standard_normal((B, H_kv, n, d)))
    vc = bf16_bits(rng.standard_normal((B, H_kv, n, d)))
    full = oracle.draft_attn(q, kc, vc, np.full(B, n, np.int32))
    one = bf16_bits(np.ones(1))[0]
    for n_parts in (2, 3, 5):
        part_of = rng.integers(0, n_parts, n)
        part_of[:n_parts] = np.arange(n_parts)            # no part is empty
        num = np.zeros_like(full)
        den = np.zeros(full.shape[:3] + (1,))
        for p in range(n_parts):
            rows = np.flatnonzero(part_of == p)
            m = rows.size
            kp, vp = kc[:, :, rows], vc[:, :, rows]
            o_p = oracle.draft_attn(q, kp, vp, np.full(B, m, np.int32))
            k_probe = np.zeros((B, H_kv, m + 1, d), np.uint16)
            v_probe = np.zeros((B, H_kv, m + 1, d), np.uint16)
            k_probe[:, :, 1:] = kp
            v_probe[:, :, 0, 0] = one
            probe = oracle.draft_attn(q, k_probe, v_probe, np.full(B, m + 1, np.int32))
            z = 1.0 / probe[..., :1] - 1.0
            num += z * o_p
            den += z
        np.testing.assert_allclose(num / den, full, rtol=1e-10, atol=1e-12)


def test_verify_equals_draft_on_last_row():
    """The last verification row sees the whole sequence: it is plain decode attention over
    the full prefix, which the draft kernel computes when its cache is the identity gather."""
    rng = np.random.default_rng(10)
    B, H_q, H_kv, d, L, n_q = 2, 4, 2, 32, 30, 3
    q = bf16_bits(rng.standard_normal((B, n_q, H_q, d)))
    k = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    v = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    sl = np.array([L, 21], np.int32)
    ver = oracle.verify_attn(q, k, v, sl, n_q)
    kc = np.ascontiguousarray(k.transpose(0, 2, 1, 3))
    vc = np.ascontiguousarray(v.transpose(0, 2, 1, 3))
    dr = oracle.draft_attn(np.ascontiguousarray(q[:, n_q - 1 : n_q]), kc, vc, sl)
    np.testing.assert_allclose(ver[:, n_q - 1], dr[:, 0], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Top-K attention draft
# --------------------------------------------------------------------------
def _topk_reference(q, k, v, seq_len, top_k):
    """Scores by numpy einsum, the kept set by a lexicographic sort (score desc, position asc),
    the attention by torch SDPA in fp64 under that keep-mask."""
    B, _, H_q, d = q.shape
    H_kv = k.shape[2]
    G = H_q // H_kv
    qf = bits_to_f64(q)[:, 0]                                          # [B,H_q,d]
    kf = np.repeat(bits_to_f64(k).transpose(0, 2, 1, 3), G, axis=1)    # [B,H_q,L,d]
    vf = np.repeat(bits_to_f64(v).transpose(0, 2, 1, 3), G, axis=1)
    s = np.einsum("bhd,bhld->bhl", qf, kf) / math.sqrt(d)
    L_cap = k.shape[1]
    mask = np.zeros((B, H_q, 1, L_cap), bool)
    idx = np.full((B, H_q, top_k), -1, np.int32)
    for b in range(B):
        n = int(seq_len[b])
        for h in range(H_q):
            order = np.lexsort((np.arange(n), -s[b, h, :n]))[:top_k]
            keep = np.sort(order)
            mask[b, h, 0, keep] = True
            idx[b, h, : keep.size] = keep
    out = sdpa_reference(qf[:, :, None, :], kf, vf, mask)[:, :, 0]     # [B,H_q,d]
    return out[:, None], idx, s


@pytest.mark.parametrize("H_q,H_kv,d,top_k", [(8, 2, 32, 7), (5, 1, 64, 3), (4, 4, 16, 12)])
def test_topk_attn_matches_masked_sdpa(H_q, H_kv, d, top_k):
    rng = np.random.default_rng(21)
    B, L_cap = 4, 50
    q = bf16_bits(rng.standard_normal((B, 1, H_q, d)))
    k = bf16_bits(rng.standard_normal((B, L_cap, H_kv, d)))
    v = bf16_bits(rng.standard_normal((B, L_cap, H_kv, d)))
    seq_len = np.array([L_cap, top_k - 1 if top_k > 1 else 1, 0, 33], np.int32)
    got, idx, scores = oracle.topk_attn(q, k, v, seq_len, top_k, want_scores=True)
    ref, ref_idx, ref_s = _topk_reference(q, k, v, seq_len, top_k)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(idx, ref_idx)
    for b in range(B):
        n = int(seq_len[b])
        np.testing.assert_allclose(scores[b, :, :n], ref_s[b, :, :n], rtol=1e-12, atol=1e-13)
    assert np.all(got[2] == 0.0) and np.all(idx[2] == -1)


def test_topk_attn_with_budget_covering_prefix_is_dense_decode():
    """top_k >= len keeps every position: plain decode attention over the prefix."""
    rng = np.random.default_rng(22)
    B, H_q, H_kv, d, L = 2, 4, 2, 32, 30
    q = bf16_bits(rng.standard_normal((B, 1, H_q, d)))
    k = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    v = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    sl = np.array([L, 17], np.int32)
    got, idx, _ = oracle.topk_attn(q, k, v, sl, L)
    G = H_q // H_kv
    qf = bits_to_f64(q).transpose(0, 2, 1, 3)
    kf = np.repeat(bits_to_f64(k).transpose(0, 2, 1, 3), G, axis=1)
    vf = np.repeat(bits_to_f64(v).transpose(0, 2, 1, 3), G, axis=1)
    mask = np.zeros((B, H_q, 1, L), bool)
    for b in range(B):
        mask[b, :, :, : sl[b]] = True
    ref = sdpa_reference(qf, kf, vf, mask).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(idx[1, :, :17], np.broadcast_to(np.arange(17), (H_q, 17)))
    assert np.all(idx[1, :, 17:] == -1)


def test_topk_attn_ties_and_single_winner():
    rng = np.random.default_rng(23)
    d, L = 32, 20
    q = bf16_bits(rng.standard_normal((2, 1, 1, d)))
    k = bf16_bits(rng.standard_normal((2, L, 1, d)))
    v = bf16_bits(rng.standard_normal((2, L, 1, d)))
    # sequence 0: every key identical -> all scores tie -> the smallest positions win
    k[0, :, 0, :] = k[0, 0, 0, :]
    # sequence 1: key 13 aligned with the query and twice as long -> top-1 is position 13
    k[1, 13, 0, :] = bf16_bits(2.0 * bits_to_f64(q[1, 0, 0, :]))
    sl = np.array([L, L], np.int32)
    out5, idx5, _ = oracle.topk_attn(q[:1], k[:1], v[:1], sl[:1], 5)
    np.testing.assert_array_equal(idx5[0, 0], np.arange(5))
    np.testing.assert_allclose(out5[0, 0, 0], bits_to_f64(v[0, :5, 0, :]).mean(0), rtol=1e-12, atol=1e-13)
    out1, idx1, _ = oracle.topk_attn(q[1:], k[1:], v[1:], sl[1:], 1)
    assert idx1[0, 0, 0] == 13
    np.testing.assert_array_equal(out1[0, 0, 0], bits_to_f64(v[1, 13, 0, :]))


# --------------------------------------------------------------------------
# PQCache-style selection
# --------------------------------------------------------------------------
def test_pq_encode_matches_numpy_argmin():
    rng = np.random.default_rng(41)
    B, L, H_kv, d, M, C = 2, 50, 2, 32, 4, 10
    ds = d // M
    k = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    cb = rng.standard_normal((B, H_kv, M, C, ds)).astype(np.float32)
    cb[:, :, :, 7] = cb[:, :, :, 3]                      # duplicate: the smaller index must win
    codes, gap = oracle.pq_encode(k, cb, want_gap=True)
    kf = bits_to_f64(k).reshape(B, L, H_kv, M, ds)
    dist = ((kf[:, :, :, :, None, :] - cb.astype(np.float64).transpose(0, 1, 2, 3, 4)[:, None]
             .reshape(B, 1, H_kv, M, C, ds)) ** 2).sum(-1)
    np.testing.assert_array_equal(codes, np.argmin(dist, axis=-1).transpose(0, 2, 1, 3))   # head-major
    assert not np.any(codes == 7)
    srt = np.sort(dist, axis=-1)
    np.testing.assert_allclose(gap, (srt[..., 1] - srt[..., 0]).transpose(0, 2, 1, 3), rtol=1e-12, atol=1e-12)


def test_pq_update_matches_groupby_mean():
    rng = np.random.default_rng(42)
    B, L, H_kv, d, M, C = 2, 60, 2, 16, 2, 6
    ds = d // M
    k = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    codes = rng.integers(0, C - 1, size=(B, H_kv, L, M)).astype(np.uint8)   # centroid C-1 stays empty
    sl = np.array([L, 37], np.int32)
    cb0 = rng.standard_normal((B, H_kv, M, C, ds)).astype(np.float32)
    cb = oracle.pq_update(k, sl, codes, cb0)
    kf = bits_to_f64(k).reshape(B, L, H_kv, M, ds)
    for b in range(B):
        for h in range(H_kv):
            for m in range(M):
                for c in range(C):
                    sel = codes[b, h, : sl[b], m] == c
                    if sel.any():
                        want = kf[b, : sl[b]][sel, h, m].mean(0).astype(np.float32)
                        np.testing.assert_array_equal(cb[b, h, m, c], want)
                    else:
                        np.testing.assert_array_equal(cb[b, h, m, c], cb0[b, h, m, c])


def test_pq_attn_with_the_keys_as_codebook_is_topk_attention():
    """One centroid per position equal to that key: approximate scores are exact, so PQ attention
    reduces to Top-K attention (itself pinned to masked SDPA)."""
    rng = np.random.default_rng(43)
    B, H_q, H_kv, d, L, M, top_k = 2, 8, 2, 32, 40, 4, 9
    ds = d // M
    q = bf16_bits(rng.standard_normal((B, 1, H_q, d)))
    k = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    v = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    cb = bits_to_f64(k).reshape(B, L, H_kv, M, ds).transpose(0, 2, 3, 1, 4).astype(np.float32)   # C = L
    codes = np.broadcast_to(np.arange(L, dtype=np.uint8)[None, None, :, None], (B, H_kv, L, M)).copy()
    sl = np.array([L, 23], np.int32)
    out, idx, _ = oracle.pq_attn(q, k, v, sl, cb, codes, top_k)
    ref, ref_idx, _ = oracle.topk_attn(q, k, v, sl, top_k)
    np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_pq_attn_matches_masked_sdpa():
    rng = np.random.default_rng(44)
    B, H_q, H_kv, d, L, M, C, top_k = 3, 8, 2, 32, 70, 4, 16, 11
    ds = d // M
    G = H_q // H_kv
    q = bf16_bits(rng.standard_normal((B, 1, H_q, d)))
    k = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    v = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    cb = rng.standard_normal((B, H_kv, M, C, ds)).astype(np.float32)
    codes = rng.integers(0, C, size=(B, H_kv, L, M)).astype(np.uint8)
    sl = np.array([L, 5, 40], np.int32)
    out, idx, approx = oracle.pq_attn(q, k, v, sl, cb, codes, top_k, want_approx=True)
    qf = bits_to_f64(q)[:, 0].reshape(B, H_q, M, ds)
    cbf = np.repeat(cb.astype(np.float64), G, axis=1)                          # [B,H_q,M,C,ds]
    lut = np.einsum("bhmi,bhmci->bhmc", qf, cbf) / math.sqrt(d)
    codes_q = np.repeat(codes, G, axis=1)                                      # [B,H_q,L,M]
    a = np.take_along_axis(lut[:, :, None, :, :], codes_q[..., None].astype(np.int64), axis=-1)[..., 0].sum(-1)
    kf = np.repeat(bits_to_f64(k).transpose(0, 2, 1, 3), G, axis=1)
    vf = np.repeat(bits_to_f64(v).transpose(0, 2, 1, 3), G, axis=1)
    mask = np.zeros((B, H_q, 1, L), bool)
    want_idx = np.full((B, H_q, top_k), -1, np.int32)
    for b in range(B):
        n = int(sl[b])
        for h in range(H_q):
            keep = np.sort(np.lexsort((np.arange(n), -a[b, h, :n]))[:top_k])
            mask[b, h, 0, keep] = True
            want_idx[b, h, : keep.size] = keep
            np.testing.assert_allclose(approx[b, h, :n], a[b, h, :n], rtol=1e-12, atol=1e-12)
    ref = sdpa_reference(bits_to_f64(q).transpose(0, 2, 1, 3), kf, vf, mask).transpose(0, 2, 1, 3)
    np.testing.assert_array_equal(idx, want_idx)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_pq_lloyd_steps_recover_planted_clusters():
    """Sub-vectors drawn around 6 well-separated prototypes per subspace: from one member of each
    cluster as the initial centroids, encode + update twice labels every key by its prototype and the
    centroids settle on the cluster means."""
    rng = np.random.default_rng(45)
    B, L, H_kv, d, M, C = 1, 300, 2, 16, 2, 6
    ds = d // M
    proto = rng.standard_normal((B, H_kv, M, C, ds)) * 4.0
    label = rng.integers(0, C, size=(B, L, H_kv, M))
    label[:, :C] = np.arange(C)[None, :, None, None]                        # positions 0..C-1 seed the clusters
    sub = np.take_along_axis(proto[:, None], label.reshape(B, L, H_kv, M, 1, 1).repeat(ds, -1), axis=4)[..., 0, :]
    k = bf16_bits((sub + 0.05 * rng.standard_normal(sub.shape)).reshape(B, L, H_kv, d))
    kf = bits_to_f64(k).reshape(B, L, H_kv, M, ds)
    cb = kf[:, :C].transpose(0, 2, 3, 1, 4).astype(np.float32).copy()     # [B,H_kv,M,C,ds]
    sl = np.array([L], np.int32)
    for _ in range(2):
        codes, _ = oracle.pq_encode(k, cb)
        cb = oracle.pq_update(k, sl, codes, cb)
    np.testing.assert_array_equal(codes, label.transpose(0, 2, 1, 3))
    for h in range(H_kv):
        for m in range(M):
            for c in range(C):
                np.testing.assert_allclose(cb[0, h, m, c], kf[0][label[0, :, h, m] == c, h, m].mean(0),
                                           rtol=1e-6, atol=1e-6)


# --------------------------------------------------------------------------
# Draft-cache update (append / rollback)
# --------------------------------------------------------------------------
def _encoded_cache(B, L, H_kv, d, version):
    """Rows whose first channels spell (position // 256, position % 256, head, version): exact in bf16."""
    k = np.zeros((B, L, H_kv, d), np.float32)
    pos = np.arange(L)
    k[:, :, :, 0] = (pos // 256)[None, :, None]
    k[:, :, :, 1] = (pos % 256)[None, :, None]
    k[:, :, :, 2] = np.arange(H_kv)[None, None, :]
    k[:, :, :, 3] = version
    return bf16_bits(k)


def _decode(kc_row):
    f = bits_to_f64(kc_row)
    return int(f[0]) * 256 + int(f[1]), int(f[2]), int(f[3])


def _slots(kc, b, n):
    """(positions, versions) held by slots [0, n) of every head of sequence b (heads must agree)."""
    out = []
    for h in range(kc.shape[1]):
        rows = [_decode(kc[b, h, i]) for i in range(n)]
        assert all(r[1] == h for r in rows)
        out.append(sorted((r[0], r[2]) for r in rows))
    assert all(o == out[0] for o in out)
    return [p for p, _ in out[0]], [v for _, v in out[0]]


def test_draft_cache_ring_tracks_streaming_selection():
    """Drafting appends, then after each verification the cache is refreshed to the accepted length:
    the occupied slots always hold exactly the StreamingLLM selection, as verified rows."""
    rng = np.random.default_rng(31)
    B, H_kv, d, L, S, W, gamma = 3, 2, 16, 400, 4, 20, 3
    drafted = _encoded_cache(B, L, H_kv, d, 0)
    verified = _encoded_cache(B, L, H_kv, d, 1)
    kc = np.zeros((B, H_kv, S + W, d), np.uint16)
    vc = np.zeros_like(kc)
    origin = np.full(B, S, np.int32)
    length = np.array([2, 10, 100], np.int32)
    z = np.zeros(B, np.int32)
    dl, skipped = oracle.draft_cache_update(verified, verified, kc, vc, z, z, length, origin, None, W)
    assert skipped == 0
    for _ in range(30):
        for i in range(gamma):           # drafted rows of the sparse model
            dl, _ = oracle.draft_cache_update(drafted, drafted, kc, vc, length + i, length + i, length + i + 1,
                                              origin, None, W)
            for b in range(B):
                idx, n_sel = oracle.streaming_select(length[b:b + 1] + i + 1, 1, S, W)
                pos, _ = _slots(kc, b, dl[b])
                assert pos == sorted(idx[0, 0, : n_sel[0]].tolist())
        n_acc = rng.integers(0, gamma + 1, size=B).astype(np.int32)
        new = length + n_acc + 1
        dl, skipped = oracle.draft_cache_update(verified, verified, kc, vc, length, length + gamma, new, origin,
                                                None, W)
        assert skipped == 0
        for b in range(B):
            idx, n_sel = oracle.streaming_select(new[b:b + 1], 1, S, W)
            assert dl[b] == n_sel[0]
            pos, ver = _slots(kc, b, dl[b])
            assert pos == sorted(idx[0, 0, : n_sel[0]].tolist())
            assert all(x == 1 for x in ver), "a drafted row survived verification"
        length = new


def test_draft_cache_rollback_restores_the_ring():
    B, H_kv, d, L, S, W = 2, 1, 16, 200, 3, 16
    full = _encoded_cache(B, L, H_kv, d, 1)
    kc = np.zeros((B, H_kv, S + W, d), np.uint16)
    vc = np.zeros_like(kc)
    origin = np.full(B, S, np.int32)
    z = np.zeros(B, np.int32)
    length = np.array([60, 18], np.int32)
    oracle.draft_cache_update(full, full, kc, vc, z, z, length, origin, None, W)
    before, dl0 = kc.copy(), None
    for grow in (1, 5, W + 7):
        dl, _ = oracle.draft_cache_update(full, full, kc, vc, length, length, length + grow, origin, None, W)
        dl, _ = oracle.draft_cache_update(full, full, kc, vc, length, length + grow, length, origin, None, W)
        for b in range(B):
            np.testing.assert_array_equal(kc[b, :, : dl[b]], before[b, :, : dl[b]])
            np.testing.assert_array_equal(vc[b, :, : dl[b]], before[b, :, : dl[b]])


def test_draft_cache_linear_appends_after_selection():
    rng = np.random.default_rng(32)
    B, H_kv, d, L, L0, n_sel, cap = 2, 2, 16, 300, 120, 40, 100
    full = _encoded_cache(B, L, H_kv, d, 1)
    kc = np.zeros((B, H_kv, cap, d), np.uint16)
    vc = np.zeros_like(kc)
    sel = np.stack([np.sort(rng.choice(L0, n_sel, replace=False)) for _ in range(B)]).astype(np.int32)
    idx = np.repeat(sel[:, None, :], H_kv, axis=1)
    kc0, vc0 = oracle.gather_kv(full, full, idx, cap)
    kc[:], vc[:] = kc0, vc0
    origin = np.full(B, L0, np.int32)
    base = np.full(B, n_sel, np.int32)
    length = np.full(B, L0, np.int32)
    for step in range(6):
        new = length + rng.integers(1, 5, size=B).astype(np.int32)
        dl, skipped = oracle.draft_cache_update(full, full, kc, vc, length, length, new, origin, base, 0)
        assert skipped == 0
        for b in range(B):
            pos, _ = _slots(kc, b, dl[b])
            assert pos == sorted(sel[b].tolist() + list(range(L0, int(new[b]))))
        length = new
    # capacity: an append past cap is skipped, reported, and draft_len clamps to cap
    big = np.full(B, L0 + (cap - n_sel) + 3, np.int32)
    dl, skipped = oracle.draft_cache_update(full, full, kc, vc, length, length, big, origin, base, 0)
    assert skipped == 3 * B and np.all(dl == cap)


# --------------------------------------------------------------------------
# StreamingLLM selection and gather
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n_sink,n_recent", [(4, 60), (16, 496), (0, 8), (5, 0)])
def test_streaming_select_is_sinks_plus_recent(n_sink, n_recent):
    lens = np.array([0, 1, 3, n_sink + n_recent - 1, n_sink + n_recent, n_sink + n_recent + 1, 1000, 32000], np.int32)
    idx, n_sel = oracle.streaming_select(lens, 3, n_sink, n_recent)
    for b, L in enumerate(lens):
        want = sorted(set(range(min(n_sink, L))) | set(range(max(0, L - n_recent), L)))
        assert n_sel[b] == len(want)
        for h in range(3):
            assert list(idx[b, h, : n_sel[b]]) == want
            assert np.all(idx[b, h, n_sel[b]:] == -1)
        if L <= n_sink + n_recent:
            assert want == list(range(L))


def test_gather_identity_and_padding():
    rng = np.random.default_rng(11)
    B, L, H, d, cap = 2, 12, 3, 16, 14
    k = bf16_bits(rng.standard_normal((B, L, H, d)))
    v = bf16_bits(rng.standard_normal((B, L, H, d)))
    idx = np.broadcast_to(np.arange(L, dtype=np.int32), (B, H, L)).copy()
    kc, vc = oracle.gather_kv(k, v, idx, cap)
    np.testing.assert_array_equal(kc[:, :, :L], k.transpose(0, 2, 1, 3))
    np.testing.assert_array_equal(vc[:, :, :L], v.transpose(0, 2, 1, 3))
    idx2 = idx.copy()
    idx2[:, :, 5:] = -1
    kc2, _ = oracle.gather_kv(k, v, idx2, cap)
    assert np.all(kc2[:, :, 5:L] == 0)


# --------------------------------------------------------------------------
# SnapKV
# --------------------------------------------------------------------------
def _snap_inputs(B=2, H_q=4, H_kv=1, d=64, L=256, w=16, seed=12):
    rng = np.random.default_rng(seed)
    q_win = bf16_bits(rng.standard_normal((B, w, H_q, d)))
    k = bf16_bits(rng.standard_normal((B, L, H_kv, d)))
    return q_win, k


def test_snapkv_scores_match_torch_softmax():
    q_win, k = _snap_inputs(B=2, H_q=4, H_kv=2, d=32, L=50, w=8)
    sl = np.array([50, 31], np.int32)
    got = oracle.snapkv_scores(q_win, k, sl)
    B, w, H_q, d = q_win.shape
    H_kv = k.shape[2]
    G = H_q // H_kv
    for b in range(B):
        L = sl[b]
        for h in range(H_kv):
            qf = torch.from_numpy(bits_to_f64(q_win[b, :, h * G : (h + 1) * G]))   # [w,G,d]
            kf = torch.from_numpy(bits_to_f64(k[b, :L, h]))                      # [L,d]
            s = torch.einsum("wgd,ld->gwl", qf, kf) / math.sqrt(d)
            pos = torch.arange(L)
            qpos = L - w + torch.arange(w)
            s = s.masked_fill(pos[None, None, :] > qpos[None, :, None], float("-inf"))
            ref = torch.softmax(s, dim=-1).sum(dim=(0, 1)).numpy()
            np.testing.assert_allclose(got[b, h, :L], ref, rtol=1e-11, atol=1e-14)
            assert np.all(got[b, h, L:] == 0)
            # every softmax row sums to one: the scores sum to w * G
            assert abs(got[b, h].sum() - w * G) < 1e-9


def test_maxpool_matches_torch_and_naive():
    rng = np.random.default_rng(13)
    x = rng.standard_normal(101)
    x[40:45] = 3.0                                                     # a plateau: exact ties
    got = oracle.maxpool1d(x, 7)
    ref = torch.nn.functional.max_pool1d(torch.from_numpy(x)[None, None], 7, stride=1, padding=3)[0, 0].numpy()
    np.testing.assert_array_equal(got, ref)
    naive = [max(x[max(0, j - 3) : j + 4]) for j in range(len(x))]
    np.testing.assert_array_equal(got, naive)


def test_snapkv_select_equals_exhaustive_sort():
    q_win, k = _snap_inputs()
    sl = np.array([256, 200], np.int32)
    w, pool, budget = 16, 7, 64
    idx, n_sel, pooled = oracle.snapkv_select(q_win, k, sl, pool, budget)
    scores = oracle.snapkv_scores(q_win, k, sl)
    for b in range(2):
        L = sl[b]
        m = L - w
        pl = np.array([max(scores[b, 0, max(0, j - 3) : min(m, j + 4)]) for j in range(m)])
        np.testing.assert_array_equal(pooled[b, 0, :m], pl)
        order = np.lexsort((np.arange(m), -pl))           # score descending, position ascending
        want = sorted(order[: budget - w].tolist()) + list(range(m, L))
        assert n_sel[b] == budget
        assert idx[b, 0].tolist() == want


def test_snapkv_keeps_planted_heavy_hitter_and_neighbours():
    B, H_q, H_kv, d, L, w = 1, 4, 1, 64, 256, 16
    rng = np.random.default_rng(14)
    hhat = rng.standard_normal(d)
    hhat /= np.linalg.norm(hhat)
    k = rng.standard_normal((B, L, H_kv, d)) * 0.2
    k[0, 100, 0] = hhat * 8.0 * math.sqrt(d)
    qw = np.broadcast_to(hhat * math.sqrt(d), (B, w, H_q, d))
    idx, n_sel, _ = oracle.snapkv_select(bf16_bits(qw), bf16_bits(k), np.array([L], np.int32), 7, 24)
    chosen = set(idx[0, 0, : n_sel[0]].tolist())
    assert set(range(97, 104)) <= chosen
    assert set(range(L - w, L)) <= chosen


def test_snapkv_short_sequence_keeps_everything():
    q_win, k = _snap_inputs()
    sl = np.array([64, 10], np.int32)
    idx, n_sel, _ = oracle.snapkv_select(q_win, k, sl, 7, 64)
    assert n_sel.tolist() == [64, 10]
    assert idx[0, 0].tolist() == list(range(64))
    assert idx[1, 0].tolist() == list(range(10)) + [-1] * 54


# --------------------------------------------------------------------------
# Speculative sampling
# --------------------------------------------------------------------------
def _softmax(x):
    e = np.exp(x - x.max())
    return e / e.sum()


def _pieces(breaks):
    pts = sorted(set([0.0, 1.0] + [float(b) for b in breaks if 0.0 < b < 1.0]))
    return [((lo + hi) / 2.0, hi - lo) for lo, hi in zip(pts[:-1], pts[1:]) if hi > lo]


def _cum_breaks(wts):
    W = wts.sum()
    return [] if W <= 0 else list(np.cumsum(wts)[:-1] / W)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_spec_sampling_exact_enumeration_gamma1(seed):
    """Integrate the accept/resample rule over u exactly: the first emitted token is ~ p_1,
    and the bonus token after an acceptance is ~ p_2 (Leviathan et al.'s guarantee)."""
    rng = np.random.default_rng(100 + seed)
    V = 4
    tl = (rng.standard_normal((2, V)) * 1.5).astype(np.float32)
    dl = (rng.standard_normal((1, V)) * 1.5).astype(np.float32)
    p1, p2 = _softmax(tl[0].astype(np.float64)), _softmax(tl[1].astype(np.float64))
    q1 = _softmax(dl[0].astype(np.float64))
    res_breaks = _cum_breaks(np.maximum(p1 - q1, 0)) + _cum_breaks(p2)
    rows, weights = [], []
    for x in range(V):
        for ua, wa in _pieces([p1[x] / q1[x]]):
            for ur, wr in _pieces(res_breaks):
                rows.append((x, ua, ur))
                weights.append(q1[x] * wa * wr)
    n = len(rows)
    target = np.broadcast_to(tl, (n, 2, V)).copy()
    draft = np.broadcast_to(dl, (n, 1, V)).copy()
    toks = np.array([[r[0]] for r in rows], np.int32)
    ua = np.array([[r[1]] for r in rows], np.float32)
    ur = np.array([r[2] for r in rows], np.float32)
    n_acc, out, _ = oracle.spec_accept(target, draft, toks, ua, ur, greedy=False)
    wts = np.array(weights)
    first = np.zeros(V)
    np.add.at(first, out[:, 0], wts)
    np.testing.assert_allclose(first, p1, atol=1e-12)
    acc = n_acc == 1
    bonus = np.zeros(V)
    np.add.at(bonus, out[acc, 1], wts[acc])
    np.testing.assert_allclose(bonus / wts[acc].sum(), p2, atol=1e-12)
    assert np.all(out[~acc, 1] == -1)


def test_spec_sampling_exact_enumeration_gamma2():
    rng = np.random.default_rng(200)
    V = 4
    tl = (rng.standard_normal((3, V)) * 1.2).astype(np.float32)
    dl = (rng.standard_normal((2, V)) * 1.2).astype(np.float32)
    p = [_softmax(t.astype(np.float64)) for t in tl]
    q = [_softmax(t.astype(np.float64)) for t in dl]
    res_breaks = (_cum_breaks(np.maximum(p[0] - q[0], 0)) + _cum_breaks(np.maximum(p[1] - q[1], 0))
                  + _cum_breaks(p[2]))
    rows, weights = [], []
    for x1, x2 in itertools.product(range(V), range(V)):
        for u1, w1 in _pieces([p[0][x1] / q[0][x1]]):
            for u2, w2 in _pieces([p[1][x2] / q[1][x2]]):
                for ur, wr in _pieces(res_breaks):
                    rows.append((x1, x2, u1, u2, ur))
                    weights.append(q[0][x1] * q[1][x2] * w1 * w2 * wr)
    n = len(rows)
    r = np.array(rows)
    n_acc, out, _ = oracle.spec_accept(np.broadcast_to(tl, (n, 3, V)).copy(), np.broadcast_to(dl, (n, 2, V)).copy(),
                                       r[:, :2].astype(np.int32), r[:, 2:4].astype(np.float32),
                                       r[:, 4].astype(np.float32), greedy=False)
    wts = np.array(weights)
    for pos in range(3):
        sel = n_acc >= pos
        dist = np.zeros(V)
        np.add.at(dist, out[sel, pos], wts[sel])
        np.testing.assert_allclose(dist / wts[sel].sum(), p[pos], atol=1e-12)


def test_greedy_mode_is_argmax_chain():
    rng = np.random.default_rng(300)
    B, gamma, V = 64, 4, 50
    target = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    am = target.argmax(-1)
    toks = am[:, :gamma].copy()
    flip = rng.random((B, gamma)) < 0.3
    toks[flip] = (toks[flip] + 1) % V
    n_acc, out, _ = oracle.spec_accept(target, None, toks.astype(np.int32), np.zeros((B, gamma), np.float32),
                                       np.zeros(B, np.float32), greedy=True)
    for b in range(B):
        k = 0
        while k < gamma and toks[b, k] == am[b, k]:
            k += 1
        assert n_acc[b] == k
        assert out[b, :k].tolist() == toks[b, :k].tolist()
        assert out[b, k] == am[b, k]
        assert np.all(out[b, k + 1:] == -1)


@pytest.mark.parametrize("gamma", [1, 3, 5])
def test_expected_tokens_matches_eq1(gamma):
    """Identical target and draft distributions at every position: acceptances are i.i.d. with
    probability alpha = sum_t min(p_t, q_t), so E[#generated] = (1 - alpha^(gamma+1)) / (1 - alpha)
    (Eq. 1, section 3.1)."""
    rng = np.random.default_rng(400 + gamma)
    V, B = 12, 40000
    tl = (rng.standard_normal(V) * 1.5).astype(np.float32)
    dl = (tl + rng.standard_normal(V) * 0.8).astype(np.float32)
    p, q = _softmax(tl.astype(np.float64)), _softmax(dl.astype(np.float64))
    alpha = np.minimum(p, q).sum()
    toks = rng.choice(V, size=(B, gamma), p=q).astype(np.int32)
    n_acc, _, _ = oracle.spec_accept(np.broadcast_to(tl, (B, gamma + 1, V)).copy(),
                                     np.broadcast_to(dl, (B, gamma, V)).copy(), toks,
                                     rng.random((B, gamma)).astype(np.float32), rng.random(B).astype(np.float32),
                                     greedy=False)
    gen = n_acc + 1.0
    omega = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(gen.mean() - omega) < 4 * gen.std() / math.sqrt(B)


def test_spec_accept_margins_at_planted_boundaries():
    """The per-decision margins the parity tests exclude by, on inputs whose p, q and running
    sums are exact dyadic numbers (logits 0 and -inf), so each margin is known in closed form:
    target p = 1/4 each; draft q = (1/2, 1/2, 0, 0); residual max(0, p - q) = (0, 0, 1/4, 1/4)."""
    V = 4
    target = np.zeros((4, 2, V), np.float32)
    draft = np.tile(np.array([0, 0, -np.inf, -np.inf], np.float32), (4, 1, 1))
    tok = np.array([[0], [0], [2], [-1]], np.int32)
    u_acc = np.array([[0.5 + 2.0 ** -24], [0.375], [0.9], [0.9]], np.float32)
    u_res = np.array([0.25, 0.5 + 2.0 ** -24, 0.125, 0.75], np.float32)
    n_acc, out, amb, acc_m, draw_m = oracle.spec_accept(target, draft, tok, u_acc, u_res, False, want_margins=True)
    # seq 0: p/q = 1/2, u just above -> reject at margin 2^-24 (one fp32 ulp); draw 0.25*W = 1/8 lands in token 2,
    #        1/8 from both of its edges (1/4 of W = 1/2)
    # seq 1: accepted 1/8 from the boundary; the bonus draw from p lands 2^-24 past the 1/2 edge
    # seq 2: q(x) = 0 < p(x): accepted exactly; bonus 1/8 -> token 0, 1/8 from its upper edge
    # seq 3: x out of range: rejected exactly; 3/8 lands in token 3, 1/8 past its lower edge
    assert n_acc.tolist() == [0, 1, 1, 0]
    assert out.tolist() == [[2, -1], [0, 2], [2, 0], [3, -1]]
    assert amb.tolist() == [1, 1, 0, 0]
    assert acc_m[0, 0] == 2.0 ** -24 and acc_m[1, 0] == 0.125
    assert np.isinf(acc_m[2, 0]) and np.isinf(acc_m[3, 0])
    assert np.all(np.isnan(acc_m[:, 1]))
    assert draw_m.tolist() == [0.25, 2.0 ** -24, 0.125, 0.25]
    # greedy: the top-2 logit gap at each decided position, the bonus row included
    tg = np.array([[[1.0, 1.0 - 2.0 ** -16, 0, 0], [0, 3, 1, 0]]], np.float32)
    n_acc, out, amb, acc_m, draw_m = oracle.spec_accept(tg, None, np.array([[0]], np.int32),
                                                        np.zeros((1, 1), np.float32), np.zeros(1, np.float32), True,
                                                        want_margins=True)
    assert n_acc.tolist() == [1] and out.tolist() == [[0, 1]] and amb.tolist() == [1]
    assert acc_m.tolist() == [[2.0 ** -16, 2.0]] and np.isnan(draw_m[0])


def test_step_lengths_follow_the_token_sequence():
    """A sequence simulated token by token: a speculative step caches the pending token and the
    accepted drafts and leaves the emitted token pending, so the cached length grows by
    n_acc + 1; draft step g of the next step appends the (g+1)-th new position.  Lengths stop
    at the cache capacity."""
    rng = np.random.default_rng(12)
    B, gamma, L_cap = 9, 4, 600
    cached = [list(range(int(n))) for n in rng.integers(0, 560, B)]
    lens = np.array([len(c) for c in cached], np.int32)
    for _ in range(12):
        n_acc = rng.integers(0, gamma + 1, B).astype(np.int32)
        got, table = oracle.step_lengths(lens, gamma, L_cap, n_acc)
        for b in range(B):
            block = [len(cached[b]) + i for i in range(gamma + 1)]    # pending token + gamma drafts
            kept = block[: n_acc[b] + 1]
            cached[b] = (cached[b] + kept)[:L_cap]
            assert got[b] == len(cached[b])
            # the next step's draft appends positions len, len+1, ... and verifies len .. len+gamma
            nxt = [p for p in range(len(cached[b]), len(cached[b]) + gamma + 2)]
            assert table[:, b].tolist() == [min(p, L_cap) for p in nxt]
        lens = got
    same, t0 = oracle.step_lengths(lens, gamma, L_cap)
    assert np.array_equal(same, lens) and np.array_equal(t0[0], lens)
