"""Shared comparison rules for the GPU-vs-oracle parity tests.

Tolerances:
  * attention (bf16 inputs, fp32 accumulation, bf16 output) against the fp64
    oracle: max-abs error <= 2e-2 and relative L2 error <= 1e-2;
  * index, length and token outputs: bit-exact, except decisions the oracle
    itself reports as lying within 1e-4 of their boundary (the margin rule),
    which are counted and excluded;
  * SnapKV top-k: positions whose pooled oracle score lies within a relative
    1e-4 of the k-th largest score form the band; outside it membership must
    match exactly.
"""
import numpy as np
import torch

ATTN_MAX_ABS = 2e-2
ATTN_REL_L2 = 1e-2
MARGIN = 1e-4


def to_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_out_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_attention(got: np.ndarray, ref: np.ndarray, what: str = "attention"):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / denom if denom > 0 else float(np.linalg.norm(got))
    assert max_abs <= ATTN_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {ATTN_MAX_ABS}"
    assert rel <= ATTN_REL_L2, f"{what}: rel-L2 {rel:.3e} > {ATTN_REL_L2}"
    return max_abs, rel


def check_topk(idx_gpu: np.ndarray, n_sel_gpu: np.ndarray, idx_ora: np.ndarray, n_sel_ora: np.ndarray,
               pooled: np.ndarray, seq_len: np.ndarray, window: int, budget: int):
    """Compare SnapKV selections under the band rule; returns the number of band positions."""
    assert np.array_equal(n_sel_gpu, n_sel_ora)
    B, H, _ = idx_ora.shape
    band_total = 0
    for b in range(B):
        L = int(seq_len[b])
        for h in range(H):
            g, o = idx_gpu[b, h], idx_ora[b, h]
            if L <= budget:
                assert np.array_equal(g, o), (b, h)
                continue
            k_top = budget - window
            assert np.array_equal(g[k_top:], o[k_top:]), (b, h, "window part")
            gs = g[:k_top]
            assert np.all(np.diff(gs) > 0), (b, h, "not ascending")
            m = L - window
            pl = pooled[b, h, :m]
            tau = np.sort(pl)[::-1][k_top - 1]
            band = np.abs(pl - tau) <= MARGIN * abs(tau)
            band_total += int(band.sum())
            sel_g = np.zeros(m, bool)
            sel_g[gs] = True
            sel_o = np.zeros(m, bool)
            sel_o[o[:k_top]] = True
            assert np.array_equal(sel_g[~band], sel_o[~band]), (b, h, "membership outside band")
    return band_total


def check_topk_attn(out_gpu: np.ndarray, idx_gpu: np.ndarray, out_ora: np.ndarray, idx_ora: np.ndarray,
                    scores: np.ndarray, seq_len: np.ndarray, top_k: int, what: str = "topk attention"):
    """Top-K attention draft under the band rule.  Outside the band |s - tau| <= MARGIN * max(|tau|, 1)
    (tau = the oracle's top_k-th score) membership must match exactly; inside it only the count.
    Heads whose kept set differs from the oracle's (inside the band) are left out of the element-wise
    output comparison.  Returns (heads with a band swap, band positions)."""
    B, H, _ = idx_ora.shape
    swapped, band_total = 0, 0
    keep = np.ones((B, H), bool)
    for b in range(B):
        L = int(seq_len[b])
        n = min(L, top_k)
        for h in range(H):
            g, o = idx_gpu[b, h], idx_ora[b, h]
            assert np.all(g[n:] == -1), (b, h, "padding")
            if L <= top_k:
                assert np.array_equal(g, o), (b, h)
                continue
            gs = g[:n]
            assert np.all(np.diff(gs) > 0) and gs[0] >= 0 and gs[-1] < L, (b, h, "not ascending / out of range")
            sc = scores[b, h, :L]
            tau = np.sort(sc)[::-1][top_k - 1]
            band = np.abs(sc - tau) <= MARGIN * max(abs(tau), 1.0)
            band_total += int(band.sum())
            sel_g = np.zeros(L, bool)
            sel_g[gs] = True
            sel_o = np.zeros(L, bool)
            sel_o[o[:n]] = True
            assert np.array_equal(sel_g[~band], sel_o[~band]), (b, h, "membership outside band")
            if not np.array_equal(sel_g, sel_o):
                swapped += 1
                keep[b, h] = False
    check_attention(out_gpu[:, 0][keep], out_ora[:, 0][keep], what)
    return swapped, band_total


SAMPLE_EDGE_TOL = 1e-7     # inverse-CDF edge margin, relative to the total weight


def check_accept(gpu, ora, what="accept", inputs=None):
    """gpu / ora = (n_acc, out_tok, n_amb) numpy.

    Sequences the oracle or the kernel flags as taking a decision at its margin are
    excluded from the exact comparison.  When `inputs` = (target, draft, u_res) is
    given, a flagged sequence whose accepted prefix agrees must still have emitted a
    valid draw: a token whose oracle inverse-CDF interval lies within the edge
    margin of u * total."""
    import oracle
    n_acc_g, tok_g, amb_g = gpu
    n_acc_o, tok_o, amb_o = ora
    amb = (amb_o > 0) | (amb_g > 0)
    ok = ~amb
    assert np.array_equal(n_acc_g[ok], n_acc_o[ok]), f"{what}: n_acc differs"
    assert np.array_equal(tok_g[ok], tok_o[ok]), f"{what}: tokens differ"
    if inputs is not None:
        target, draft, u_res = inputs
        gamma = target.shape[1] - 1
        for b in np.nonzero(amb)[0]:
            a = int(n_acc_g[b])
            if a != n_acc_o[b] or not np.array_equal(tok_g[b, :a], tok_o[b, :a]):
                continue                      # an acceptance decision at its margin
            t = int(tok_g[b, a])
            if a < gamma:
                wts = oracle.resample_weights(target[b, a], draft[b, a])
            else:
                wts = oracle.resample_weights(target[b, gamma])
            cdf = np.cumsum(wts)
            W = cdf[-1]
            x = float(u_res[b]) * W
            lo = cdf[t - 1] if t > 0 else 0.0
            assert 0 <= t < len(wts) and wts[t] > 0, f"{what}: seq {b} drew a zero-weight token"
            assert lo - 1e-6 * W <= x <= cdf[t] + 1e-6 * W, f"{what}: seq {b} token {t} not a valid draw"
    return int(amb.sum())
