"""Shared comparison rules for the GPU-vs-oracle parity tests.

Tolerances:
  * attention (bf16 inputs, fp32 accumulation, bf16 output) against the fp64
    oracle: max-abs error <= 2e-2 and relative L2 error <= 1e-2;
  * index, length and token outputs: bit-exact, except decisions the fp64
    oracle itself reports as lying within 1e-4 of their boundary (the margin
    rule), which are counted and excluded -- never on the kernel's say-so;
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
            m = L - window
            assert np.all(np.diff(gs) > 0), (b, h, "not ascending")
            assert gs.size == 0 or (gs[0] >= 0 and gs[-1] < m), (b, h, "kept position out of [0, L - window)")
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
                    scores: np.ndarray, seq_len: np.ndarray, top_k: int, what: str = "topk attention", qkv=None):
    """Top-K attention draft under the band rule.  Outside the band |s - tau| <= MARGIN * max(|tau|, 1)
    (tau = the oracle's top_k-th score) membership must match exactly; inside it only the count.
    A head whose kept set differs from the oracle's (inside the band, so the kernel's set is
    as valid) is compared with the oracle's attention over the kernel's own kept positions when
    `qkv` = (q, k, v) (bf16 bits, [B, 1, H_q, d] and [B, L, H_kv, d]) is given, and left out of
    the element-wise comparison otherwise.  Returns (heads with a band swap, band positions)."""
    B, H, _ = idx_ora.shape
    swapped, band_total = 0, 0
    keep = np.ones((B, H), bool)
    own = []
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
                own.append((b, h, gs))
    check_attention(out_gpu[:, 0][keep], out_ora[:, 0][keep], what)
    if qkv is not None and own:
        import oracle
        q, k, v = qkv
        G = H // k.shape[2]
        got, ref = [], []
        for b, h, gs in own:
            kc = np.ascontiguousarray(k[b, gs, h // G][None, None])       # [1, 1, n, d]: the kernel's rows
            vc = np.ascontiguousarray(v[b, gs, h // G][None, None])
            qh = np.ascontiguousarray(q[b:b + 1, :, h:h + 1])
            ref.append(oracle.draft_attn(qh, kc, vc, np.array([gs.size], np.int32))[0, 0, 0])
            got.append(out_gpu[b, 0, h])
        check_attention(np.array(got), np.array(ref), what + " (heads with a band swap, over their own kept set)")
    return swapped, band_total


SAMPLE_EDGE_TOL = 1e-7     # inverse-CDF edge margin, relative to the total weight
# How far past a threshold the kernel's own margin estimate may still flag a decision.  Its
# p/q ratios carry ~1e-7 relative error (fp32 exponentials, fp64 normalisers): 1 % of the 1e-4
# acceptance margin.  Its inverse-CDF running sums add fp32 exponentials with ~2e-7 relative
# error each, which at a 16-token vocabulary can move an edge by ~1e-7 of the total: 3x the
# 1e-7 edge margin.
KERNEL_ACC_SLACK = 1.01
KERNEL_EDGE_SLACK = 3.0


def oracle_accept(target, draft, tok, u_acc, u_res, greedy):
    """The oracle's accept step with its per-decision margins (the 5-tuple check_accept takes)."""
    import oracle
    return oracle.spec_accept(target, draft, tok, u_acc, u_res, greedy, want_margins=True)


def check_accept(gpu, ora, what="accept", inputs=None, greedy=False, report=True):
    """gpu = (n_acc, out_tok, n_amb) from the kernel; ora = oracle_accept(...) (5-tuple).

    Only the fp64 oracle decides what is excluded: a sequence is excluded from the exact
    comparison iff the oracle took one of its decisions within the margin (|u - p/q| < 1e-4,
    top-2 logit gap < 1e-4, inverse-CDF edge within 1e-7 of the total).  Every other sequence
    must match exactly, whatever the kernel reports.  An excluded sequence that differs must
    differ first at a decision the oracle itself places within the margin, and (sampling mode,
    same acceptance) must still have drawn a token whose fp64 inverse-CDF interval holds
    u * total within 1e-6 of the total.  The kernel's own flag count is reported beside the
    oracle's; on sequences the oracle does not exclude it may flag only where an oracle margin
    lies just past its threshold (the kernel evaluates the same rule from fp32 exponentials;
    KERNEL_ACC_SLACK, KERNEL_EDGE_SLACK).
    Returns the number of excluded sequences."""
    import oracle
    n_acc_g, tok_g, amb_g = gpu
    n_acc_o, tok_o, amb_o, acc_m, draw_m = ora
    B = n_acc_o.shape[0]
    gamma = tok_o.shape[1] - 1
    excl = amb_o > 0
    ok = ~excl
    assert np.array_equal(n_acc_g[ok], n_acc_o[ok]), f"{what}: n_acc differs on a sequence the oracle does not exclude"
    assert np.array_equal(tok_g[ok], tok_o[ok]), f"{what}: tokens differ on a sequence the oracle does not exclude"
    assert np.all((n_acc_g >= 0) & (n_acc_g <= gamma)), f"{what}: n_acc out of range"
    # the kernel's flags on sequences the oracle calls clear: only next to a threshold
    with np.errstate(invalid="ignore"):
        near = np.any(acc_m < MARGIN * KERNEL_ACC_SLACK, axis=1)
        if not greedy:
            near |= draw_m < SAMPLE_EDGE_TOL * KERNEL_EDGE_SLACK
    stray = ok & (amb_g > 0) & ~near
    assert not stray.any(), f"{what}: kernel flags sequences {np.nonzero(stray)[0][:8]} the oracle places off every margin"
    for b in np.nonzero(excl)[0]:
        a_g, a_o = int(n_acc_g[b]), int(n_acc_o[b])
        m = min(a_g, a_o)
        # accepted tokens are the draft tokens themselves: the common prefix must agree
        assert np.array_equal(tok_g[b, :m], tok_o[b, :m]), f"{what}: seq {b} accepted prefix differs"
        if a_g != a_o:
            assert acc_m[b, m] < MARGIN, (f"{what}: seq {b} accepts {a_g} vs {a_o}; the oracle's decision at "
                                          f"position {m} is {acc_m[b, m]:.3e} from its boundary")
            continue
        t = int(tok_g[b, a_g])
        assert np.all(tok_g[b, a_g + 1:] == -1), f"{what}: seq {b} padding"
        if t == tok_o[b, a_g]:
            continue
        if greedy:
            assert acc_m[b, a_g] < MARGIN, f"{what}: seq {b} emits {t} vs {tok_o[b, a_g]} off the argmax margin"
            continue
        assert draw_m[b] < SAMPLE_EDGE_TOL, (f"{what}: seq {b} draws {t} vs {tok_o[b, a_g]}; the oracle's draw is "
                                             f"{draw_m[b]:.3e} of the total from a token edge")
        if inputs is not None:
            target, draft, u_res = inputs
            if a_g < gamma:
                wts = oracle.resample_weights(target[b, a_g], draft[b, a_g])
            else:
                wts = oracle.resample_weights(target[b, gamma])
            cdf = np.cumsum(wts)
            W = cdf[-1]
            x = float(u_res[b]) * W
            assert 0 <= t < len(wts) and wts[t] > 0, f"{what}: seq {b} drew a zero-weight token"
            lo = cdf[t - 1] if t > 0 else 0.0
            assert lo - 1e-6 * W <= x <= cdf[t] + 1e-6 * W, f"{what}: seq {b} token {t} not a valid draw"
    if report:
        print(f"[{what}] B={B}: oracle-excluded {int(excl.sum())}, kernel-flagged {int((amb_g > 0).sum())}")
    return int(excl.sum())
