"""Drafting-strategy selector (MagicDec section 3.1 Eq. 1-2, section 4.1 Eq. 3-4).

Pinned to Eq. 1's series, to the paper's printed step-time tables (Table 2 of section 5.2,
Tables 4, 6 and 7 of appendices A.3-A.5: the acceptance rate is recovered from the printed
Omega by inverting Eq. 1, then the selector's objective must reproduce the printed T_SD and
speedup, and never exceed the printed T_SD by more than rounding, since what the model
leaves out is extra time), and to exhaustive search for the argmin."""
import itertools
import math
import os
import random

import pytest

from long_context_self_gb300 import costmodel as cm

GOLDEN_DIR = os.path.join(os.path.dirname(__file__), "golden")
# printed tables with the columns gamma, gamma*T_D, T_V, Omega, T_AR, T_SD, x -> row count
STEP_TABLES = {"magicdec_table2.tsv": 6, "magicdec_table4.tsv": 3, "magicdec_table6.tsv": 8,
               "magicdec_table7.tsv": 6}


def read_table(path):
    lines = [l for l in open(path) if l.strip() and not l.startswith("#")]
    hdr = lines[0].split("\t")
    hdr = [h.strip() for h in hdr]
    return [dict(zip(hdr, (x.strip() for x in l.split("\t")))) for l in lines[1:]]


def alpha_from_omega(gamma, omega):
    lo, hi = 0.0, 1.0 - 1e-12
    for _ in range(200):
        mid = (lo + hi) / 2
        if cm.expected_tokens(gamma, mid) < omega:
            lo = mid
        else:
            hi = mid
    return lo


@pytest.mark.parametrize("gamma", [0, 1, 3, 7])
@pytest.mark.parametrize("alpha", [0.0, 0.3, 0.8, 0.99])
def test_eq1_equals_geometric_series(gamma, alpha):
    assert math.isclose(cm.expected_tokens(gamma, alpha), sum(alpha ** k for k in range(gamma + 1)), rel_tol=1e-12)


def test_eq1_limits():
    assert cm.expected_tokens(4, 1.0) == 5.0
    assert cm.expected_tokens(4, 0.0) == 1.0


@pytest.mark.parametrize("name", sorted(STEP_TABLES))
def test_objective_reproduces_printed_step_tables(name):
    rows = read_table(os.path.join(GOLDEN_DIR, name))
    assert len(rows) == STEP_TABLES[name]
    for r in rows:
        g = int(r["gamma"])
        a = alpha_from_omega(g, float(r["Omega"]))
        t_sd = cm.avg_time_per_token(g, a, float(r["gT_D"]) / g, 0.0, float(r["T_V"]))
        printed = float(r["T_SD"])
        assert abs(t_sd - printed) / printed < 0.06, r
        assert t_sd <= printed * 1.005, r                 # the unmodelled remainder is extra time
        assert abs(float(r["T_AR"]) / t_sd - float(r["x"])) < 0.08, r
        # the printed speedup is the printed ratio T_AR / T_SD (to the printed rounding)
        assert abs(float(r["T_AR"]) / printed - float(r["x"])) < 0.051, r


def test_select_is_the_exhaustive_argmin():
    rnd = random.Random(5)
    for _ in range(50):
        budgets = [256, 512, 1024, 2048]
        gammas = [1, 2, 3, 4, 5, 6]
        t_t = rnd.uniform(1, 3)
        tim = cm.Timings(t_target=t_t, t_verify={g: t_t * (1 + 0.05 * g * rnd.random()) for g in gammas},
                         t_draft={K: 0.02 + K / 32000 * t_t for K in budgets},
                         t_select={("snapkv", K): rnd.uniform(0, 0.05) for K in budgets})
        alpha = {(m, K): rnd.uniform(0.3, 0.95) for m in ("streaming", "snapkv") for K in budgets}
        c = cm.select(tim, alpha)
        best = min(((m, K, g) for (m, K) in alpha for g in gammas),
                   key=lambda x: cm.avg_time_per_token(x[2], alpha[(x[0], x[1])], tim.t_draft[x[1]],
                                                       tim.t_select.get((x[0], x[1]), 0.0), tim.t_verify[x[2]]))
        assert (c.method, c.budget, c.gamma) == best
        assert math.isclose(c.speedup * c.ratio, 1.0)


def test_free_draft_and_kv_bound_verify_give_omega():
    """T_D -> 0 and T_V = T_T (the long-context, KV-bound limit of section 3.2): speedup = Omega."""
    tim = cm.Timings(t_target=1.0, t_verify={3: 1.0}, t_draft={512: 0.0})
    c = cm.select(tim, {("streaming", 512): 0.8})
    assert math.isclose(c.speedup, cm.expected_tokens(3, 0.8))


def test_higher_acceptance_prefers_longer_speculation():
    gammas = range(1, 12)
    tim = cm.Timings(t_target=1.0, t_verify={g: 1.0 + 0.02 * g for g in gammas}, t_draft={512: 0.05})
    g_lo = cm.select(tim, {("streaming", 512): 0.5}).gamma
    g_hi = cm.select(tim, {("streaming", 512): 0.95}).gamma
    assert g_hi > g_lo


@pytest.mark.gpu
def test_calibrated_times_show_the_kv_bound_regime():
    """Section 3.2: at long context verification and decoding load the same KV, so
    T_V(gamma) / T_T stays close to 1, and a 512-row draft costs a small fraction."""
    tim = cm.calibrate(B=32, S=32000, budgets=[512], gammas=[3], reps=5)
    assert 0.9 < tim.t_verify[3] / tim.t_target < 1.3
    assert tim.t_draft[512] / tim.t_target < 0.2
    c = cm.select(tim, {("streaming", 512): 0.8})
    assert c.speedup > 1.0


@pytest.mark.gpu
def test_dynamic_draft_search_cost_dominates_at_large_batch():
    """Section 4.4: Top-K attention and the PQCache-style draft keep a small budget but search the
    cache at every draft step, so their draft cost is a large fraction of verification; with equal
    acceptance rates the static StreamingLLM draft wins, and a dynamic draft needs a clearly higher
    acceptance rate to be chosen."""
    tim = cm.calibrate(B=32, S=32000, budgets=[512], gammas=[3], reps=3, topk=True, pq=True)
    for method in ("topk", "pq"):
        t_dyn = tim.t_draft[512] + tim.t_select[(method, 512)]
        assert t_dyn / tim.t_target > 0.2, method
    c = cm.select(tim, {("streaming", 512): 0.8, ("topk", 512): 0.8, ("pq", 512): 0.8})
    assert c.method == "streaming"
