"""The bench's speculative-step arithmetic against the paper's printed numbers.

tests/golden/magicdec_table1.tsv holds MagicDec section 5.1 Table 1 as printed.  The
table's T_SD follows T_SD = (gamma*T_D + T_V) / Omega (section 3.1) up to the
overheads the paper does not model (a few percent), and its speedup is T_AR / T_SD."""
import math
import os

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "magicdec_table1.tsv")


def rows():
    lines = [l for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    hdr = lines[0].split()
    for l in lines[1:]:
        yield dict(zip(hdr, l.split()))


def test_table1_step_time_convention():
    n = 0
    for r in rows():
        t_sd = bench.spec_step_time(float(r["gT_D"]), float(r["T_V"]), float(r["Omega"]))
        assert abs(t_sd - float(r["T_SD"])) / float(r["T_SD"]) < 0.06, r
        assert abs(float(r["T_AR"]) / float(r["T_SD"]) - float(r["x"])) < 0.011, r
        n += 1
    assert n == 6


def test_expected_tokens_closed_form():
    # Eq. 1 limits: alpha -> 0 gives 1 token, alpha -> 1 gives gamma + 1
    assert bench.expected_tokens(0.0, 5) == 1.0
    assert bench.expected_tokens(1.0, 5) == 6.0
    assert math.isclose(bench.expected_tokens(0.5, 2), 1.75)


def test_aggregate_rate_is_whole_job():
    assert math.isclose(bench.aggregate_rate(4, 10, 2000.0), 20.0)


def test_recorded_traffic_is_read_from_the_committed_profile():
    """The bench reports the verification kernel's ncu DRAM bytes from profiles/ while attn_heads.cu is
    the source the capture was taken on; the recorded traffic equals the algorithmic bytes within 1 %."""
    t = bench.recorded_traffic("llama8b_b128_l32k")
    assert t is not None
    w = bench.synth.WORKLOADS["llama8b_b128_l32k"]
    algorithmic = 2.0 * w.B * w.L * w.H_kv * w.d * 2 + 2.0 * w.B * w.n_q * w.H_q * w.d * 2
    assert abs(t / algorithmic - 1.0) < 0.01
    assert bench.recorded_traffic("tiny") is None
