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


def test_recorded_traffic_follows_the_kernel_source(tmp_path):
    """The bench reports the verification kernel's ncu DRAM bytes from a JSON record only while
    the kernel's source is the one the capture was taken on; the committed record's traffic
    equals the algorithmic bytes within 1 % (no re-reads)."""
    import json
    from long_context_self_gb300.ncu_record import source_sha16
    rec = json.load(open(bench.TRAFFIC_RECORD))
    w = bench.synth.WORKLOADS["llama8b_b128_l32k"]
    algorithmic = 2.0 * w.B * w.L * w.H_kv * w.d * 2 + 2.0 * w.B * w.n_q * w.H_q * w.d * 2
    assert rec["workload"] == "llama8b_b128_l32k"
    assert abs(rec["dram_bytes_per_launch"] / algorithmic - 1.0) < 0.01
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_per_captured_launch"] * rec["scale"]
    current = dict(rec, source_sha16=source_sha16(os.path.join(bench.ROOT, rec["source"])))
    path = tmp_path / "rec.json"
    path.write_text(json.dumps(current))
    assert bench.recorded_traffic("llama8b_b128_l32k", str(path)) == rec["dram_bytes_per_launch"]
    assert bench.recorded_traffic("tiny", str(path)) is None
    path.write_text(json.dumps(dict(current, source_sha16="0" * 16)))
    assert bench.recorded_traffic("llama8b_b128_l32k", str(path)) is None


def test_ncu_record_reads_raw_csv(tmp_path):
    """ncu --page raw --csv: a header row, a units row, one row per launch."""
    from long_context_self_gb300 import ncu_record
    raw = tmp_path / "raw.csv"
    raw.write_text('"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum"\n'
                   '"","","Gbyte","Mbyte"\n'
                   '"0","void magicdec::verify_heads_kernel(...)","4.20","7.00"\n'
                   '"1","gather_kv_kernel","1.00","1.00"\n')
    assert ncu_record.launch_traffic(str(raw), "verify_heads") == [4.20e9 + 7.00e6]
