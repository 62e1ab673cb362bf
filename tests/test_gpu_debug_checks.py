"""The range-checking build (long_context_self_gb300.build --debug, loaded with
MAGICDEC_LIBRARY=debug): every kernel that reads a caller's length or gather index
records one outside its range as device error 4, and writes the same outputs as the
release build, which clamps or skips the value without recording it."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CASES = ("gather_kv", "verify_attn", "verify_attn_heads16", "verify_attn_heads20", "draft_attn", "draft_cache_update",
         "snapkv_select", "topk_draft_attn", "pq_draft_attn")


def child(library):
    env = dict(os.environ)
    env.pop("MAGICDEC_LIBRARY", None)
    if library:
        env["MAGICDEC_LIBRARY"] = library
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_checks_child.py")], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def libraries():
    from long_context_self_gb300 import build
    build.build()
    build.build(debug=True)


def test_debug_build_records_out_of_range_lengths_and_indices(libraries):
    res = child("debug")
    assert res["library"] == "libmagicdec_debug.so"
    for case in CASES:
        r = res[case]
        assert r["err_in_range"] == 0, (case, r)
        assert r["err_out_of_range"] == 4, (case, r)
        assert r["clamped_output"], (case, r)


def test_release_build_clamps_without_recording(libraries):
    res = child(None)
    assert res["library"] == "libmagicdec.so"
    for case in CASES:
        r = res[case]
        assert r["err_in_range"] == 0 and r["err_out_of_range"] == 0, (case, r)
        assert r["clamped_output"], (case, r)
