"""bench.py's host-side accounting, without a GPU: the algorithmic bytes and
FLOPs the roofline fractions divide by (counted here by hand from the
definition of attention over a paged cache), the guard that drops a profiled
DRAM traffic figure once the kernel code differs from the profiled code,
and the JSON line of the reference arm (the fp64 oracle on the host)."""
import json
import os
import shutil
import subprocess
import sys

import pytest

import bench
from chunked_prefill_decode_gb300.workloads import Shape, layout_from_rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_counts_by_hand():
    # 8 q / 2 kv heads, D 64: one decode row over 100 keys and one 20-token
    # chunk at offset 30 (its tokens see 31 .. 50 keys)
    lay = layout_from_rows(Shape(8, 2, 64), [(1, 100), (20, 50)], 0)
    c = bench.algorithmic_counts(lay)
    kv_tok = 2 * 2 * 64 * 2          # K and V of one cached token, all kv heads
    qo_tok = 2 * 8 * 64 * 2          # q read + out written per new token
    assert c["decode_flops"] == 4 * 8 * 64 * 100
    # c*o + c(c+1)/2 visible keys over the chunk's tokens
    assert c["chunk_flops"] == 4 * 8 * 64 * (20 * 30 + 20 * 21 // 2)
    assert c["decode_bytes"] == 100 * kv_tok + 1 * qo_tok
    assert c["chunk_bytes"] == 50 * kv_tok + 20 * qo_tok
    assert c["append_bytes"] == 2 * 21 * kv_tok
    assert c["bytes"] == c["decode_bytes"] + c["chunk_bytes"] + c["append_bytes"]
    assert c["flops"] == c["decode_flops"] + c["chunk_flops"]


def test_algorithmic_counts_with_a_window():
    # window W = 16: the decode row (position 99) sees keys 84 .. 99; the
    # chunk's first token (position 30) sees 15 .. 30, so the chunk needs keys
    # 15 .. 49 and each of its tokens sees 16
    lay = layout_from_rows(Shape(8, 2, 64, sliding_window=16), [(1, 100), (20, 50)], 0)
    c = bench.algorithmic_counts(lay)
    kv_tok, qo_tok = 2 * 2 * 64 * 2, 2 * 8 * 64 * 2
    assert c["decode_flops"] == 4 * 8 * 64 * 16
    assert c["chunk_flops"] == 4 * 8 * 64 * 20 * 16
    assert c["decode_bytes"] == 16 * kv_tok + qo_tok
    assert c["chunk_bytes"] == 35 * kv_tok + 20 * qo_tok


def test_window_wider_than_the_context_counts_like_no_window():
    rows = [(1, 100), (20, 50), (7, 7)]
    full = bench.algorithmic_counts(layout_from_rows(Shape(8, 2, 64), rows, 0))
    wide = bench.algorithmic_counts(layout_from_rows(Shape(8, 2, 64, sliding_window=100), rows, 0))
    assert full == wide


def _copy_tree_for_profiles(dst):
    os.makedirs(os.path.join(dst, "profiles"))
    os.makedirs(os.path.join(dst, "chunked_prefill_decode_gb300", "csrc"))
    for name in os.listdir(os.path.join(ROOT, "profiles")):
        shutil.copy(os.path.join(ROOT, "profiles", name), os.path.join(dst, "profiles", name))
    for src in bench.ATTN_SOURCES:
        shutil.copy(os.path.join(ROOT, "chunked_prefill_decode_gb300", "csrc", src),
                    os.path.join(dst, "chunked_prefill_decode_gb300", "csrc", src))


def test_profiled_traffic_follows_the_code(tmp_path, monkeypatch):
    """A summary's traffic is used while the attention sources' code
    (comments and layout aside) digests to the value it records, and dropped
    (None) once the code of any of them changes.  Run on a copy of the tree
    with summaries written for the code as it is now."""
    dst = str(tmp_path / "repo")
    _copy_tree_for_profiles(dst)
    monkeypatch.setattr(bench, "ROOT", dst)
    digest = bench.attention_sources_digest()
    names = {"mistral_b512": 638478336, "yi_b2048": 1179897184, "decode_only": 4893324288}
    for w, traffic in names.items():
        with open(os.path.join(dst, "profiles", f"attention_{w}.md"), "w") as f:
            f.write(f"# summary\n\ntraffic_bytes_per_launch: {traffic}\ncode_sha256: {digest}\n")
    got = {w: bench.profiled_traffic(w) for w in names}
    assert got == names
    assert bench.profiled_traffic("tiny") is None          # no summary for it
    plan_h = os.path.join(dst, "chunked_prefill_decode_gb300", "csrc", "decode_plan.h")
    with open(plan_h, "a") as f:                           # comments and blank lines
        f.write("\n// a note\n/* another\n   note */\n\n")
    assert {w: bench.profiled_traffic(w) for w in names} == got
    with open(plan_h, "a") as f:                           # code
        f.write("static const int hb_unused_constant = 1;\n")
    assert all(bench.profiled_traffic(w) is None for w in names)


def test_committed_summaries_record_a_digest_and_traffic():
    """Each committed attention summary names its traffic and the digest of
    the code it was taken on (the bench uses the traffic only while that
    digest matches the current sources)."""
    for w in ("mistral_b512", "yi_b2048", "decode_only"):
        text = open(os.path.join(ROOT, "profiles", f"attention_{w}.md")).read()
        fields = dict(l.split(":", 1) for l in text.splitlines()
                      if l.split(":")[0] in ("traffic_bytes_per_launch", "code_sha256"))
        assert int(fields["traffic_bytes_per_launch"]) > 0
        assert len(fields["code_sha256"].strip()) == 16


def test_source_code_tokens():
    src = ('int a = 1;   // tail comment\n'
           '/* block\n comment */ const char* s = "x // y /* z */";\n'
           "char q = '\"'; char e = '\\''; int b;\n")
    assert bench.source_code_tokens(src) == (
        'int a = 1; const char* s = "x // y /* z */"; '
        "char q = '\"'; char e = '\\''; int b;")
    assert bench.source_code_tokens("a/*x*/b") == "a b"
    assert bench.source_code_tokens("a  +\n\tb") == bench.source_code_tokens("a + b")


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on the host and prints one
    JSON line with the contract's keys."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "3"], cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 3)
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_builder_host_time_is_measured_in_steady_state():
    """The batch-build timing runs the native builder at the batch's shape
    (its decode rows running, a prompt chunked beside them) and returns a
    finite positive median."""
    import math
    from _hbutil import lib
    from chunked_prefill_decode_gb300 import workloads
    lib()
    for name in ("tiny", "decode_only"):
        us = bench.builder_host_us(workloads.WORKLOADS[name](), reps=20, num_pages=50_000)
        assert math.isfinite(us) and us > 0
