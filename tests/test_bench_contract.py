"""The bench's host-side logic (CPU): the reference arm's JSON line, the
profile-validity check that feeds the roofline's DRAM traffic, and the query
split between ranks."""
import importlib.util
import json
import os
import subprocess
import sys

from conftest import ROOT


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` times the oracle and prints one JSON line
    with the contract's keys, the reference marker and its own e2e figure."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["metric"] == "constrained decode steps/s" and d["unit"] == "steps/s"
    assert d["config"]["workload"] == "large_head"
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1


def test_source_hash_ignores_comments_only(tmp_path):
    b = _bench()
    a = tmp_path / "a.cu"
    a.write_text("int f() {  // first\n  return 1;\n}\n")
    h0 = b.source_code_sha256(str(a))
    a.write_text("// a new header comment\nint f() {  // changed\n\n  return 1;   \n}\n")
    assert b.source_code_sha256(str(a)) == h0
    a.write_text("int f() {\n  return 2;\n}\n")
    assert b.source_code_sha256(str(a)) != h0


def test_recorded_traffic_follows_the_kernel_source():
    """The committed one-CTA-step capture is read only while its source hash
    matches the kernel files; the default line's traffic comes from it."""
    b = _bench()
    t = b.recorded_traffic("step_kernels.cu+kernels.h", "sparse_step1_kernel_large_head.md")
    assert t is not None and t > 0
    assert b.recorded_traffic("step_kernels.cu+kernels.h", "no_such_profile.md") is None
    assert b.recorded_traffic("gemm_tc.cu", "sparse_step1_kernel_large_head.md") is None  # no hash for that file


def test_query_split_is_disjoint_across_ranks():
    b = _bench()
    n, world, count = 1000, 4, 100
    per_rank = [b.query_ids(n, r, world, count) for r in range(world)]
    flat = [q for ids in per_rank for q in ids]
    assert len(set(flat)) == len(flat) == world * count
