"""The bench's reference arm (the oracle timed on the host cores) runs on the
CPU and prints the one JSON line the bench contract asks for."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_the_contract_line():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in j, k
    assert j["n_gpus"] == 1 and j["steps"] == 1 and j["warmup"] == 3
    assert j["value"] > 0 and j["higher_is_better"] is True and j["dtype"] == "f64"
    assert "workload" in j["config"]
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and cb["sample"]
    e = j["e2e"]
    assert e["value"] == j["value"] and e["unit"] == j["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_fewer_than_three_warmup_steps_are_refused():
    r = _bench("--steps", "1", "--warmup", "2", timeout=120)
    assert r.returncode != 0
    assert "warmup" in r.stderr


def test_kernel_source_hash_ignores_comments():
    # the recorded ncu traffic stays valid across comment edits, not code edits
    import bench
    a = 'int x = 1; // one\n/* two */ const char *s = "a//b";'
    b = 'int x = 1;   /* other words */\nconst char *s = "a//b"; // trailing'
    c = 'int x = 2; const char *s = "a//b";'
    assert bench.code_only(a) == bench.code_only(b) == 'int x = 1; const char *s = "a//b";'
    assert bench.code_only(c) != bench.code_only(a)
    src = {n: "int f() { return 1; } // " + n for n in bench.DECODE_SOURCES}
    moved = {n: "/* header */\nint f()\n{\n  return 1;\n}" for n in bench.DECODE_SOURCES}
    assert bench.kernel_sources_sha256(src.get) == bench.kernel_sources_sha256(moved.get)
