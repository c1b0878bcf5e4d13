"""bench.py's reference arm (the CPU oracle, timed on the host) prints one JSON line with the
metric, unit and direction of the GPU arm, a cpu_baseline block and a zero-copy e2e block."""

import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["higher_is_better"] is True and line["n_gpus"] == 1
    assert line["steps"] == 1 and line["warmup"] == 1
    assert line["value"] > 0 and line["ms_per_step"] > 0
    cfg = line["config"]
    assert cfg["workload"] == bench.DEFAULT_WORKLOAD
    # the same workload keys as the GPU arm's config
    for key in ("batch", "query_heads", "kv_heads", "head_dim", "page_size",
                "max_pages_per_sequence", "context_tokens", "parallelism"):
        assert key in cfg, key
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_kernel_hash_ignores_comments_only():
    """A recorded ncu capture stays attached to the code it measured: comment and layout
    edits keep the hash, code edits change it."""
    base = 'int f(int a) {\n  return a + 1;  // one\n}\n/* note */ const char *s = "x // y";\n'
    assert bench.code_of(base) == bench.code_of(base.replace("// one", "// two"))
    assert bench.code_of(base) == bench.code_of(base.replace("/* note */", ""))
    assert bench.code_of(base) == bench.code_of(base.replace("  return", "\n\n    return"))
    assert bench.code_of(base) != bench.code_of(base.replace("a + 1", "a + 2"))
    assert bench.code_of(base) != bench.code_of(base.replace('"x // y"', '"x / y"'))
    assert bench.code_of("a + +b") != bench.code_of("a ++b")
