"""The bench's reference arm (the CPU oracle timed on bands of the workload) on
CPU: one JSON line with the contract's keys from rank 0, nothing from other
ranks."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [l for l in r.stdout.splitlines() if l.strip()]


def test_reference_arm_prints_one_contract_line():
    lines = _run({"RANK": "0"})
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["warmup"] >= 3 and d["steps"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "tiny" in d["config"]["workload"]


def test_reference_arm_other_ranks_print_nothing():
    assert _run({"RANK": "1"}) == []


def test_capture_hash_ignores_comments_and_sees_code():
    """The committed ncu capture's figures are reported only while the fused
    kernel's code is the one captured: its hash drops comments and blank lines
    (an edited comment keeps the figures) and changes with any code token."""
    sys.path.insert(0, ROOT)
    import bench
    src = 'int a = 1; // one\n/* block\n comment */\n\nfloat b = 2.0f;  \n'
    assert bench._code_only(src) == "int a = 1;\nfloat b = 2.0f;"
    assert bench._code_only(src.replace("// one", "// uno")) == bench._code_only(src)
    assert bench._code_only(src.replace("1;", "2;")) != bench._code_only(src)
    assert len(bench.source_sha()) == 64
