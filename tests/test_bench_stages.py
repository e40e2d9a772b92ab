"""bench.py's prolog and epilog stages on the CPU: their reference legs run the fp64 oracle."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    return lines[0]


def test_prolog_reference_leg():
    line = _run("--stage", "prolog", "--impl", "reference", "--workload", "tiny", "--steps", "1")
    assert line["impl"] == "reference" and line["stage"] == "prolog"
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["config"]["tokens"] == 4


def test_epilog_reference_leg():
    line = _run("--stage", "epilog", "--impl", "reference", "--workload", "tiny", "--steps", "1")
    assert line["impl"] == "reference" and line["stage"] == "epilog"
    assert line["value"] > 0 and line["config"]["tokens"] == 4


def test_layer_reference_leg():
    line = _run("--stage", "layer", "--impl", "reference", "--workload", "tiny")
    assert line["impl"] == "reference" and line["stage"] == "layer" and line["value"] > 0
    assert set(line["phases_s"]) == {"prolog", "decode_extrapolated", "epilog"}
    assert line["cpu_baseline"]["kind"] == "oracle"
