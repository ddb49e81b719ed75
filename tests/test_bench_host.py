"""Host-side checks of bench.py's helpers (no GPU)."""
import importlib.util
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_code_only_drops_comments_and_blank_lines():
    b = _bench()
    src = ('int a = 1;  // trailing\n'
           '/* block\n   comment */ int b = 2;\n'
           '\n'
           '    // a whole-line comment\n'
           'asm("mov.b64 %0, {%1, %2};  // kept: inside a string");\n'
           "char c = '/';\n")
    got = b._code_only(src)
    assert "trailing" not in got and "block" not in got and "whole-line" not in got
    assert '"mov.b64 %0, {%1, %2};  // kept: inside a string"' in got
    assert "char c = '/';" in got
    assert "\n\n" not in got


def test_code_only_sees_code_changes_but_not_comment_edits():
    b = _bench()
    base = "int f(int x) {\n    return x + 1;  // add one\n}\n"
    assert b._code_only(base) == b._code_only(base.replace("add one", "increment"))
    assert b._code_only(base) == b._code_only(base.replace("    return", "    // note\n    return"))
    assert b._code_only(base) != b._code_only(base.replace("x + 1", "x + 2"))


def test_reference_arm_prints_one_contract_line():
    """``bench.py --impl reference`` (the fp64 oracle on the host cores) prints one
    JSON line with the fields the measurement contract asks of that arm."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "calls/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]
    # the line describes what this arm ran: one oracle call + inject-add per step, one weight set
    assert d["config"]["calls_per_step"] == 1 and d["config"]["weight_sets"] == 1
