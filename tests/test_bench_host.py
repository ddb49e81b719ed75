"""Host-side checks of bench.py's helpers (no GPU)."""
import importlib.util
import os

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
