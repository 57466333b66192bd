"""The product path has no CPU fallback: without the built library the binding
raises before computing anything, CPU tensors are refused rather than
computed on the host, and no module of the package imports the oracle."""
import ast
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import invariant_token_log_gb300 as bil

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PACKAGE = os.path.join(ROOT, "invariant_token_log_gb300")


def test_missing_library_raises():
    code = textwrap.dedent("""
        import invariant_token_log_gb300._lib as L
        L._build.library_path = lambda: "/nonexistent/libbil.so"
        try:
            L.load()
        except RuntimeError as e:
            assert "no CPU fallback" in str(e), str(e)
            print("raised")
        else:
            raise SystemExit("loaded a library that does not exist")
    """)
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "raised"


def test_cpu_tensors_are_refused():
    x = torch.zeros(2, 16, dtype=torch.bfloat16)
    t = torch.zeros(2, dtype=torch.int64)
    with pytest.raises(ValueError, match="no CPU path"):
        bil.logp_fwd(x, t, -100, 8)


def _imports(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            yield from (a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            yield node.module or ""


def test_package_never_imports_the_oracle():
    sources = [os.path.join(d, f) for d, _, fs in os.walk(PACKAGE) for f in fs if f.endswith(".py")]
    assert sources
    for path in sources:
        for name in _imports(path):
            assert not name.split(".")[0] == "oracle", f"{path} imports {name}"
        text = open(path).read()
        assert "bil_oracle" not in text, path


def test_bench_imports_the_oracle_only_in_its_cpu_legs():
    """bench.py may run the oracle only for the CPU baseline and the reference
    arm; the timed CUDA path never imports it."""
    allowed = {"oracle_rows_per_s", "run_reference", "_linear_oracle_step", "oracle_linear_rows_per_s",
               "run_linear_reference"}
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    for node in tree.body:
        assert "oracle" not in set(_imports_of(node)), "bench.py imports the oracle at module level"
    found = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if "oracle" in set(_imports_of(node)):
                    found.add(fn.name)
    assert found and found <= allowed, found - allowed


def _imports_of(node):
    if isinstance(node, ast.Import):
        return [a.name.split(".")[0] for a in node.names]
    if isinstance(node, ast.ImportFrom):
        return [(node.module or "").split(".")[0]]
    return []
