"""The oracle and the CUDA path stay independent, and the product has no fallback.

- Nothing in the package (Python or CUDA sources, headers) imports, includes or reads
  the oracle, and the oracle imports nothing of the package, its seeded generator or
  torch: its only dependencies are numpy, scipy and the standard library.
- bench.py touches the oracle only in its CPU-baseline leg and its reference arm.
- Without the built library the binding raises; there is no other code path.
"""
import ast
import glob
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "routing_token_shuffle_gb300")


def _imports(path):
    """Top-level module names imported anywhere in a Python file."""
    tree = ast.parse(open(path).read(), path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.level == 0 and node.module:
            names.add(node.module.split(".")[0])
    return names


def test_package_never_imports_the_oracle():
    for path in glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True):
        assert "oracle" not in _imports(path), path
        src = open(path).read()
        assert "oracle/" not in src and "'oracle'" not in src and '"oracle"' not in src, path
    for path in (glob.glob(os.path.join(PKG, "csrc", "*")) +
                 glob.glob(os.path.join(ROOT, "include", "*"))):
        for line in open(path, errors="replace"):
            if line.lstrip().startswith("#include"):
                assert "oracle" not in line, (path, line)
            assert "oracle/" not in line and "smoe_oracle" not in line, (path, line)


def test_oracle_depends_on_numpy_scipy_and_the_standard_library_only():
    allowed = {"numpy", "scipy", "itertools", "__future__", "math", "fractions"}
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        mods = _imports(path)
        assert mods <= allowed, (path, sorted(mods - allowed))


def test_bench_uses_the_oracle_only_in_its_baseline_legs():
    path = os.path.join(ROOT, "bench.py")
    tree = ast.parse(open(path).read(), path)
    allowed = {"cpu_oracle_rate", "run_reference", "reference_inputs"}
    found = []

    def visit(node, stack):
        for child in ast.iter_child_nodes(node):
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)):
                visit(child, stack + [child.name])
                continue
            if isinstance(child, (ast.Import, ast.ImportFrom)):
                names = ([a.name for a in child.names] if isinstance(child, ast.Import)
                         else [child.module or ""])
                if any(n.split(".")[0] == "oracle" for n in names):
                    found.append((child.lineno, stack[-1] if stack else "<module>"))
            visit(child, stack)

    visit(tree, [])
    assert found, "bench.py's baseline legs import the oracle"
    assert all(fn in allowed for _, fn in found), found


def test_missing_library_raises():
    code = ("from routing_token_shuffle_gb300 import binding as B\n"
            "B.LIB_PATH = '/nonexistent/libsmoe.so'\n"
            "try:\n"
            "    B.lib()\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n"
            "else:\n"
            "    raise SystemExit('no error')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "raised:" in r.stdout and "not built" in r.stdout, (
        r.stdout + r.stderr)
