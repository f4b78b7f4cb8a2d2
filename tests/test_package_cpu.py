"""What may reach what, checked on the sources: the product (the package and its C
headers) never reaches the oracle, the oracle never reaches the product, the shared
input generator reaches neither, and bench.py and the entry module reach the oracle only
from their CPU legs. The package refuses to import without its compiled library (no
fallback)."""
import ast
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "expert_token_dispatch_gemm_b300"


def files(sub, exts):
    out = []
    for d, _, names in os.walk(os.path.join(ROOT, sub)):
        if "__pycache__" in d:
            continue
        out += [os.path.join(d, n) for n in names if n.endswith(exts)]
    return out


def imported_modules(path):
    """(top-level module, enclosing function or None) for every import in a file."""
    tree = ast.parse(open(path).read())
    found = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(child, ast.Import):
                found.extend((a.name.split(".")[0], fn) for a in child.names)
            elif isinstance(child, ast.ImportFrom) and child.module and child.level == 0:
                found.append((child.module.split(".")[0], fn))
            visit(child, f)
    visit(tree, None)
    return found


def test_product_never_reaches_the_oracle():
    for path in files(PKG, (".py",)):
        assert "oracle" not in [m for m, _ in imported_modules(path)], path
    for path in files(PKG, (".cu", ".cuh", ".h")) + files("include", (".h",)):
        assert "oracle" not in open(path).read().lower(), path


def test_oracle_and_input_generator_do_not_reach_the_product():
    for sub, banned in (("oracle", {PKG}), ("workloads", {PKG, "oracle"})):
        for path in files(sub, (".py",)):
            mods = {m for m, _ in imported_modules(path)}
            assert not (mods & banned), (path, mods & banned)


def test_bench_and_entry_reach_the_oracle_only_from_their_cpu_legs():
    allowed = {"bench.py": {"time_oracle_slice"}, "__graft_entry__.py": {"smoke"}}
    for name, fns in allowed.items():
        uses = [fn for m, fn in imported_modules(os.path.join(ROOT, name)) if m == "oracle"]
        assert uses and set(uses) <= fns, (name, uses)


def test_import_fails_loudly_without_the_library(tmp_path):
    """A copy of the package without libmoe.so: importing it raises ImportError naming
    the missing library instead of falling back to anything."""
    dst = tmp_path / PKG
    dst.mkdir()
    for n in os.listdir(os.path.join(ROOT, PKG)):
        if n.endswith(".py"):
            shutil.copy(os.path.join(ROOT, PKG, n), dst / n)
    r = subprocess.run([sys.executable, "-c", f"import {PKG}"], cwd=tmp_path,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libmoe.so is missing" in r.stderr
