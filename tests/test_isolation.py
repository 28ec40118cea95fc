"""The oracle and the CUDA path stay apart (checked on the source, no GPU).

The float64 oracle is test infrastructure: only the tests, the smoke check and
the bench's CPU legs may reach it, and it shares no code with the library.  This
test parses the sources and checks that the product package never imports it,
that it never imports the product package, that in `bench.py` it is imported
only by the function the CPU-baseline and reference legs call, that in
`__graft_entry__.py` only `smoke()` imports it, and that no CUDA source includes
anything from it.
"""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "rank_orthonormalized_optimizer_03_b300")
ORACLE = os.path.join(ROOT, "oracle")


def imported_modules(node):
    """Top-level names of the modules that `node`'s subtree imports (relative imports: '.')."""
    out = set()
    for n in ast.walk(node):
        if isinstance(n, ast.Import):
            out |= {a.name.split(".")[0] for a in n.names}
        elif isinstance(n, ast.ImportFrom):
            out.add("." if n.level else (n.module or "").split(".")[0])
    return out


def parse(path):
    with open(path) as f:
        return ast.parse(f.read(), filename=path)


def test_product_package_never_imports_the_oracle():
    files = glob.glob(os.path.join(PKG, "*.py"))
    assert files
    for path in files:
        assert "oracle" not in imported_modules(parse(path)), path


def test_oracle_never_imports_the_product_package():
    files = glob.glob(os.path.join(ORACLE, "*.py"))
    assert files
    for path in files:
        mods = imported_modules(parse(path))
        assert "rank_orthonormalized_optimizer_03_b300" not in mods, path
        assert mods <= {"__future__", ".", "math", "numpy", "torch", "typing"}, (path, mods)


def functions_importing_oracle(tree):
    """Names of the top-level functions whose bodies import the oracle; None marks module level."""
    names = set()
    for node in tree.body:
        if isinstance(node, (ast.FunctionDef, ast.AsyncFunctionDef)):
            if "oracle" in imported_modules(node):
                names.add(node.name)
        elif "oracle" in imported_modules(node):
            names.add(None)
    return names


def callers_of(tree, fname):
    out = set()
    for node in tree.body:
        if isinstance(node, (ast.FunctionDef, ast.AsyncFunctionDef)) and node.name != fname:
            for n in ast.walk(node):
                if isinstance(n, ast.Call) and isinstance(n.func, ast.Name) and n.func.id == fname:
                    out.add(node.name)
    return out


def test_bench_reaches_the_oracle_only_from_its_cpu_legs():
    tree = parse(os.path.join(ROOT, "bench.py"))
    assert functions_importing_oracle(tree) == {"oracle_time"}
    assert callers_of(tree, "oracle_time") == {"cpu_baseline", "run_reference"}
    # the timed CUDA arm itself never calls those legs
    for leg in ("cpu_baseline", "run_reference", "oracle_time"):
        assert "measure" not in callers_of(tree, leg)


def test_graft_entry_imports_the_oracle_only_in_smoke():
    tree = parse(os.path.join(ROOT, "__graft_entry__.py"))
    assert functions_importing_oracle(tree) == {"smoke"}


def test_cuda_sources_include_nothing_from_the_oracle():
    srcs = glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    assert srcs
    for path in srcs:
        with open(path) as f:
            for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', f.read()):
                assert "oracle" not in inc, (path, inc)
