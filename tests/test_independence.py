"""The oracle and the CUDA path share no code (static checks, CPU only).

- The product (the package, its CUDA sources, the headers) never names the
  oracle.
- The oracle imports only the standard library, NumPy and itself: no torch,
  no package code, not even the input generators.
- The input generators hold no method code: they import neither side.
- The benchmark imports the oracle only inside the functions of its CPU
  legs (the reference arm and cpu_baseline), never at module level.
"""
import ast
import glob
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _files(*patterns):
    out = []
    for p in patterns:
        out += glob.glob(os.path.join(ROOT, p), recursive=True)
    return sorted(out)


def _imports(path):
    tree = ast.parse(open(path).read())
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            mods.add("." if node.level else (node.module or "").split(".")[0])
    return mods


def test_product_never_names_the_oracle():
    files = _files("rl_step_gb300/**/*.py", "rl_step_gb300/csrc/*", "include/*.h")
    assert files
    for f in files:
        assert "oracle" not in open(f, errors="replace").read().lower(), f


def test_oracle_imports_only_numpy_and_the_standard_library():
    allowed = {"numpy", "struct", "typing", "__future__", "math", "."}
    for f in _files("oracle/*.py"):
        extra = _imports(f) - allowed
        assert not extra, (f, extra)


def test_input_generators_import_neither_side():
    for f in _files("workloads/*.py"):
        mods = _imports(f)
        assert not mods & {"oracle", "rl_step_gb300", "torch"}, (f, mods)


def test_bench_imports_the_oracle_only_inside_its_cpu_legs():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    for node in tree.body:                       # module level
        if isinstance(node, (ast.Import, ast.ImportFrom)):
            names = [a.name for a in node.names] + [getattr(node, "module", None) or ""]
            assert not any(n.split(".")[0] == "oracle" for n in names)
    users = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.Import) and any(a.name == "oracle" for a in node.names):
                    users.add(fn.name)
    assert users == {"make_oracle"}, users
