"""The oracle and the CUDA path stay apart, and the product path has no
fallback.

- Nothing in the package or in the shared input generators imports the
  oracle, and the oracle imports nothing of theirs (numpy and the standard
  library only).
- In bench.py the oracle is reached only from its CPU-baseline and
  reference legs.
- The binding raises when the built library is missing instead of falling
  back to anything else.
"""

import ast
import importlib
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "block_speculative_decoding_dflash2_gb300"


def _py_files(*dirs):
    for d in dirs:
        for base, _, files in os.walk(os.path.join(ROOT, d)):
            for f in files:
                if f.endswith(".py"):
                    yield os.path.join(base, f)


def _imported_roots(tree):
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.level == 0 and node.module:
            out.add(node.module.split(".")[0])
    return out


def test_product_and_generators_never_import_the_oracle():
    for path in _py_files(PKG, "dflash2_synth"):
        roots = _imported_roots(ast.parse(open(path).read()))
        assert "oracle" not in roots, path


def test_oracle_imports_only_numpy_and_the_standard_library():
    allowed = {"math", "numpy"}
    for path in _py_files("oracle"):
        roots = _imported_roots(ast.parse(open(path).read()))
        assert roots <= allowed, (path, roots - allowed)


def test_native_sources_do_not_reach_into_the_oracle():
    for d in (os.path.join(PKG, "csrc"), "include"):
        for f in os.listdir(os.path.join(ROOT, d)):
            for line in open(os.path.join(ROOT, d, f)).read().splitlines():
                if line.lstrip().startswith("#include"):
                    assert "oracle" not in line, (f, line)


def test_only_smoke_runs_the_oracle_in_the_entry_module():
    tree = ast.parse(open(os.path.join(ROOT, "__graft_entry__.py")).read())
    funcs = [n for n in tree.body if isinstance(n, ast.FunctionDef)]
    assert {f.name for f in funcs if "oracle" in _imported_roots(f)} == {"smoke"}
    assert "oracle" not in _imported_roots(ast.Module(body=[n for n in tree.body if not isinstance(
        n, ast.FunctionDef)], type_ignores=[]))


def test_bench_reaches_the_oracle_only_from_its_cpu_legs():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    funcs = {n.name: n for n in tree.body if isinstance(n, ast.FunctionDef)}
    assert "oracle" not in _imported_roots(ast.Module(body=[n for n in tree.body if not isinstance(
        n, ast.FunctionDef)], type_ignores=[]))
    importers = {name for name, fn in funcs.items() if "oracle" in _imported_roots(fn)}
    assert importers == {"oracle_state", "oracle_step"}

    def calls(fn):
        return {c.func.id for c in ast.walk(fn) if isinstance(c, ast.Call) and isinstance(c.func, ast.Name)}

    # every function that reaches an oracle entry, directly or through another
    reach = set(importers)
    while True:
        more = {name for name, fn in funcs.items() if calls(fn) & reach} - reach
        if not more:
            break
        reach |= more
    cpu_legs = {"time_oracle", "cpu_baseline", "run_cpu_step_only", "run_reference"}
    # main dispatches to the legs (and adds the cpu_baseline object to the
    # line after the GPU arm has run); the GPU arm itself never reaches them
    assert reach - importers <= cpu_legs | {"main"}, reach
    assert "run_ours" not in reach


def test_binding_raises_without_the_library(monkeypatch, tmp_path):
    B = importlib.import_module(f"{PKG}.binding")
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        B.lib()
