"""The product path and the oracle stay apart (CPU, static): nothing in the
package or its CUDA sources imports or includes the oracle; the oracle
imports nothing of the package but the seeded input generators; bench.py
touches the oracle only in its CPU-baseline and reference-arm functions."""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mamba_selective_state_gb300")


def _imports(tree):
    """(module, enclosing function name or None) for every import."""
    out = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            name = fn
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef, ast.ClassDef)):
                name = child.name if fn is None else f"{fn}.{child.name}"
            if isinstance(child, ast.Import):
                out.extend((a.name, fn) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                out.append((child.module or "", fn))
            visit(child, name)
    visit(tree, None)
    return out


def _py(path):
    return ast.parse(open(path).read(), filename=path)


def test_package_never_imports_the_oracle():
    for f in glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True):
        for mod, _ in _imports(_py(f)):
            assert not mod.startswith("oracle"), (f, mod)


def test_cuda_sources_never_include_the_oracle():
    for f in glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*")):
        src = open(f).read()
        assert not re.search(r'#\s*include\s*[<"][^>"]*oracle', src), f


def test_oracle_imports_only_the_input_generators_of_the_package():
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        for mod, _ in _imports(_py(f)):
            if mod.startswith("mamba_selective_state_gb300"):
                assert mod == "mamba_selective_state_gb300.inputs", (f, mod)
    src = open(os.path.join(ROOT, "oracle", "ssd_oracle.c")).read()
    assert "ssd.h" not in src and "csrc" not in src


def test_bench_uses_the_oracle_only_for_cpu_timing():
    # the oracle leg: CPU timing, and (called from cpu_baseline, after the
    # timed region) the parity of the benched outputs
    allowed = {"OracleSample.__init__", "OracleSample.run", "cpu_baseline", "run_reference",
               "norm_oracle_seconds", "run_norm_reference", "oracle_parity"}
    for mod, fn in _imports(_py(os.path.join(ROOT, "bench.py"))):
        if mod.startswith("oracle"):
            assert fn in allowed, (mod, fn)
