"""The product path never reaches the oracle (static checks, no GPU).

The oracle is test infrastructure: the library, its binding and the timed part of the benchmark
must not import, link or load it.  These checks read the sources and the built library's
dynamic section and symbol table; they run nothing on a GPU.
"""
import ast
import glob
import os
import subprocess

from sparse_attention_indexer_spin_gb300 import spin

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sparse_attention_indexer_spin_gb300")


def _oracle_imports(path):
    """(line, enclosing function names) of every import of the oracle package in a file."""
    hits = []

    class Visitor(ast.NodeVisitor):
        def __init__(self):
            self.stack = []

        def visit_FunctionDef(self, node):
            self.stack.append(node.name)
            self.generic_visit(node)
            self.stack.pop()

        def visit_Import(self, node):
            if any(a.name.split(".")[0] == "oracle" for a in node.names):
                hits.append((node.lineno, tuple(self.stack)))

        def visit_ImportFrom(self, node):
            if (node.module or "").split(".")[0] == "oracle":
                hits.append((node.lineno, tuple(self.stack)))

    with open(path) as f:
        Visitor().visit(ast.parse(f.read(), path))
    return hits


def _callers(path, name):
    """Names of the top-level functions whose bodies call `name`."""
    with open(path) as f:
        tree = ast.parse(f.read(), path)
    out = set()
    for fn in tree.body:
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.Call) and isinstance(node.func, ast.Name) and node.func.id == name:
                    out.add(fn.name)
    return out


def test_package_never_imports_or_names_the_oracle():
    for path in glob.glob(os.path.join(PKG, "*.py")):
        assert _oracle_imports(path) == [], path
    for path in glob.glob(os.path.join(PKG, "csrc", "*")) + [os.path.join(ROOT, "include", "spin.h")]:
        with open(path) as f:
            text = f.read()
        for needle in ("liboracle", "spin_oracle", "oracle/", "oracle_"):
            assert needle not in text, (path, needle)


def test_bench_reaches_the_oracle_only_in_its_cpu_legs():
    bench = os.path.join(ROOT, "bench.py")
    funcs = {fn for _, stack in _oracle_imports(bench) for fn in stack}
    assert all(stack for _, stack in _oracle_imports(bench)), "no module-level oracle import"
    assert funcs <= {"oracle_sample", "run_reference"}, funcs
    # the sampled oracle run is called by the reference arm and by the CPU-baseline leg of
    # main(), which runs after the timed GPU region
    assert _callers(bench, "oracle_sample") <= {"run_reference", "main"}


def test_library_links_and_exports_nothing_of_the_oracle(spin_lib):
    dyn = subprocess.run(["readelf", "-d", spin.LIB_PATH], capture_output=True, text=True, check=True).stdout
    needed = [line for line in dyn.splitlines() if "(NEEDED)" in line]
    assert needed and not any("oracle" in line for line in needed), needed
    syms = subprocess.run(["nm", "-D", spin.LIB_PATH], capture_output=True, text=True, check=True).stdout
    assert "oracle" not in syms
