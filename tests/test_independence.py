"""Static checks, on the CPU, that the CUDA path and the oracle share no code.

The oracle is test infrastructure: the library (its Python binding, its CUDA
sources and the public header) never imports, includes or loads anything of
it, and the oracle never uses the library's code.  The seeded input
generators in `synthetic` serve both sides and depend on neither.  The bench
may run the oracle only in its CPU-baseline leg (one function).
"""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "transformer_attention_iha_gb300"


def _py(pattern: str):
    return sorted(glob.glob(os.path.join(ROOT, pattern), recursive=True))


def _imports(path: str):
    """(top-level module, enclosing function or None) of every import."""
    tree = ast.parse(open(path).read(), path)
    out = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(child, ast.Import):
                out.extend((a.name.split(".")[0], func) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                if child.level == 0 and child.module:
                    out.append((child.module.split(".")[0], func))
            visit(child, f)

    visit(tree, None)
    return out


def test_library_python_never_imports_the_oracle_or_the_generators():
    files = _py(f"{PKG}/**/*.py")
    assert files
    for f in files:
        mods = {m for m, _ in _imports(f)}
        assert "oracle" not in mods, f
        assert "synthetic" not in mods, f


def test_cuda_sources_and_header_never_reference_the_oracle():
    files = _py(f"{PKG}/csrc/*") + _py("include/*.h")
    assert any(f.endswith(".cu") for f in files)
    inc = re.compile(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', re.M)
    for f in files:
        text = open(f).read()
        for name in inc.findall(text):
            assert "oracle" not in name, (f, name)
        assert "iha_oracle" not in text and "dlopen" not in text, f


def test_oracle_never_uses_the_library():
    for f in _py("oracle/*.py"):
        mods = {m for m, _ in _imports(f)}
        assert PKG not in mods and "synthetic" not in mods, f
        assert "csrc" not in open(f).read(), f
    inc = re.compile(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', re.M)
    for f in _py("oracle/*.c") + _py("oracle/*.h"):
        for name in inc.findall(open(f).read()):
            assert name in ("math.h", "stdlib.h", "stdint.h", "string.h", "omp.h",
                            "stddef.h", "stdio.h"), (f, name)


def test_generators_depend_on_neither_side():
    for f in _py("synthetic/*.py"):
        mods = {m for m, _ in _imports(f)}
        assert not mods & {"oracle", PKG, "torch"}, (f, mods)


def test_bench_runs_the_oracle_only_in_its_cpu_leg():
    uses = [(m, fn) for m, fn in _imports(os.path.join(ROOT, "bench.py")) if m == "oracle"]
    assert uses, "the CPU-baseline leg imports the oracle"
    assert {fn for _, fn in uses} == {"oracle_sample"}, uses
