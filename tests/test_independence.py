"""Static checks (no GPU) that the oracle and the CUDA path stay apart: the
package never imports the oracle, the oracle never imports the package or
loads the library, and the two allowed callers outside tests/ (bench.py's
oracle timing, __graft_entry__.smoke) reach the oracle only from those
functions."""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "chunked_causal_attention_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(folder, exts):
    for dirpath, _, names in os.walk(folder):
        if "_build" in dirpath or "__pycache__" in dirpath:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(dirpath, n)


def _imports(tree):
    """(module name, enclosing function name or None) of every import in a module."""
    out = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(child, ast.Import):
                out.extend((a.name, fn) for a in child.names)
            elif isinstance(child, ast.ImportFrom) and child.module and child.level == 0:
                out.append((child.module, fn))
            visit(child, f)

    visit(tree, None)
    return out


def _top(name):
    return name.split(".")[0]


def test_package_never_imports_the_oracle():
    for path in _files(PKG, (".py",)):
        with open(path) as f:
            mods = _imports(ast.parse(f.read()))
        assert all(_top(m) != "oracle" for m, _ in mods), path
    for path in _files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".cpp", ".h")):
        with open(path) as f:
            src = f.read()
        assert "oracle/" not in src and '#include "oracle' not in src, path


def test_oracle_never_imports_the_package_or_the_library():
    for path in _files(ORACLE, (".py",)):
        with open(path) as f:
            src = f.read()
        mods = {_top(m) for m, _ in _imports(ast.parse(src))}
        # the standard library and numpy only: no package, no ctypes, no torch
        assert mods <= {"__future__", "typing", "dataclasses", "decimal", "math", "numpy", "oracle"}, (path, mods)
        assert "libattn" not in src, path


def test_oracle_callers_outside_tests():
    allowed = {"bench.py": {"time_oracle_sample"}, "__graft_entry__.py": {"smoke"}}
    for name, fns in allowed.items():
        with open(os.path.join(ROOT, name)) as f:
            mods = _imports(ast.parse(f.read()))
        callers = {fn for m, fn in mods if _top(m) == "oracle"}
        assert callers <= fns, (name, callers)
