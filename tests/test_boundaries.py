"""The oracle and the CUDA path share no code: product sources neither import
nor include anything under oracle/, the oracle neither imports the package nor
includes its headers, the shared input generators import neither side, and the
only callers of the oracle outside tests/ are bench.py's CPU timers and the
entry module's build (which compiles it) and smoke (which checks against it)."""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "causal_scaled_dot_gb300")


def _imports(path):
    """(module, enclosing function name or None) for every import in a file."""
    tree = ast.parse(open(path).read(), path)
    found = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)):
                visit(child, child.name)
            elif isinstance(child, ast.ClassDef):
                visit(child, fn)
            else:
                if isinstance(child, ast.Import):
                    found.extend((a.name, fn) for a in child.names)
                elif isinstance(child, ast.ImportFrom) and child.module:
                    found.append((child.module, fn))
                visit(child, fn)

    visit(tree, None)
    return found


def _includes(path):
    return re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', open(path).read(), re.M)


def _top(mod):
    return mod.split(".")[0]


def test_product_path_never_reaches_the_oracle():
    for path in glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True):
        assert all(_top(m) != "oracle" for m, _ in _imports(path)), path
    for path in (glob.glob(os.path.join(PKG, "csrc", "*.cu*")) + glob.glob(os.path.join(PKG, "csrc", "*.h"))
                 + glob.glob(os.path.join(ROOT, "include", "*.h"))):
        assert not any("oracle" in inc for inc in _includes(path)), path


def test_oracle_never_reaches_the_product_path():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        assert all(_top(m) != "causal_scaled_dot_gb300" for m, _ in _imports(path)), path
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.c")) + glob.glob(os.path.join(ROOT, "oracle", "*.h")):
        for inc in _includes(path):
            assert "attn.h" not in inc and "csrc" not in inc and ".cuh" not in inc, (path, inc)


def test_shared_input_generators_import_neither_side():
    mods = {_top(m) for m, _ in _imports(os.path.join(PKG, "inputs.py"))}
    assert "oracle" not in mods
    assert not any(m.startswith("causal_scaled_dot_gb300.native") for m, _ in
                   _imports(os.path.join(PKG, "inputs.py")))


def test_oracle_callers_outside_tests():
    bench = [fn for m, fn in _imports(os.path.join(ROOT, "bench.py")) if _top(m) == "oracle"]
    assert bench and None not in bench  # only inside the CPU timers, never at module level
    entry = {fn for m, fn in _imports(os.path.join(ROOT, "__graft_entry__.py")) if _top(m) == "oracle"}
    assert entry <= {"build", "smoke"}
