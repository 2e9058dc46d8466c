"""The oracle and the CUDA path share no code, and the product never reaches the oracle.

Checked on the source text: the oracle imports only numpy, math and copy (nothing from the
package, the library or torch). The package and the CUDA sources never import,
include or load anything under oracle/.
"""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "linear_cross_entropy_forward_gb300")


def _imports(path):
    tree = ast.parse(open(path).read())
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            mods.add("." if node.level else (node.module or "").split(".")[0])
    return mods


def test_oracle_imports_only_the_standard_library_and_numpy():
    for name in os.listdir(os.path.join(ROOT, "oracle")):
        if name.endswith(".py"):
            mods = _imports(os.path.join(ROOT, "oracle", name)) - {"__future__", "."}
            assert mods <= {"numpy", "math", "copy"}, (name, mods)


def test_product_never_reaches_the_oracle():
    for name in os.listdir(PKG):
        if name.endswith(".py"):
            assert "oracle" not in _imports(os.path.join(PKG, name)), name
    for name in os.listdir(os.path.join(PKG, "csrc")):
        text = open(os.path.join(PKG, "csrc", name)).read()
        assert "oracle" not in text, name
    header = open(os.path.join(ROOT, "include", "flce.h")).read()
    assert "oracle" not in header
