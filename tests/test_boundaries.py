"""The CUDA path and the oracle share no code: the package and its CUDA sources
never import or include anything under oracle/, the oracle never imports the
package or includes its sources, and the only module both sides read is the
seeded-input generator (scenes.py), which holds none of the method's
arithmetic."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "differentiable_rasterizer_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, dirs, files in os.walk(top):
        dirs[:] = [x for x in dirs if x not in ("_build", "__pycache__")]
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def _imports(path):
    tree = ast.parse(open(path).read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield ("." * node.level) + (node.module or "")


def test_package_never_imports_the_oracle():
    for p in _files(PKG, (".py",)):
        for name in _imports(p):
            assert not name.split(".")[0] == "oracle", (p, name)


def test_cuda_sources_include_nothing_from_the_oracle():
    for p in _files(PKG, (".cu", ".cuh", ".h")):
        for inc in re.findall(r'#include\s+"([^"]+)"', open(p).read()):
            assert "oracle" not in inc, (p, inc)


def test_oracle_never_imports_the_package_or_its_sources():
    for p in _files(ORACLE, (".py",)):
        for name in _imports(p):
            assert "differentiable_rasterizer_gb300" not in name, (p, name)
    for p in _files(ORACLE, (".c", ".h")):
        src = open(p).read()
        for inc in re.findall(r'#include\s+[<"]([^>"]+)[>"]', src):
            assert "csrc" not in inc and not inc.endswith((".cuh", "gs.h")), (p, inc)


def test_the_input_generator_holds_no_method_arithmetic():
    """scenes.py builds parameters, cameras and options; it calls neither side."""
    names = set(_imports(os.path.join(PKG, "scenes.py")))
    assert not any(n.split(".")[-1] in ("abi", "pipeline", "oracle") for n in names), names
