"""The oracle and the CUDA path share no code, and only test infrastructure
reaches the oracle (CPU only, a static check of imports and includes).

- The package (binding, stack driver, input generators, CUDA sources)
  neither imports nor includes anything under oracle/.
- The oracle imports nothing from the package and its C includes only
  system headers.
- bench.py imports the oracle only in its CPU-baseline and reference-arm
  functions; __graft_entry__.py only in build() (compiling it) and smoke().
"""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "int4_weight_only_q4f16_gb300")


def _imported_modules(tree):
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield node, a.name
        elif isinstance(node, ast.ImportFrom):
            yield node, node.module or ""


def _functions_importing(path, module):
    """Names of the top-level functions of `path` that import `module`
    (None for an import at module level)."""
    tree = ast.parse(open(path).read())
    found = []
    for top in tree.body:
        for node, name in _imported_modules(top):
            if name == module or name.startswith(module + "."):
                found.append(top.name if isinstance(top, ast.FunctionDef) else None)
    return found


def test_package_does_not_reach_the_oracle():
    for path in glob.glob(os.path.join(PKG, "*.py")):
        tree = ast.parse(open(path).read())
        for _, name in _imported_modules(tree):
            assert name.split(".")[0] != "oracle", path
    for path in glob.glob(os.path.join(PKG, "csrc", "*")):
        for line in open(path, errors="replace"):
            assert not re.match(r'\s*#\s*include\s*[<"].*oracle', line), (path, line)


def test_oracle_does_not_reach_the_package():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        tree = ast.parse(open(path).read())
        for _, name in _imported_modules(tree):
            assert not name.startswith("int4_weight_only_q4f16_gb300"), (path, name)
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.c")) + glob.glob(os.path.join(ROOT, "oracle", "*.h")):
        for line in open(path):
            if re.match(r"\s*#\s*include", line):
                assert re.match(r"\s*#\s*include\s*<[\w/.]+>", line), (path, line)


def test_only_test_infrastructure_imports_the_oracle():
    assert sorted(set(_functions_importing(os.path.join(ROOT, "bench.py"), "oracle"))) == \
        ["oracle_sample_rate", "run_oracle_table", "run_reference"]
    assert sorted(set(_functions_importing(os.path.join(ROOT, "__graft_entry__.py"), "oracle"))) == \
        ["build", "smoke"]
