"""The oracle and the CUDA path share nothing, and the product never reaches
the oracle: no module of the package imports it, no CUDA source includes its
files, the oracle includes or imports nothing of the package, and the
benchmark loads it only inside its CPU legs (the baseline and the reference
arm), never at module level."""
import ast
import glob
import os
import re

from conftest import ROOT

PKG = os.path.join(ROOT, "product_vq_kv_gb300")


def imported_modules(path: str, top_level_only: bool = False) -> set[str]:
    tree = ast.parse(open(path).read(), filename=path)
    nodes = tree.body if top_level_only else ast.walk(tree)
    names = set()
    for node in nodes:
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            names.add(node.module.split(".")[0])
    return names


def test_package_never_imports_the_oracle():
    files = glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True)
    assert files
    for path in files:
        assert "oracle" not in imported_modules(path), path


def test_cuda_sources_include_nothing_of_the_oracle():
    for path in glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*.h")):
        for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', open(path).read()):
            assert "oracle" not in inc, (path, inc)


def test_oracle_uses_nothing_of_the_package():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.c")) + glob.glob(os.path.join(ROOT, "oracle", "*.h")):
        for inc in re.findall(r'#include\s*[<"]([^>"]+)[>"]', open(path).read()):
            assert not inc.startswith("vq_") and "csrc" not in inc, (path, inc)
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        assert "product_vq_kv_gb300" not in imported_modules(path), path


def test_bench_loads_the_oracle_only_in_its_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    assert "oracle" not in imported_modules(path, top_level_only=True)
    tree = ast.parse(open(path).read())
    users = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.Import) and any(a.name == "oracle" for a in node.names):
                    users.add(fn.name)
    # the encode's CPU baseline, the reference arm, and the attention bench's
    # CPU baseline (skipped with --no-cpu-baseline)
    assert users == {"cpu_baseline", "bench_reference", "bench_attention"}, users
