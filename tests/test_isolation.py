"""The oracle and the CUDA path stay apart, and the product stands alone (CPU).

The parity tests mean something only while the checker and the checked share
nothing: the package and the C header must not reach the oracle, the oracle
must not reach the CUDA sources, the seeded input generators must hold none of
either side, and nothing committed may depend on scratch files.
"""
import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sparse_attention_02_gb300")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d or "_objs" in d:
            continue
        for n in sorted(names):
            if n.endswith(exts):
                yield os.path.join(d, n)


SCRATCH = re.compile(r"(?<![A-Za-z0-9_])_work(?![A-Za-z0-9_])")


def _imports(path):
    """Top-level module names a Python file imports, anywhere in its body."""
    with open(path) as f:
        tree = ast.parse(f.read(), path)
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            mods.add(node.module.split(".")[0])
    return mods


PRODUCT_SOURCES = list(_files(PKG, (".py", ".cu", ".cuh", ".h"))) + list(_files(os.path.join(ROOT, "include"), (".h",)))


def test_product_sources_found():
    names = {os.path.basename(p) for p in PRODUCT_SOURCES}
    assert {"__init__.py", "sparse_mla.cu", "indexer.cu", "topk.cu", "warmup.cu", "dsa.h"} <= names


@pytest.mark.parametrize("path", PRODUCT_SOURCES, ids=lambda p: os.path.relpath(p, ROOT))
def test_product_never_reaches_the_oracle_or_scratch(path):
    with open(path, errors="replace") as f:
        text = f.read()
    if path.endswith(".py"):
        assert "oracle" not in _imports(path), "the product imports the oracle"
    assert not re.search(r"dsa_oracle|libdsa_oracle|[\"'/]oracle/", text), "the product names the oracle's files"
    assert not SCRATCH.search(text), "the product names the scratch folder"


def test_oracle_reaches_no_cuda_source():
    odir = os.path.join(ROOT, "oracle")
    for path in _files(odir, (".c", ".h", ".py")):
        with open(path) as f:
            text = f.read()
        # C: system headers only; Python: no import of the package, the generators or torch
        assert not re.search(r"#\s*include\s+\"", text), f"{path}: the oracle includes a local header"
        if path.endswith(".py"):
            assert not (_imports(path) & {"sparse_attention_02_gb300", "dsa_workloads", "torch"}), path


def test_input_generators_hold_neither_side():
    path = os.path.join(ROOT, "dsa_workloads", "__init__.py")
    assert not (_imports(path) & {"oracle", "sparse_attention_02_gb300"})


def test_bench_imports_the_oracle_only_inside_its_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    with open(path) as f:
        tree = ast.parse(f.read(), path)
    top = {a.name.split(".")[0] for n in tree.body if isinstance(n, ast.Import) for a in n.names}
    top |= {n.module.split(".")[0] for n in tree.body if isinstance(n, ast.ImportFrom) and n.module}
    assert "oracle" not in top
    inside = [f.name for f in ast.walk(tree) if isinstance(f, ast.FunctionDef)
              and any(isinstance(n, ast.Import) and any(a.name == "oracle" for a in n.names) for n in ast.walk(f))]
    assert inside == ["oracle_sample"], inside


def test_nothing_committed_reads_scratch():
    tracked = [os.path.join(ROOT, p) for p in ("bench.py", "__graft_entry__.py")]
    tracked += list(_files(os.path.join(ROOT, "tests"), (".py",)))
    tracked += list(_files(os.path.join(ROOT, "dsa_workloads"), (".py",)))
    me = os.path.abspath(__file__)
    for path in tracked:
        if os.path.abspath(path) == me:
            continue
        with open(path) as f:
            assert not SCRATCH.search(f.read()), path
