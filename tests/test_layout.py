"""Repository-level checks that need no GPU: the build compiles every CUDA
source of the package, and the product path never reaches the oracle."""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "dynamic_sparse_attention_slash_gb300")


def test_build_lists_every_cuda_source():
    from dynamic_sparse_attention_slash_gb300 import build
    on_disk = sorted(f for f in os.listdir(os.path.join(PKG, "csrc")) if f.endswith(".cu"))
    assert sorted(build.SOURCES) == on_disk


def _imported_modules(path):
    tree = ast.parse(open(path).read(), filename=path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom) and node.module:
            yield node.module


def test_package_never_imports_the_oracle():
    """Only tests, smoke() and the bench's CPU legs may use oracle/."""
    for f in sorted(os.listdir(PKG)):
        if f.endswith(".py"):
            mods = list(_imported_modules(os.path.join(PKG, f)))
            assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), f


def test_oracle_imports_nothing_from_the_package():
    path = os.path.join(ROOT, "oracle", "msa_oracle.py")
    mods = list(_imported_modules(path))
    assert not any(m.startswith("dynamic_sparse_attention_slash_gb300") for m in mods)
