"""The product path (the package and its CUDA sources) never imports, includes
or calls the oracle, and the oracle never includes the CUDA sources: the two
share only the seeded input generators."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "hybrid_linear_attention_kda_gb300")


def _files(top, exts):
    for dirpath, _, names in os.walk(top):
        if "_lib" in dirpath.split(os.sep) or "__pycache__" in dirpath:
            continue
        for nm in names:
            if nm.endswith(exts):
                yield os.path.join(dirpath, nm)


def test_package_does_not_use_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle[\s.]|#\s*include\s*[\"<][^\">]*oracle)", re.M)
    bad = [p for p in _files(PKG, (".py", ".cu", ".cuh", ".cpp", ".h")) if pat.search(open(p).read())]
    assert not bad, bad


def test_oracle_does_not_use_the_product():
    pat = re.compile(r"(hybrid_linear_attention_kda_gb300|#\s*include\s*[\"<][^\">]*(kda\.h|csrc))")
    bad = [p for p in _files(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")) if pat.search(open(p).read())]
    assert not bad, bad
