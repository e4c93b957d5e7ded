"""The oracle and the CUDA path share nothing (no host code).

The product package never imports or links the oracle, the oracle includes only standard
C headers and imports neither the package nor its sources, and the seeded input
generators (synth/) import neither side.  Static checks of the source text.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _files(sub, exts):
    out = []
    for d, _, names in os.walk(os.path.join(ROOT, sub)):
        if "_build" in d or "__pycache__" in d:
            continue
        out += [os.path.join(d, n) for n in names if n.endswith(exts)]
    return out


def test_product_never_touches_the_oracle():
    for path in _files("gemm_decode_gb300", (".py", ".cu", ".cuh", ".h")):
        text = open(path).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), path
        assert "q4_oracle" not in text and "liboracle" not in text, path
    for path in _files("include", (".h",)):
        assert "oracle" not in open(path).read(), path


def test_oracle_uses_standard_headers_and_no_product_code():
    src = open(os.path.join(ROOT, "oracle", "q4_oracle.c")).read()
    includes = re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', src, re.M)
    assert includes and all(i in {"math.h", "stddef.h", "stdint.h", "string.h", "stdlib.h", "stdio.h"}
                            for i in includes), includes
    py = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert not re.search(r"^\s*(import|from)\s+(gemm_decode_gb300|synth)\b", py, re.M)
    assert "csrc" not in py and "libq4gemv" not in py


def test_input_generators_import_neither_side():
    py = open(os.path.join(ROOT, "synth", "__init__.py")).read()
    assert not re.search(r"^\s*(import|from)\s+(gemm_decode_gb300|oracle)\b", py, re.M)
