"""The CUDA path and the oracle share no code.

The product package (``combine_ep_plan_gb300/``: binding, CUDA sources,
input generators) never imports, includes or loads the oracle, and the
oracle (``oracle/``) uses only the C and Python standard libraries and
numpy: neither side can pass the other's arithmetic off as its own.  The
seeded input generators are the one module both are fed from; they draw
inputs and do none of the method's arithmetic (no plan, no scatter, no
quantisation, no reduction).
"""
import ast
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PKG = os.path.join(ROOT, "combine_ep_plan_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _files(top, exts):
    for d, dirs, names in os.walk(top):
        dirs[:] = [x for x in dirs if not x.startswith((".", "_build", "__pycache__"))]
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _imports(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name.split(".")[0]
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            yield node.module.split(".")[0]


def test_package_never_imports_the_oracle():
    for path in _files(PKG, (".py",)):
        assert "oracle" not in set(_imports(path)), path


def test_cuda_sources_reference_no_oracle_file():
    for path in _files(PKG, (".cu", ".cuh", ".h", ".cpp", ".c")):
        text = open(path).read()
        assert "ep_oracle" not in text and "oracle/" not in text, path
    for path in _files(os.path.join(ROOT, "include"), (".h",)):
        assert "ep_oracle" not in open(path).read(), path


def test_oracle_uses_only_standard_headers_and_numpy():
    src = open(os.path.join(ORACLE, "ep_oracle.c")).read()
    includes = re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', src, re.M)
    # omp.h: the compiler's OpenMP runtime, for the multi-core build of the same source
    assert includes and set(includes) <= {"math.h", "stdint.h", "stdlib.h", "string.h", "omp.h"}, includes
    mods = set(_imports(os.path.join(ORACLE, "__init__.py")))
    assert mods <= {"__future__", "contextlib", "ctypes", "os", "subprocess", "tempfile", "dataclasses",
                    "numpy"}, mods


def test_input_generators_do_no_method_arithmetic():
    path = os.path.join(PKG, "inputs.py")
    mods = set(_imports(path))
    assert "oracle" not in mods and "combine_ep_plan_gb300" not in mods, mods
    # nothing that plans, scatters, quantises or reduces: only draws
    text = open(path).read()
    for word in ("e4m3", "float8", "448", "argsort(slot", "exp_src", "send_head", "recv_src_idx"):
        assert word not in text, word
