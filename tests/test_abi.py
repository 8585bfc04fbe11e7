"""The C ABI library builds for sm_103a, loads without a GPU, and exports every
function that include/*.h declares."""
import ctypes
import glob
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="no CUDA toolkit")
def test_library_exports_every_declared_symbol():
    from transformer_lm_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    names = _declared_functions()
    assert len(names) >= 25, names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_declares_the_same_names():
    from transformer_lm_gb300 import gpt2
    names = set(_declared_functions())
    assert names == set(gpt2._SIGS), names ^ set(gpt2._SIGS)
    # and a Python function of the same name for each
    missing = [n for n in names if not callable(getattr(gpt2, n, None))]
    assert not missing, missing


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="no CUDA toolkit")
def test_status_queries_through_the_binding_need_no_gpu():
    from transformer_lm_gb300 import build, gpt2
    build.build()
    assert gpt2.gpt2_last_status() in gpt2.ERRORS
    assert isinstance(gpt2.gpt2_last_error(), str) and gpt2.gpt2_last_error()
    assert gpt2.gpt2_launch_count() >= 0
