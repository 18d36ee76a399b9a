"""The C-ABI library builds, loads and exports every function include/np.h
declares (no GPU needed: nothing is called)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "np.h")


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:np_status|const char\*|int64_t)\s+(np_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from sparse_activation_decode_gb300.build import build
    path = build()
    import torch  # noqa: F401  (CUDA runtime)
    return ctypes.CDLL(path)


def test_header_declares_the_path():
    names = declared_functions()
    for required in ("np_init_model", "np_predict", "np_delta", "np_scatter", "np_sparse_mlp",
                     "np_decode_token", "np_free_model"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_header():
    from sparse_activation_decode_gb300 import _lib
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_status_strings_without_gpu(lib):
    lib.np_status_str.restype = ctypes.c_char_p
    assert lib.np_status_str(0) == b"ok"
    assert lib.np_status_str(-4) == b"storage read failed"


def test_init_rejects_null_desc_without_gpu(lib):
    out = ctypes.c_void_p()
    assert lib.np_init_model(None, ctypes.byref(out)) == -1
    assert not out.value
