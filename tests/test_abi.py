"""The C-ABI library builds, loads and exports every declared symbol (CPU only:
no compute call is made, only host-side argument checks that return before
any CUDA call)."""
import ctypes
import os
import re

import pytest

import chunked_prefill_gqa_gb300 as cp
from chunked_prefill_gqa_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ctypes.CDLL(B.LIB)


def test_header_declares_the_entry_points():
    names = _declared()
    assert set(names) == set(cp.EXPORTS), (sorted(names), sorted(cp.EXPORTS))


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_strerror_and_version(lib):
    cp._lib = None
    for code in range(-9, 1):
        assert cp.strerror(code) and "unknown" not in cp.strerror(code)
    assert "unknown" in cp.strerror(-99)
    assert "sm_103a" in cp.version()


def test_host_argument_checks_return_before_any_cuda_call():
    f = cp.raw("attn_prefill")
    good = 0x10000  # never dereferenced: every case below fails validation first
    assert f(good, good, good, good, -1, 0, None) == cp.ATTN_EINVAL
    assert f(good, good, good, good, 4, -1, None) == cp.ATTN_EINVAL
    assert f(good, good, good, good, cp.MAX_TOKENS + 1, 0, None) == cp.ATTN_ERANGE
    assert f(good, good, good, good, 16, cp.MAX_TOKENS, None) == cp.ATTN_ERANGE
    assert f(None, good, good, good, 4, 0, None) == cp.ATTN_EINVAL
    assert f(good, good, good, None, 4, 0, None) == cp.ATTN_EINVAL
    assert f(good + 4, good, good, good, 4, 0, None) == cp.ATTN_EALIGN
    assert f(good, good, good + 8, good, 4, 0, None) == cp.ATTN_EALIGN
    # an empty chunk is a valid no-op, pointers unused
    assert f(None, None, None, None, 0, 5, None) == cp.ATTN_OK
    for name in ("attn_prefill_ffma", "attn_reference_prefill"):
        g = cp.raw(name)
        assert g(good, good, good, good, -1, 0, None) == cp.ATTN_EINVAL
        assert g(None, None, None, None, 0, 0, None) == cp.ATTN_OK
    assert cp.raw("attn_full_causal")(good, good, good, good, -3, None) == cp.ATTN_EINVAL


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "chunked_prefill_gqa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in text.lower().replace("oracle-free", ""), os.path.join(dirpath, fn)
