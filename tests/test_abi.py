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
    codes = [v for k, v in vars(cp).items() if k.startswith("ATTN_E") or k == "ATTN_OK"]
    assert sorted(codes) == list(range(-11, 1))
    for code in codes:
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


def test_header_and_binding_codes_agree():
    """Every ATTN_E* code and size constant in the header has the same value in
    the binding."""
    text = open(os.path.join(ROOT, "include", "attn_prefill.h")).read()
    defs = dict(re.findall(r"#define (ATTN_\w+)\s+(-?\d+)", text))
    for name, val in defs.items():
        if name.startswith("ATTN_E") or name == "ATTN_OK":
            assert getattr(cp, name) == int(val), name
    assert cp.PAGE == int(defs["ATTN_PAGE"])
    assert cp.DECODE_SCRATCH_BYTES == 4 << 20 and "(4u << 20)" in text


def test_size_helpers_reject_bad_sizes_without_a_gpu(lib):
    lib.attn_naive_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_naive_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    assert lib.attn_naive_workspace_bytes(-1, 0) == 0
    assert lib.attn_naive_workspace_bytes(17, 5) == 32 * 17 * 22 * 4
    lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_decode_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    assert lib.attn_decode_workspace_bytes(0, 100, 0) == 0
    assert lib.attn_decode_workspace_bytes(4, -1, 0) == 0


@pytest.mark.parametrize("name", ["attn_prefill_host", "attn_prefill_bf16x3_host", "attn_prefill_bf16kv_host"])
def test_host_buffer_argument_checks_return_before_any_cuda_call(name):
    f = cp.raw(name)
    good = 0x10000
    host = [good] * 4
    dev = [good] * 4
    assert f(*host, *dev, 0, 5, None) == cp.ATTN_OK  # empty chunk: nothing is touched
    assert f(None, None, None, None, None, None, None, None, 0, 5, None) == cp.ATTN_OK
    assert f(*host, *dev, -1, 0, None) == cp.ATTN_EINVAL
    assert f(*host, *dev, 4, -1, None) == cp.ATTN_EINVAL
    assert f(*host, *dev, cp.MAX_TOKENS + 1, 0, None) == cp.ATTN_ERANGE
    for i in range(4):
        h = list(host); h[i] = None
        assert f(*h, *dev, 4, 0, None) == cp.ATTN_EINVAL, i
        d = list(dev); d[i] = None
        assert f(*host, *d, 4, 0, None) == cp.ATTN_EINVAL, i
        d = list(dev); d[i] = good + 4
        assert f(*host, *d, 4, 0, None) == cp.ATTN_EALIGN, i


def test_host_buffer_binding_checks_tensors():
    torch = pytest.importorskip("torch")
    C, P = 3, 2
    q = torch.zeros(C, 32, 64)
    kv = torch.zeros(P + C, 8, 64)
    with pytest.raises(ValueError):  # device buffers on the CPU
        cp.attn_prefill_host(q, kv, kv, q, q, kv, kv, q, P)
    with pytest.raises(ValueError):  # wrong K/V shape
        cp.attn_prefill_host(q, kv[:-1], kv, q, q, kv, kv, q, P)
    with pytest.raises(ValueError):  # fp32 where the bf16 cache is required
        cp.attn_prefill_bf16kv_host(q, kv, kv, q, q, kv, kv, q, P)
    with pytest.raises(TypeError):
        cp.attn_prefill_host(q.numpy(), kv, kv, q, q, kv, kv, q, P)


def test_decode_and_matrix_argument_checks_return_before_any_cuda_call():
    good = 0x10000
    f = cp.raw("attn_decode_paged")
    assert f(good, good, good, good, good, good, -1, 1, 1, 16, 0, None, 0, None) == cp.ATTN_EINVAL
    assert f(good, good, good, good, good, good, 2, 0, 1, 16, 0, None, 0, None) == cp.ATTN_EINVAL
    assert f(good, good, good, good, good, good, 2, 1, 1, 17, 0, None, 0, None) == cp.ATTN_ERANGE  # > 16 * maxBlocks
    assert f(None, None, None, None, None, None, 0, 1, 1, 16, 0, None, 0, None) == cp.ATTN_OK
    g = cp.raw("attn_decode_paged_noalloc")
    assert g(good, good, good, good, good, good, 70000, 1, 1, 16, 0, None) == cp.ATTN_ERANGE
    assert g(None, good, good, good, good, good, 2, 1, 1, 16, 0, None) == cp.ATTN_EINVAL
    h = cp.raw("attn_naive_prefill")
    assert h(good, good, good, good, good, 1 << 30, -1, 0, None) == cp.ATTN_EINVAL
    assert h(None, None, None, None, None, 0, 0, 7, None) == cp.ATTN_OK
    assert cp.raw("attn_prefill_bf16kv")(good, good + 2, good, good, 4, 0, None) == cp.ATTN_EALIGN


def test_tensor_peak_argument_checks_return_before_any_cuda_call():
    f = cp.raw("attn_tensor_peak")
    assert f(2, 128, 16, 1, None) == cp.ATTN_EINVAL       # kind is 0 (tf32) or 1 (bf16)
    assert f(0, 0, 16, 1, None) == cp.ATTN_EINVAL         # n in [16, 256], a multiple of 16
    assert f(0, 264, 16, 1, None) == cp.ATTN_EINVAL
    assert f(0, 120, 16, 1, None) == cp.ATTN_EINVAL
    assert f(0, 128, 0, 1, None) == cp.ATTN_EINVAL        # iters in [1, 2^22]
    assert f(0, 128, (1 << 22) + 1, 1, None) == cp.ATTN_EINVAL
    assert f(1, 256, 16, 0, None) == cp.ATTN_EINVAL       # ctas in [1, 65535]
