"""The double-precision CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (and its ``--impl reference`` arm) may import this package. The product
path (``chunked_prefill_gqa_gb300``) never imports it, and it never imports the
product path: the two share no code, header, table or constant. Inputs come
from ``workloads.py`` and are handed to both.

What it computes, and the passages it follows, is stated in
``attn_oracle.c``: exact causal grouped-query attention of a chunk of C query
rows at positions P..P+C-1 against keys 0..P+C-1, in double precision, two
passes per (row, head) with the maximum taken first.

The check rule of the attention-v1 oracle ("Inference Attention 2: Flash
Prefill Against a Cached Prefix", Lesson; "Inference Attention 1: The Full
Score Matrix", Lesson) is ``|got - ref| <= 1e-4 + 1e-3 * |ref|`` on every
value; :func:`check` applies it, and a non-finite value always fails.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

ATOL = 1e-4
RTOL = 1e-3


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` with gcc (-O2, OpenMP, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    lib.oracle_prefill.restype = ctypes.c_int
    lib.oracle_prefill.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_void_p, ctypes.c_long, ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def load_variant(path: str):
    """An ``attention`` callable bound to another build of the same C source.

    Used by the tests that compile deliberately broken copies of the oracle to
    show that the pins catch each mistake.
    """
    lib = _bind(ctypes.CDLL(path))
    return lambda *a, **kw: _attention(lib, *a, **kw)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def attention(q, k, v, P: int, scale: float = 0.125, rows=None, threads: int = 0) -> np.ndarray:
    """Exact causal GQA attention of chunk rows ``rows`` (default: all).

    q is [C][HQ][D], k and v are [P + C][HKV][D], fp32. Returns float64
    [len(rows)][HQ][D].
    """
    return _attention(_load(), q, k, v, P, scale, rows, threads)


def _attention(lib, q, k, v, P, scale=0.125, rows=None, threads=0):
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    if q.ndim != 3 or k.ndim != 3 or v.shape != k.shape:
        raise ValueError("q must be [C][HQ][D]; k and v [T][HKV][D] with equal shapes")
    C, HQ, D = q.shape
    T, HKV, Dk = k.shape
    if Dk != D or T != P + C or HQ % HKV != 0:
        raise ValueError(f"shape mismatch: q {q.shape}, k {k.shape}, P={P}")
    if rows is None:
        rows_arr = None
        nrows = C
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32)
        nrows = rows_arr.size
    out = np.empty((nrows, HQ, D), dtype=np.float64)
    rc = lib.oracle_prefill(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, out.ctypes.data,
        C, P, HQ, HKV, D, float(scale),
        None if rows_arr is None else rows_arr.ctypes.data, nrows, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_prefill failed with code {rc}")
    return out


def prefill(inp, rows=None, threads: int = 0) -> np.ndarray:
    """The oracle on a ``workloads.Inputs`` (scale 1/8)."""
    return attention(inp.q, inp.k, inp.v, inp.P, 0.125, rows=rows, threads=threads)


def gather_pages(pages, table, T: int, page: int = 16) -> np.ndarray:
    """The contiguous [T][HKV][D] cache a paged one stands for: token t is slot
    t % page of physical page table[t // page] ("FlashAttention and inference
    kernels", PagedAttention)."""
    t = np.arange(T)
    return np.ascontiguousarray(pages[np.asarray(table)[t // page], t % page])


def prefill_paged(q, k_pages, v_pages, table, P: int, rows=None, threads: int = 0) -> np.ndarray:
    """The oracle against a paged cache: gather by the block table, then the
    same exact attention as :func:`attention` (scale 1/8)."""
    T = P + q.shape[0]
    return attention(q, gather_pages(k_pages, table, T), gather_pages(v_pages, table, T), P, 0.125,
                     rows=rows, threads=threads)


def score_matrix(q, k, P: int, scale: float = 0.125) -> np.ndarray:
    """The score workspace of the three-kernel pipeline ("Inference Attention 1:
    The Full Score Matrix", Lesson): S[h][i][j] = q[i][h] . k[j][h / 4] * scale
    in float64 for keys j <= P + i, -inf above that diagonal. Shape
    [HQ][C][P + C]; one float64 matmul per head."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    C, HQ, _ = q.shape
    T, HKV, _ = k.shape
    if T != P + C:
        raise ValueError(f"k has {T} rows, expected P + C = {P + C}")
    group = HQ // HKV
    allowed = np.arange(T)[None, :] <= (P + np.arange(C))[:, None]
    S = np.empty((HQ, C, T))
    for h in range(HQ):
        S[h] = np.where(allowed, (q[:, h, :] @ k[:, h // group, :].T) * scale, -np.inf)
    return S


def probability_matrix(S) -> np.ndarray:
    """Each row of a score workspace replaced by its softmax, maximum subtracted
    first (same page: the row softmax of the middle kernel; -inf becomes 0)."""
    S = np.asarray(S, dtype=np.float64)
    E = np.exp(S - S.max(axis=-1, keepdims=True))
    return E / E.sum(axis=-1, keepdims=True)


def bf16_to_float(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) as the fp32 values they encode: a bf16 is
    the upper half of the IEEE binary32 with the same sign, exponent and leading
    fraction bits, so the value is the binary32 whose low 16 bits are zero."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def prefill_bf16kv(q, k_bits, v_bits, P: int, rows=None, threads: int = 0) -> np.ndarray:
    """The oracle for a bf16 K/V cache: the exact attention (scale 1/8) over
    the values the stored bf16 keys and values encode."""
    return attention(q, bf16_to_float(k_bits), bf16_to_float(v_bits), P, 0.125, rows=rows, threads=threads)


def violations(got, ref, atol: float = ATOL, rtol: float = RTOL) -> np.ndarray:
    """Boolean mask of elements failing |got - ref| <= atol + rtol * |ref| (NaN fails)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ok = np.abs(got - ref) <= atol + rtol * np.abs(ref)
    ok &= np.isfinite(got)
    return ~ok


def check(got, ref, atol: float = ATOL, rtol: float = RTOL) -> dict:
    """Apply the attention-v1 rule; report the worst element as err / tolerance."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = violations(got, ref, atol, rtol)
    with np.errstate(invalid="ignore"):
        ratio = np.abs(got - ref) / (atol + rtol * np.abs(ref))
    ratio = np.where(np.isfinite(got), ratio, np.inf)
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return {"n": int(got.size), "n_bad": int(bad.sum()), "worst_ratio": worst,
            "max_abs_err": float(np.nanmax(np.abs(got - ref))) if got.size else 0.0}
