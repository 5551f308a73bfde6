"""Python binding of libattnprefill.so (argument marshalling only).

Every function here has the name of a C entry point declared in
``include/attn_prefill.h`` and does nothing but check tensor shapes, dtypes
and devices, pass raw device pointers and the current CUDA stream, and raise
:class:`AttnError` on a nonzero return code. All arithmetic runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback. If the library
is missing, importing the functions works but every call raises.

Tensors (attention-v1 contract): q [C][32][64], kCache and vCache
[P + C][8][64], out [C][32][64], fp32, contiguous, on the current CUDA device.
"""
from __future__ import annotations

import ctypes
import os
import threading

HQ, HKV, D = 32, 8, 64

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libattnprefill.so")

ATTN_OK = 0
ATTN_EINVAL = -1
ATTN_EALIGN = -2
ATTN_ERANGE = -3
ATTN_ELAUNCH = -4
ATTN_ETIMEOUT = -5
ATTN_EBOUNDS = -6
ATTN_EDEVICE = -7
ATTN_ETMA = -8
ATTN_ECUDA = -9
ATTN_ESPACE = -10
ATTN_ESCRATCH = -11
DECODE_SCRATCH_BYTES = 4 << 20
MAX_TOKENS = 1 << 24
PAGE = 16

# Every symbol the header declares (the CPU tests check the library exports them).
EXPORTS = ("attn_prefill", "attn_prefill_bf16x3", "attn_prefill_bf16kv", "attn_prefill_host",
           "attn_prefill_bf16x3_host", "attn_prefill_bf16kv_host", "attn_full_causal", "attn_prefill_paged", "attn_decode_paged",
           "attn_decode_workspace_bytes", "attn_decode_paged_noalloc",
           "attn_naive_workspace_bytes", "attn_naive_scores", "attn_naive_softmax", "attn_naive_weighted_sum",
           "attn_naive_prefill", "attn_prefill_ffma", "attn_reference_prefill", "attn_selftest_timeout",
           "attn_selftest_decode_timeout", "attn_tensor_peak", "attn_get_device_error", "attn_strerror",
           "attn_version")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


def library_path() -> str:
    return LIB_PATH


def load():
    """Load the shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m chunked_prefill_gqa_gb300.build` "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(LIB_PATH)
            vp, ci = ctypes.c_void_p, ctypes.c_int
            for name in ("attn_prefill", "attn_prefill_bf16x3", "attn_prefill_ffma", "attn_reference_prefill",
                         "attn_selftest_timeout"):
                fn = getattr(lib, name)
                fn.restype = ci
                fn.argtypes = [vp, vp, vp, vp, ci, ci, vp]
            lib.attn_prefill_bf16kv.restype = ci
            lib.attn_prefill_bf16kv.argtypes = [vp, vp, vp, vp, ci, ci, vp]
            for name in ("attn_prefill_host", "attn_prefill_bf16x3_host", "attn_prefill_bf16kv_host"):
                fn = getattr(lib, name)
                fn.restype = ci
                fn.argtypes = [vp] * 8 + [ci, ci, vp]
            lib.attn_prefill_paged.restype = ci
            lib.attn_prefill_paged.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, vp]
            for name in ("attn_decode_paged", "attn_selftest_decode_timeout"):
                fn = getattr(lib, name)
                fn.restype = ci
                fn.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, vp, ctypes.c_size_t, vp]
            lib.attn_decode_paged_noalloc.restype = ci
            lib.attn_decode_paged_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, vp]
            lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_decode_workspace_bytes.argtypes = [ci, ci, ci]
            lib.attn_naive_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_naive_workspace_bytes.argtypes = [ci, ci]
            lib.attn_naive_scores.restype = ci
            lib.attn_naive_scores.argtypes = [vp, vp, vp, ci, ci, vp]
            lib.attn_naive_softmax.restype = ci
            lib.attn_naive_softmax.argtypes = [vp, ci, ci, vp]
            lib.attn_naive_weighted_sum.restype = ci
            lib.attn_naive_weighted_sum.argtypes = [vp, vp, vp, ci, ci, vp]
            lib.attn_naive_prefill.restype = ci
            lib.attn_naive_prefill.argtypes = [vp, vp, vp, vp, vp, ctypes.c_size_t, ci, ci, vp]
            lib.attn_full_causal.restype = ci
            lib.attn_full_causal.argtypes = [vp, vp, vp, vp, ci, vp]
            lib.attn_tensor_peak.restype = ci
            lib.attn_tensor_peak.argtypes = [ci, ci, ci, ci, vp]
            lib.attn_get_device_error.restype = ci
            lib.attn_get_device_error.argtypes = []
            lib.attn_strerror.restype = ctypes.c_char_p
            lib.attn_strerror.argtypes = [ci]
            lib.attn_version.restype = ctypes.c_char_p
            lib.attn_version.argtypes = []
            _lib = lib
    return _lib


def strerror(code: int) -> str:
    try:
        return load().attn_strerror(int(code)).decode()
    except Exception:  # library missing: still produce a message
        return f"error {code}"


def version() -> str:
    return load().attn_version().decode()


def _stream_handle(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_tensors(q, k, v, out, C, P):
    import torch
    for name, t, shape in (("q", q, (C, HQ, D)), ("kCache", k, (P + C, HKV, D)),
                           ("vCache", v, (P + C, HKV, D)), ("out", out, (C, HQ, D))):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32, got {t.dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")


def _call(name, q, k, v, out, P, stream):
    C = q.shape[0]
    _check_tensors(q, k, v, out, C, P)
    rc = getattr(load(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(out), C, P, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, name)
    return out


def attn_prefill(q, kCache, vCache, out, P: int, stream=None):
    """out <- causal GQA attention of chunk q at offset P (tensor-core path)."""
    return _call("attn_prefill", q, kCache, vCache, out, P, stream)


def attn_prefill_bf16x3(q, kCache, vCache, out, P: int, stream=None):
    """attn_prefill on the bf16 tensor-core path (three of four split products)."""
    return _call("attn_prefill_bf16x3", q, kCache, vCache, out, P, stream)


def attn_prefill_bf16kv(q, kCache, vCache, out, P: int, stream=None):
    """attn_prefill against a bf16 K/V cache: kCache, vCache are contiguous
    torch.bfloat16 (or int16/uint16 bit patterns) CUDA tensors [P + C][8][64];
    q and out fp32 [C][32][64]."""
    import torch
    C = q.shape[0]
    for name, t, shape in (("q", q, (C, HQ, D)), ("out", out, (C, HQ, D))):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape {shape}")
    for name, t in (("kCache", kCache), ("vCache", vCache)):
        if (t.dtype not in (torch.bfloat16, torch.int16, torch.uint16) or not t.is_cuda or not t.is_contiguous()
                or tuple(t.shape) != (P + C, HKV, D)):
            raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor of shape ({P + C}, {HKV}, {D})")
    rc = load().attn_prefill_bf16kv(_ptr(q), _ptr(kCache), _ptr(vCache), _ptr(out), C, int(P),
                                    _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_prefill_bf16kv")
    return out


def _check_host_call(host, dev, C, P, kv_dtypes):
    import torch
    shapes = ((C, HQ, D), (P + C, HKV, D), (P + C, HKV, D), (C, HQ, D))
    names = ("q", "kCache", "vCache", "out")
    for i, (name, shape) in enumerate(zip(names, shapes)):
        dtypes = kv_dtypes if i in (1, 2) else (torch.float32,)
        for where, t, on_gpu in (("_host", host[i], False), ("_dev", dev[i], True)):
            if not isinstance(t, torch.Tensor):
                raise TypeError(f"{name}{where} must be a torch.Tensor")
            if t.dtype not in dtypes or t.is_cuda != on_gpu or not t.is_contiguous() or tuple(t.shape) != shape:
                raise ValueError(f"{name}{where} must be a contiguous {'CUDA' if on_gpu else 'CPU'} tensor "
                                 f"of dtype {dtypes[0]} and shape {shape}")


def _call_host(name, host, dev, P, stream, kv_dtypes):
    C = host[0].shape[0]
    _check_host_call(host, dev, C, P, kv_dtypes)
    rc = getattr(load(), name)(*[_ptr(t) for t in host], *[_ptr(t) for t in dev], C, int(P), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, name)
    return host[3]


def attn_prefill_host(q_host, k_host, v_host, out_host, q_dev, k_dev, v_dev, out_dev, P: int, stream=None):
    """attn_prefill from CPU tensors (pin them for copy/compute overlap) through
    the caller's CUDA tensors of the same shapes; returns out_host, complete
    once the stream is synchronised."""
    import torch
    return _call_host("attn_prefill_host", (q_host, k_host, v_host, out_host), (q_dev, k_dev, v_dev, out_dev), P,
                      stream, (torch.float32,))


def attn_prefill_bf16x3_host(q_host, k_host, v_host, out_host, q_dev, k_dev, v_dev, out_dev, P: int, stream=None):
    """attn_prefill_bf16x3 from CPU tensors, as attn_prefill_host."""
    import torch
    return _call_host("attn_prefill_bf16x3_host", (q_host, k_host, v_host, out_host), (q_dev, k_dev, v_dev, out_dev),
                      P, stream, (torch.float32,))


def attn_prefill_bf16kv_host(q_host, k_host, v_host, out_host, q_dev, k_dev, v_dev, out_dev, P: int, stream=None):
    """attn_prefill_bf16kv from CPU tensors, as attn_prefill_host; the K/V
    tensors (host and device) are bfloat16 or their int16/uint16 patterns."""
    import torch
    return _call_host("attn_prefill_bf16kv_host", (q_host, k_host, v_host, out_host), (q_dev, k_dev, v_dev, out_dev),
                      P, stream, (torch.bfloat16, torch.int16, torch.uint16))


def attn_full_causal(q, k, v, out, stream=None):
    """out <- causal GQA attention of a whole prompt (P = 0)."""
    T = q.shape[0]
    _check_tensors(q, k, v, out, T, 0)
    rc = load().attn_full_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), T, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_full_causal")
    return out


def attn_prefill_paged(q, kPages, vPages, blockTable, out, P: int, stream=None):
    """out <- attn_prefill against a paged cache: token t at slot t % 16 of page
    blockTable[t // 16]; kPages / vPages [numPages][16][8][64] fp32, blockTable
    int32 with at least ceil((P + C) / 16) entries."""
    import torch
    C = q.shape[0]
    if not (isinstance(kPages, torch.Tensor) and kPages.dim() == 4 and tuple(kPages.shape[1:]) == (PAGE, HKV, D)):
        raise ValueError("kPages must be [numPages][16][8][64]")
    if vPages.shape != kPages.shape:
        raise ValueError("vPages must have kPages' shape")
    if not (isinstance(blockTable, torch.Tensor) and blockTable.dtype == torch.int32 and blockTable.is_cuda
            and blockTable.is_contiguous()):
        raise TypeError("blockTable must be a contiguous int32 CUDA tensor")
    if blockTable.numel() < (P + C + PAGE - 1) // PAGE:
        raise ValueError("blockTable has fewer than ceil((P + C) / 16) entries")
    num_pages = kPages.shape[0]
    flat_k = kPages.view(num_pages * PAGE, HKV, D)
    flat_v = vPages.view(num_pages * PAGE, HKV, D)
    for name, t in (("q", q), ("out", out)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (C, HQ, D):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape ({C}, {HQ}, {D})")
    for name, t in (("kPages", flat_k), ("vPages", flat_v)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    rc = load().attn_prefill_paged(_ptr(q), _ptr(kPages), _ptr(vPages), _ptr(blockTable), _ptr(out),
                                   C, P, num_pages, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_prefill_paged")
    return out


def attn_decode_workspace_bytes(B: int, max_context: int, num_splits: int = 0) -> int:
    """Bytes of workspace attn_decode_paged needs on the current device."""
    return int(load().attn_decode_workspace_bytes(int(B), int(max_context), int(num_splits)))


def attn_decode_paged(q, kPages, vPages, blockTable, contextLens, out, max_context: int,
                      num_splits: int = 0, workspace=None, stream=None):
    """One decode step: q, out [B][32][64]; kPages/vPages [numPages][16][8][64];
    blockTable int32 [B][maxBlocks]; contextLens int32 [B] (device), each <=
    max_context. ``workspace``: a CUDA tensor of at least
    attn_decode_workspace_bytes(B, max_context, num_splits) bytes, or None when
    none is needed."""
    import torch
    B = q.shape[0]
    for name, t in (("q", q), ("out", out)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, HQ, D):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape ({B}, {HQ}, {D})")
    for name, t in (("kPages", kPages), ("vPages", vPages)):
        if (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4
                or tuple(t.shape[1:]) != (PAGE, HKV, D)):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor [numPages][16][8][64]")
    if blockTable.dtype != torch.int32 or not blockTable.is_cuda or blockTable.dim() != 2 or blockTable.shape[0] != B:
        raise ValueError("blockTable must be an int32 CUDA tensor [B][maxBlocks]")
    if contextLens.dtype != torch.int32 or not contextLens.is_cuda or contextLens.numel() != B:
        raise ValueError("contextLens must be an int32 CUDA tensor [B]")
    return _decode_call("attn_decode_paged", q, kPages, vPages, blockTable.contiguous(), contextLens, out,
                        max_context, num_splits, workspace, stream)


def _decode_call(name, q, kPages, vPages, blockTable, contextLens, out, max_context, num_splits, workspace, stream):
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = getattr(load(), name)(_ptr(q), _ptr(kPages), _ptr(vPages), _ptr(blockTable), _ptr(contextLens),
                               _ptr(out), q.shape[0], blockTable.shape[1], kPages.shape[0], int(max_context),
                               int(num_splits), ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, name)
    return out


def attn_selftest_decode_timeout(q, kPages, vPages, blockTable, contextLens, out, max_context: int,
                                 num_splits: int = 0, workspace=None, stream=None):
    """Failure-path test of the decode kernel (arguments as attn_decode_paged):
    every block's first K/V tile is withheld, its wait expires after 20 ms and
    ATTN_ETIMEOUT is recorded; read it with attn_get_device_error()."""
    return _decode_call("attn_selftest_decode_timeout", q, kPages, vPages, blockTable.contiguous(), contextLens, out,
                        max_context, num_splits, workspace, stream)


def _check_decode_args(q, kPages, vPages, blockTable, contextLens, out):
    import torch
    B = q.shape[0]
    for name, t in (("q", q), ("out", out)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, HQ, D):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape ({B}, {HQ}, {D})")
    for name, t in (("kPages", kPages), ("vPages", vPages)):
        if (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4
                or tuple(t.shape[1:]) != (PAGE, HKV, D)):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor [numPages][16][8][64]")
    if blockTable.dtype != torch.int32 or not blockTable.is_cuda or blockTable.dim() != 2 or blockTable.shape[0] != B:
        raise ValueError("blockTable must be an int32 CUDA tensor [B][maxBlocks]")
    if contextLens.dtype != torch.int32 or not contextLens.is_cuda or contextLens.numel() != B:
        raise ValueError("contextLens must be an int32 CUDA tensor [B]")


def attn_decode_paged_noalloc(q, kPages, vPages, blockTable, contextLens, out, max_context: int,
                              num_splits: int = 0, stream=None):
    """attn_decode_paged with the partials in the library's fixed 4 MiB device
    scratch instead of a caller workspace: nothing is allocated. For callers
    that cannot provide device memory. Calls that may overlap (other streams,
    other threads) race on the shared scratch; the first call on a device looks
    up its address and should come before any stream capture."""
    _check_decode_args(q, kPages, vPages, blockTable, contextLens, out)
    blockTable = blockTable.contiguous()
    rc = load().attn_decode_paged_noalloc(_ptr(q), _ptr(kPages), _ptr(vPages), _ptr(blockTable),
                                          _ptr(contextLens), _ptr(out), q.shape[0], blockTable.shape[1],
                                          kPages.shape[0], int(max_context), int(num_splits),
                                          _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_paged_noalloc")
    return out


def attn_naive_workspace_bytes(C: int, P: int) -> int:
    """Bytes of the score matrix [32][C][P + C] fp32."""
    return int(load().attn_naive_workspace_bytes(int(C), int(P)))


def _naive_scores_arg(scores, C: int, P: int):
    import torch
    if (scores.dtype != torch.float32 or not scores.is_cuda or not scores.is_contiguous()
            or scores.numel() * 4 < attn_naive_workspace_bytes(C, P)):
        raise ValueError(f"scores must be a contiguous float32 CUDA tensor of at least 32 x {C} x {P + C} elements")
    return scores.data_ptr()


def attn_naive_prefill(q, kCache, vCache, out, scores, P: int, stream=None):
    """The three-kernel score-matrix pipeline: scores, in-place row softmax,
    weighted sum, with ``scores`` the [32][C][P + C] fp32 workspace."""
    C = q.shape[0]
    _check_tensors(q, kCache, vCache, out, C, P)
    ws = _naive_scores_arg(scores, C, P)
    rc = load().attn_naive_prefill(_ptr(q), _ptr(kCache), _ptr(vCache), _ptr(out), ws,
                                   scores.numel() * 4, C, int(P), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_naive_prefill")
    return out


def attn_naive_scores(q, kCache, scores, P: int, stream=None):
    """Step 1: scores[h][i][j] = q[i][h] . k[j][h/4] / 8, -inf above the diagonal."""
    C = q.shape[0]
    ws = _naive_scores_arg(scores, C, P)
    rc = load().attn_naive_scores(_ptr(q), _ptr(kCache), ws, C, int(P), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_naive_scores")
    return scores


def attn_naive_softmax(scores, C: int, P: int, stream=None):
    """Step 2: every row of the score matrix replaced by its softmax, in place."""
    ws = _naive_scores_arg(scores, C, P)
    rc = load().attn_naive_softmax(ws, int(C), int(P), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_naive_softmax")
    return scores


def attn_naive_weighted_sum(scores, vCache, out, P: int, stream=None):
    """Step 3: out[i][h][:] = sum_j scores[h][i][j] v[j][h/4][:]."""
    C = out.shape[0]
    ws = _naive_scores_arg(scores, C, P)
    rc = load().attn_naive_weighted_sum(ws, _ptr(vCache), _ptr(out), C, int(P), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_naive_weighted_sum")
    return out


def attn_prefill_ffma(q, kCache, vCache, out, P: int, stream=None):
    """The same operation on the FP32 CUDA cores."""
    return _call("attn_prefill_ffma", q, kCache, vCache, out, P, stream)


def attn_reference_prefill(q, kCache, vCache, out, P: int, stream=None):
    """The starter-design in-run reference (slow by design)."""
    return _call("attn_reference_prefill", q, kCache, vCache, out, P, stream)


def attn_selftest_timeout(q, kCache, vCache, out, P: int, stream=None):
    """Run the tensor-core kernel with a load withheld so a bounded wait expires
    (a failure-path test); read the outcome with attn_get_device_error()."""
    return _call("attn_selftest_timeout", q, kCache, vCache, out, P, stream)


def attn_tensor_peak(bf16: bool, n: int, iters: int, ctas: int, stream=None) -> float:
    """Launch the tensor-pipe rate measurement (one CTA per SM for ctas <= SMs:
    ``iters`` dense M = 128, N = n MMAs each, kind::tf32 or, with bf16,
    kind::f16); returns the flops one launch performs."""
    rc = load().attn_tensor_peak(int(bool(bf16)), int(n), int(iters), int(ctas), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_tensor_peak")
    return float(ctas) * iters * 2 * 128 * n * (16 if bf16 else 8)


def attn_get_device_error() -> int:
    """Synchronise the device; return and clear the device error word."""
    return int(load().attn_get_device_error())


def raw(name: str):
    """The raw ctypes function ``name`` (pointers and ints in, code out)."""
    return getattr(load(), name)
