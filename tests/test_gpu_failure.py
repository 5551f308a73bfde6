"""Failure detection on the GPU without a GPU fault: a bounded wait is made to
expire on purpose (a K tile that is never loaded), the kernel records
ATTN_ETIMEOUT in the device error word and winds down, and the context stays
usable for the next call."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import run_entry  # noqa: E402


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


def test_expired_wait_is_reported_and_context_survives(cp):
    assert cp.attn_get_device_error() == 0
    inp = W.edge(64, 1000)
    q = torch.from_numpy(inp.q).cuda()
    k = torch.from_numpy(inp.k).cuda()
    v = torch.from_numpy(inp.v).cuda()
    out = torch.empty_like(q)
    cp.attn_selftest_timeout(q, k, v, out, inp.P)
    assert cp.attn_get_device_error() == cp.ATTN_ETIMEOUT
    assert cp.attn_get_device_error() == 0          # read-and-clear
    # the next call on the same context is correct
    got, guards = run_entry(cp.attn_prefill, inp)
    assert guards
    rep = oracle.check(got, oracle.prefill(inp))
    assert rep["n_bad"] == 0, rep
    assert cp.attn_get_device_error() == 0


def test_selftest_rejects_empty_chunk(cp):
    f = cp.raw("attn_selftest_timeout")
    assert f(None, None, None, None, 0, 0, None) == cp.ATTN_EINVAL


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_expired_wait_is_reported_and_context_survives(cp, splits):
    """The decode kernel's bounded wait: every block's first tile is withheld,
    each block records ATTN_ETIMEOUT and returns; the next decode is correct."""
    assert cp.attn_get_device_error() == 0
    batch = W.decode_batch([300, 1000], seed=21)
    q = torch.from_numpy(batch.q).cuda()
    kp = torch.from_numpy(batch.k_pages).cuda()
    vp = torch.from_numpy(batch.v_pages).cuda()
    tb = torch.from_numpy(batch.table).cuda()
    cl = torch.from_numpy(batch.ctx).cuda()
    out = torch.empty_like(q)
    nbytes = cp.attn_decode_workspace_bytes(2, batch.max_context, splits)
    ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device="cuda")
    cp.attn_selftest_decode_timeout(q, kp, vp, tb, cl, out, batch.max_context, splits, ws)
    assert cp.attn_get_device_error() == cp.ATTN_ETIMEOUT
    assert cp.attn_get_device_error() == 0
    cp.attn_decode_paged(q, kp, vp, tb, cl, out, batch.max_context, splits, ws)
    got = out.cpu().numpy()
    assert cp.attn_get_device_error() == 0
    for b, T in enumerate(batch.ctx.tolist()):
        k = oracle.gather_pages(batch.k_pages, batch.table[b], T)
        v = oracle.gather_pages(batch.v_pages, batch.table[b], T)
        rep = oracle.check(got[b], oracle.attention(batch.q[b:b + 1], k, v, T - 1)[0])
        assert rep["n_bad"] == 0, rep


def test_decode_selftest_rejects_empty_batch(cp):
    f = cp.raw("attn_selftest_decode_timeout")
    assert f(None, None, None, None, None, None, 0, 1, 1, 16, 0, None, 0, None) == cp.ATTN_EINVAL


def test_decode_expired_wait_leaves_no_stale_partial(cp):
    """A block whose wait expires writes its segment record empty (m = -inf,
    l = 0): a workspace still holding a finished call's finite records must
    not leak them into the merge. Every block of the self-test fails, so every
    record is empty and the merged output is exactly zero."""
    assert cp.attn_get_device_error() == 0
    batch = W.decode_batch([300, 1000], seed=22)
    q = torch.from_numpy(batch.q).cuda()
    kp = torch.from_numpy(batch.k_pages).cuda()
    vp = torch.from_numpy(batch.v_pages).cuda()
    tb = torch.from_numpy(batch.table).cuda()
    cl = torch.from_numpy(batch.ctx).cuda()
    out = torch.empty_like(q)
    splits = 3
    nbytes = cp.attn_decode_workspace_bytes(2, batch.max_context, splits)
    ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device="cuda")
    cp.attn_decode_paged(q, kp, vp, tb, cl, out, batch.max_context, splits, ws)  # finite records
    assert cp.attn_get_device_error() == 0
    assert torch.isfinite(out).all() and out.abs().max().item() > 0
    out.fill_(float("nan"))
    cp.attn_selftest_decode_timeout(q, kp, vp, tb, cl, out, batch.max_context, splits, ws)
    assert cp.attn_get_device_error() == cp.ATTN_ETIMEOUT
    assert torch.equal(out, torch.zeros_like(out))
