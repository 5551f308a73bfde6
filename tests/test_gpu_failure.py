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
