"""The host-buffer entry points (attn_prefill_host and its bf16x3 and bf16-cache
twins): the chunk runs as up to four sub-chunks of whole query tiles with the
copies overlapped; each sub-chunk is one full round of units (19 query tiles
on 152 SMs). Each case is checked against the oracle, and against the
device-pointer entry point: bit for bit where the whole call and its sub-chunks
take the same units in the same order, to a tight tolerance where one of them
splits units over CTA pairs and the other does not (the serving chunk, whose
sub-chunks are then each checked bit for bit against a device call of their
own). Rows before and after out_host must stay untouched,
pageable memory must work, and back-to-back calls that reuse the same device
buffers must not race."""
import threading

import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import sample_rows  # noqa: E402

PATHS = {  # host entry -> (device entry, bf16 cache)
    "attn_prefill_host": ("attn_prefill", False),
    "attn_prefill_bf16x3_host": ("attn_prefill_bf16x3", False),
    "attn_prefill_bf16kv_host": ("attn_prefill_bf16kv", True),
}
NAN_BITS = -1  # 0xFFFFFFFF


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


def host_tensors(inp, bf16, pinned=True):
    q = torch.from_numpy(inp.q)
    if bf16:
        kv = W.to_bf16(inp)
        k, v = torch.from_numpy(kv.k.view(np.int16)), torch.from_numpy(kv.v.view(np.int16))
    else:
        kv = None
        k, v = torch.from_numpy(inp.k), torch.from_numpy(inp.v)
    # out_host sits between two poisoned guard rows of the same buffer.
    big = torch.empty(inp.C + 2, 32, 64, dtype=torch.float32)
    if pinned:
        q, k, v, big = q.pin_memory(), k.pin_memory(), v.pin_memory(), big.pin_memory()
    big.view(torch.int32).fill_(NAN_BITS)
    return q, k, v, big, kv


def device_tensors(inp, bf16):
    q = torch.empty(inp.C, 32, 64, device="cuda")
    kvt = torch.int16 if bf16 else torch.float32
    k = torch.full((inp.P + inp.C, 8, 64), -1, dtype=kvt, device="cuda")
    v = torch.full((inp.P + inp.C, 8, 64), -1, dtype=kvt, device="cuda")
    out = torch.full_like(q, float("nan"))
    return q, k, v, out


def expected(inp, kv, rows=None):
    if kv is None:
        return oracle.prefill(inp, rows=rows)
    return oracle.prefill_bf16kv(inp.q, kv.k, kv.v, inp.P, rows=rows)


def run_host(cp, name, inp, pinned=True, stream=None):
    bf16 = PATHS[name][1]
    hq, hk, hv, big, kv = host_tensors(inp, bf16, pinned)
    dq, dk, dv, dout = device_tensors(inp, bf16)
    getattr(cp, name)(hq, hk, hv, big[1:1 + inp.C], dq, dk, dv, dout, inp.P, stream)
    (stream or torch.cuda.current_stream()).synchronize()
    guards = bool((big[0].view(torch.int32) == NAN_BITS).all() and (big[-1].view(torch.int32) == NAN_BITS).all())
    return big[1:1 + inp.C].numpy().copy(), guards, (dq, dk, dv, dout), kv


def run_device(cp, name, inp, kv):
    dev_name, bf16 = PATHS[name]
    q = torch.from_numpy(inp.q).cuda()
    if bf16:
        k = torch.from_numpy(kv.k.view(np.int16)).cuda()
        v = torch.from_numpy(kv.v.view(np.int16)).cuda()
    else:
        k, v = torch.from_numpy(inp.k).cuda(), torch.from_numpy(inp.v).cuda()
    out = torch.full_like(q, float("nan"))
    getattr(cp, dev_name)(q, k, v, out, inp.P)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check(got, ref, what):
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{what}: {rep}"


# (C, P) spanning one sub-chunk (C <= 608), two (1057 = 19 + 15 tiles, the
# second one ragged), and four (2118 rows: 67 tiles as 19, 19, 19, 10).
@pytest.mark.parametrize("name", list(PATHS))
@pytest.mark.parametrize("C,P", [(1, 0), (17, 31), (100, 77), (1057, 300), (2118, 5)])
def test_matches_oracle_and_the_device_entry(cp, name, C, P):
    inp = W.edge(C, P, seed=C + 7 * P)
    got, guards, dev, kv = run_host(cp, name, inp)
    assert guards, "a row outside out_host was written"
    assert np.isfinite(got).all()
    rows = sample_rows(C, extra=(511, 512, 543, 544, 1055, 1056, 1599, 1600), n_random=8, seed=C)
    check(got[rows], expected(inp, kv, rows=rows), f"{name} C={C} P={P}")
    assert np.array_equal(got, run_device(cp, name, inp, kv)), "differs from the device-pointer entry point"
    # The device buffers hold the inputs and the result after the call.
    dq, dk, dv, dout = dev
    assert np.array_equal(dq.cpu().numpy(), inp.q)
    assert np.array_equal(dout.cpu().numpy(), got)
    want_k = kv.k.view(np.int16) if kv is not None else inp.k
    assert np.array_equal(dk.cpu().numpy(), want_k)


def test_serving_chunk_sub_chunks(cp):
    """Sub-chunks of 608, 608, 608 and 224 rows. Each one's rows are exactly
    the device call on that sub-chunk (the last one's 56 units split over CTA
    pairs); the device call on the whole chunk splits its last round's units
    instead (another summation order), so against it the comparison is to a
    tolerance far inside the oracle's."""
    inp = W.serve()
    got, guards, _, kv = run_host(cp, "attn_prefill_host", inp)
    assert guards and np.isfinite(got).all()
    np.testing.assert_allclose(got, run_device(cp, "attn_prefill_host", inp, kv), rtol=1e-5, atol=1e-6)
    for r0, r1 in ((0, 608), (608, 1216), (1824, 2048)):
        sub = W.Inputs(q=inp.q[r0:r1], k=inp.k[:inp.P + r1], v=inp.v[:inp.P + r1],
                       C=r1 - r0, P=inp.P + r0, name=f"rows {r0}..{r1 - 1}")
        assert np.array_equal(got[r0:r1], run_device(cp, "attn_prefill_host", sub, None)), r0
    rows = sample_rows(inp.C, extra=(607, 608, 1215, 1216, 1823, 1824), n_random=6, seed=11)
    check(got[rows], expected(inp, kv, rows=rows), "serve via host buffers")


def test_pageable_host_memory(cp):
    inp = W.edge(1100, 64, seed=5)
    got, guards, _, kv = run_host(cp, "attn_prefill_host", inp, pinned=False)
    assert guards
    assert np.array_equal(got, run_device(cp, "attn_prefill_host", inp, kv))


def test_back_to_back_calls_reusing_device_buffers(cp):
    """Three calls on one side stream with one set of device buffers and
    different inputs, synchronised once at the end: each call's copies wait
    for the previous call's compute and copy-out."""
    a, b, c = (W.edge(1200, 900, seed=s) for s in (1, 2, 3))
    s = torch.cuda.Stream()
    dq, dk, dv, dout = device_tensors(a, False)
    outs = []
    for inp in (a, b, c):
        hq, hk, hv = (torch.from_numpy(x).pin_memory() for x in (inp.q, inp.k, inp.v))
        ho = torch.full((inp.C, 32, 64), float("nan")).pin_memory()
        cp.attn_prefill_host(hq, hk, hv, ho, dq, dk, dv, dout, inp.P, s)
        outs.append((inp, ho, (hq, hk, hv)))
    s.synchronize()
    for inp, ho, _ in outs:
        assert np.array_equal(ho.numpy(), run_device(cp, "attn_prefill_host", inp, None))


def test_concurrent_host_threads(cp):
    """Four host threads, each with its own stream and buffers, enqueue at the
    same time (the library's streams and events are shared and locked)."""
    inps = [W.edge(600 + 100 * i, 50 * i, seed=40 + i) for i in range(4)]
    results, errors = {}, []
    barrier = threading.Barrier(len(inps))

    def run(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            inp = inps[i]
            hq, hk, hv, big, _ = host_tensors(inp, False)
            dq, dk, dv, dout = device_tensors(inp, False)
            barrier.wait()
            cp.attn_prefill_host(hq, hk, hv, big[1:1 + inp.C], dq, dk, dv, dout, inp.P, s)
            s.synchronize()
            results[i] = big[1:1 + inp.C].numpy().copy()
        except Exception as e:  # reported below
            errors.append(repr(e))

    ts = [threading.Thread(target=run, args=(i,)) for i in range(len(inps))]
    [t.start() for t in ts]
    [t.join() for t in ts]
    assert not errors, errors
    for i, inp in enumerate(inps):
        # 700 and 800 rows: the whole call splits its tail, the sub-chunks do not.
        np.testing.assert_allclose(results[i], run_device(cp, "attn_prefill_host", inp, None), rtol=1e-5, atol=1e-6)
        rep = oracle.check(results[i], oracle.prefill(inp))
        assert rep["n_bad"] == 0, (i, rep)
    assert cp.attn_get_device_error() == 0


def test_errors(cp):
    inp = W.edge(40, 8)
    hq, hk, hv, big, _ = host_tensors(inp, False)
    dq, dk, dv, dout = device_tensors(inp, False)
    f = cp.raw("attn_prefill_host")
    s = torch.cuda.current_stream().cuda_stream
    hp = [t.data_ptr() for t in (hq, hk, hv, big[1:1 + inp.C])]
    dp = [t.data_ptr() for t in (dq, dk, dv, dout)]
    assert f(*hp, dp[0], dp[1] + 4, dp[2], dp[3], inp.C, inp.P, s) == cp.ATTN_EALIGN
    assert f(hp[0], None, hp[2], hp[3], *dp, inp.C, inp.P, s) == cp.ATTN_EINVAL
    assert f(*hp, *dp, 0, inp.P, s) == cp.ATTN_OK
    torch.cuda.synchronize()
    assert (big.view(torch.int32) == NAN_BITS).all(), "an empty or rejected call wrote out_host"
