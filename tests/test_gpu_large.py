"""Large sizes: a 262,144-token cached prefix (1 GiB of fp32 K/V, far past L2;
row indices past 2^18 in the TMA coordinates and 64-bit offsets in every index
computation) for each prefill path, and a 131,072-token decode context, checked
on sampled rows against the oracle."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import GuardedOut, device_inputs, sample_rows  # noqa: E402

P_LONG = 1 << 18
C_LONG = 256


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


@pytest.fixture(scope="module")
def very_long():
    return W.make_inputs(C_LONG, P_LONG, seed=77, dist="normal", name=f"very long C={C_LONG} P={P_LONG}")


def check(got, ref, what):
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{what}: {rep}"


@pytest.mark.parametrize("path", ["attn_prefill", "attn_prefill_bf16x3"])
def test_very_long_prefix_fp32_cache(cp, very_long, path):
    inp = very_long
    q, k, v = device_inputs(inp)
    g = GuardedOut(inp.C)
    getattr(cp, path)(q, k, v, g.out, inp.P)
    torch.cuda.synchronize()
    got = g.numpy()
    assert g.guards_intact() and np.isfinite(got).all()
    rows = sample_rows(inp.C, n_random=4, seed=7)
    check(got[rows], oracle.prefill(inp, rows=rows), f"{path} P={inp.P}")


def test_very_long_prefix_bf16_cache(cp, very_long):
    inp = very_long
    kv = W.to_bf16(inp)
    q = torch.from_numpy(inp.q).cuda()
    k = torch.from_numpy(kv.k.view(np.int16)).cuda().view(torch.bfloat16)
    v = torch.from_numpy(kv.v.view(np.int16)).cuda().view(torch.bfloat16)
    g = GuardedOut(inp.C)
    cp.attn_prefill_bf16kv(q, k, v, g.out, inp.P)
    torch.cuda.synchronize()
    got = g.numpy()
    assert g.guards_intact() and np.isfinite(got).all()
    rows = sample_rows(inp.C, n_random=4, seed=8)
    check(got[rows], oracle.prefill_bf16kv(inp.q, kv.k, kv.v, inp.P, rows=rows), f"bf16kv P={inp.P}")


def test_long_decode_context(cp):
    batch = W.decode_batch([131072, 5, 70000], seed=31, spare_pages=2)
    q = torch.from_numpy(batch.q).cuda()
    kp = torch.from_numpy(batch.k_pages).cuda()
    vp = torch.from_numpy(batch.v_pages).cuda()
    tb = torch.from_numpy(batch.table).cuda()
    cl = torch.from_numpy(batch.ctx).cuda()
    out = torch.empty_like(q)
    nbytes = cp.attn_decode_workspace_bytes(3, batch.max_context)
    ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device="cuda")
    cp.attn_decode_paged(q, kp, vp, tb, cl, out, batch.max_context, 0, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b, T in enumerate(batch.ctx.tolist()):
        k = oracle.gather_pages(batch.k_pages, batch.table[b], T)
        v = oracle.gather_pages(batch.v_pages, batch.table[b], T)
        check(got[b], oracle.attention(batch.q[b:b + 1], k, v, T - 1)[0], f"decode ctx={T}")
    assert cp.attn_get_device_error() == 0
