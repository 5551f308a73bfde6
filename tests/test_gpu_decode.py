"""attn_decode_paged (one query per sequence and head, split-KV + merge) against
the oracle: each sequence's answer is the exact attention of its query over its
gathered cache, i.e. the oracle with C = 1 and P = ctx - 1."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


def reference(batch):
    out = np.zeros(batch.q.shape, dtype=np.float64)
    for b, T in enumerate(batch.ctx.tolist()):
        if T == 0:
            continue
        k = oracle.gather_pages(batch.k_pages, batch.table[b], T)
        v = oracle.gather_pages(batch.v_pages, batch.table[b], T)
        out[b] = oracle.attention(batch.q[b:b + 1], k, v, T - 1)[0]
    return out


def run_decode(cp, batch, num_splits=0, max_context=None):
    mc = batch.max_context if max_context is None else max_context
    q = torch.from_numpy(batch.q).cuda()
    kp = torch.from_numpy(batch.k_pages).cuda()
    vp = torch.from_numpy(batch.v_pages).cuda()
    tb = torch.from_numpy(batch.table).cuda()
    cl = torch.from_numpy(batch.ctx).cuda()
    out = torch.empty_like(q)
    out.view(torch.int32).fill_(-1)
    nbytes = cp.attn_decode_workspace_bytes(q.shape[0], mc, num_splits)
    ws = torch.empty(max(nbytes, 16) // 4 + 4, dtype=torch.float32, device="cuda") if nbytes else None
    cp.attn_decode_paged(q, kp, vp, tb, cl, out, mc, num_splits, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), nbytes


def check(got, ref, what):
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{what}: {rep}"


@pytest.mark.parametrize("splits", [0, 1, 3, 7])
def test_page_context_lengths(cp, splits):
    """The teaching program's context lengths 1, 17, 1000 and 4096."""
    batch = W.decode_batch([1, 17, 1000, 4096], seed=2)
    got, _ = run_decode(cp, batch, splits)
    check(got, reference(batch), f"splits={splits}")


def test_single_key_returns_its_value(cp):
    batch = W.decode_batch([1, 1], seed=3)
    got, _ = run_decode(cp, batch, 0)
    for b in range(2):
        v0 = batch.v_pages[batch.table[b, 0], 0]
        np.testing.assert_allclose(got[b], np.repeat(v0, 4, axis=0), rtol=1e-6, atol=1e-7)


def test_planted_scores_stay_finite(cp):
    batch = W.decode_batch([40, 700, 2048], seed=4, planted=(0, 5, 39, 650))
    got, _ = run_decode(cp, batch, 0)
    assert np.isfinite(got).all()
    check(got, reference(batch), "planted")


def test_many_sequences_mixed_lengths(cp):
    lens = [int(x) for x in (W.splitmix64(9, 48) % np.uint64(3000)).tolist()]
    lens[0], lens[1] = 0, 16
    batch = W.decode_batch(lens, seed=5)
    got, nbytes = run_decode(cp, batch, 0)
    check(got, reference(batch), "mixed lengths")
    assert np.all(got[0] == 0.0)   # an empty context gives zeros


@pytest.mark.parametrize("splits", [2, 16])
def test_workspace_starts_as_garbage_and_is_reused(cp, splits):
    """Nothing in the workspace needs to start at zero: it is filled with 0xFF
    bytes (every m_s, l_s and O_s reads NaN), then three calls in a row on one
    stream reuse it unchanged. Their short second sequences leave most of 16
    segments empty, whose records carry l_s = 0 and a stale O_s that the merge
    must skip."""
    mc = 3000
    nbytes = cp.attn_decode_workspace_bytes(2, mc, splits)
    assert nbytes > 0
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device="cuda")
    ws.view(torch.int32).fill_(-1)
    calls = []
    for i, lens in enumerate(([3000, 5], [3000, 1], [3000, 2048])):
        batch = W.decode_batch(lens, seed=30 + i)
        t = [torch.from_numpy(x).cuda() for x in (batch.q, batch.k_pages, batch.v_pages, batch.table, batch.ctx)]
        out = torch.full_like(t[0], float("nan"))
        cp.attn_decode_paged(t[0], t[1], t[2], t[3], t[4], out, mc, splits, ws)
        calls.append((batch, out, t))
    torch.cuda.synchronize()
    for batch, out, _ in calls:
        check(out.cpu().numpy(), reference(batch), f"splits={splits} ctx={batch.ctx.tolist()}")
    assert cp.attn_get_device_error() == 0


def test_long_context_split(cp):
    batch = W.decode_batch([32768, 5000], seed=6)
    got, nbytes = run_decode(cp, batch, 0)
    assert nbytes > 0
    check(got, reference(batch), "long")


def test_workspace_and_bounds_errors(cp):
    batch = W.decode_batch([1000, 300], seed=7)
    q = torch.from_numpy(batch.q).cuda()
    kp = torch.from_numpy(batch.k_pages).cuda()
    vp = torch.from_numpy(batch.v_pages).cuda()
    tb = torch.from_numpy(batch.table).cuda()
    cl = torch.from_numpy(batch.ctx).cuda()
    out = torch.empty_like(q)
    need = cp.attn_decode_workspace_bytes(2, 1000, 4)
    assert need > 0
    small = torch.empty(need // 4 - 4, dtype=torch.float32, device="cuda")
    with pytest.raises(cp.AttnError) as e:
        cp.attn_decode_paged(q, kp, vp, tb, cl, out, 1000, 4, small)
    assert e.value.code == cp.ATTN_ESPACE
    with pytest.raises(cp.AttnError) as e:
        cp.attn_decode_paged(q, kp, vp, tb, cl, out, 1000, 4, None)
    assert e.value.code == cp.ATTN_ESPACE
    # a context length above max_context is recorded and clamped
    assert cp.attn_get_device_error() == 0
    ws = torch.empty(need // 4 + 4, dtype=torch.float32, device="cuda")
    cp.attn_decode_paged(q, kp, vp, tb, cl, out, 500, 4, ws[: cp.attn_decode_workspace_bytes(2, 500, 4) // 4 + 4])
    assert cp.attn_get_device_error() == cp.ATTN_EBOUNDS
    assert cp.attn_get_device_error() == 0


@pytest.mark.parametrize("splits", [0, 1, 3])
def test_table_entry_out_of_range_reads_zeros(cp, splits):
    """A block-table entry outside [0, numPages) is recorded as ATTN_EBOUNDS and
    its 16 tokens read as zero keys and values (scores 0, no value), as the
    header states; the next call on the same context is correct again."""
    batch = W.decode_batch([40, 300], seed=12)
    n_pages = batch.k_pages.shape[0]
    table = batch.table.copy()
    table[0, 1] = n_pages + 5   # tokens 16..31 of sequence 0
    table[1, 7] = -7            # tokens 112..127 of sequence 1
    want = np.zeros(batch.q.shape, dtype=np.float64)
    for b, T in enumerate(batch.ctx.tolist()):
        k = np.zeros((T, W.HKV, W.D), dtype=np.float32)
        v = np.zeros((T, W.HKV, W.D), dtype=np.float32)
        for t in range(T):
            page = table[b, t // W.PAGE]
            if 0 <= page < n_pages:
                k[t] = batch.k_pages[page, t % W.PAGE]
                v[t] = batch.v_pages[page, t % W.PAGE]
        want[b] = oracle.attention(batch.q[b:b + 1], k, v, T - 1)[0]
    bad = W.DecodeBatch(q=batch.q, k_pages=batch.k_pages, v_pages=batch.v_pages, table=table, ctx=batch.ctx)
    assert cp.attn_get_device_error() == 0
    got, _ = run_decode(cp, bad, splits)
    assert cp.attn_get_device_error() == cp.ATTN_EBOUNDS
    assert cp.attn_get_device_error() == 0
    check(got, want, f"bad table entries, splits={splits}")
    got, _ = run_decode(cp, batch, splits)
    assert cp.attn_get_device_error() == 0
    check(got, reference(batch), "after a bounds error")
