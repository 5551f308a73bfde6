"""attn_decode_paged_noalloc, called through the C ABI, against attn_decode_paged
on the same inputs: the partials live in the library's fixed device scratch
instead of a caller workspace, and the results must agree within the
attention-v1 tolerance. Collected last, so it runs both alone in a fresh
process and after every other test has used the library."""
import ctypes

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


def to_device(batch):
    d = dict(q=torch.from_numpy(batch.q).cuda(), kp=torch.from_numpy(batch.k_pages).cuda(),
             vp=torch.from_numpy(batch.v_pages).cuda(), tb=torch.from_numpy(batch.table).cuda(),
             cl=torch.from_numpy(batch.ctx).cuda())
    d["B"], d["max_blocks"] = batch.table.shape
    d["num_pages"] = batch.k_pages.shape[0]
    return d


def poisoned_out(d):
    out = torch.empty_like(d["q"])
    out.view(torch.int32).fill_(-1)   # NaN bits: an unwritten element fails the check
    return out


def with_workspace(cp, d, max_context, splits):
    out = poisoned_out(d)
    nbytes = cp.attn_decode_workspace_bytes(d["B"], max_context, splits)
    ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device="cuda") if nbytes else None
    cp.attn_decode_paged(d["q"], d["kp"], d["vp"], d["tb"], d["cl"], out, max_context, splits, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), nbytes


def no_alloc(cp, d, max_context, splits):
    """The raw C-ABI call: plain device pointers and sizes, no workspace."""
    f = cp.raw("attn_decode_paged_noalloc")
    out = poisoned_out(d)
    rc = f(d["q"].data_ptr(), d["kp"].data_ptr(), d["vp"].data_ptr(), d["tb"].data_ptr(), d["cl"].data_ptr(),
           out.data_ptr(), d["B"], d["max_blocks"], d["num_pages"], max_context, splits,
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == cp.ATTN_OK, cp.strerror(rc)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check(got, ref, what):
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{what}: {rep}"


def test_two_calls_in_a_row_match_the_workspace_entry_point(cp):
    """Two different batches back to back through the shared scratch: the
    second call must not see anything the first left behind."""
    first = W.decode_batch([1, 17, 1000, 4096], seed=21)
    lens = [int(x) for x in (W.splitmix64(23, 12) % np.uint64(2500)).tolist()]
    lens[3] = 0
    second = W.decode_batch(lens, seed=22)
    for batch, splits in ((first, 0), (second, 5)):
        d = to_device(batch)
        want, nbytes = with_workspace(cp, d, batch.max_context, splits)
        assert nbytes > 0   # these cases do use the scratch
        got = no_alloc(cp, d, batch.max_context, splits)
        check(got, want, f"no-alloc vs workspace, B={d['B']} splits={splits}")
    assert cp.attn_get_device_error() == 0


def test_same_call_twice_and_against_the_oracle(cp):
    batch = W.decode_batch([700, 3000, 64], seed=24)
    d = to_device(batch)
    want, _ = with_workspace(cp, d, batch.max_context, 0)
    a = no_alloc(cp, d, batch.max_context, 0)
    b = no_alloc(cp, d, batch.max_context, 0)
    check(a, want, "first call")
    check(b, want, "second call")
    for i, T in enumerate(batch.ctx.tolist()):
        k = oracle.gather_pages(batch.k_pages, batch.table[i], T)
        v = oracle.gather_pages(batch.v_pages, batch.table[i], T)
        check(b[i], oracle.attention(batch.q[i:i + 1], k, v, T - 1)[0], f"oracle, sequence {i}")


def test_partials_beyond_the_scratch_are_rejected(cp):
    """64 sequences x 16 segments need 64 * 8 * 16 records of 1056 bytes, more
    than the 4 MiB scratch: refused on the host, nothing enqueued."""
    batch = W.decode_batch([1024] * 64, seed=25, spare_pages=0)
    d = to_device(batch)
    assert cp.attn_decode_workspace_bytes(64, 1024, 16) > cp.DECODE_SCRATCH_BYTES
    out = poisoned_out(d)
    f = cp.raw("attn_decode_paged_noalloc")
    rc = f(d["q"].data_ptr(), d["kp"].data_ptr(), d["vp"].data_ptr(), d["tb"].data_ptr(), d["cl"].data_ptr(),
           out.data_ptr(), 64, d["max_blocks"], d["num_pages"], 1024, 16, None)
    assert rc == cp.ATTN_ESCRATCH
    assert "scratch" in cp.strerror(rc)
    torch.cuda.synchronize()
    assert (out.view(torch.int32) == -1).all()
    # the automatic split count fits
    got = no_alloc(cp, d, 1024, 0)
    want, _ = with_workspace(cp, d, 1024, 0)
    check(got, want, "automatic splits, B=64")


def test_automatic_split_count_fits_the_scratch(cp):
    """With numSplits = 0 the partials of any batch fit the fixed scratch on
    this device, so an automatic call never returns ATTN_ESCRATCH: a sweep of B
    and maxContext through attn_decode_workspace_bytes (no launch)."""
    worst = (0, 0, 0)
    for ctx in (256, 512, 1000, 2048, 4096, 16384, 1 << 20, 1 << 24):
        for B in list(range(1, 2049)) + list(range(2049, 65536, 211)):
            nbytes = cp.attn_decode_workspace_bytes(B, ctx, 0)
            if nbytes > worst[0]:
                worst = (nbytes, B, ctx)
    assert 0 < worst[0] <= cp.DECODE_SCRATCH_BYTES, worst
