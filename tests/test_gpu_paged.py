"""attn_prefill_paged against the oracle on shuffled, NaN-padded page pools
("FlashAttention and inference kernels", PagedAttention: token t in slot t % 16
of physical page blockTable[t / 16])."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import full_refs  # noqa: E402
from gpu_util import GuardedOut  # noqa: E402


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


def run_paged(cp, inp, pg, table=None):
    q = torch.from_numpy(inp.q).cuda()
    kp = torch.from_numpy(pg.k_pages).cuda()
    vp = torch.from_numpy(pg.v_pages).cuda()
    tb = torch.from_numpy(pg.table if table is None else table).cuda()
    g = GuardedOut(inp.C)
    cp.attn_prefill_paged(q, kp, vp, tb, g.out, inp.P)
    torch.cuda.synchronize()
    return g.numpy(), g.guards_intact()


def check(got, ref, what):
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{what}: {rep}"


@pytest.mark.parametrize("C,P", [(1, 0), (17, 31), (33, 0), (64, 1000), (100, 77), (257, 0)])
def test_paged_matches_oracle(cp, C, P):
    inp = W.edge(C, P)
    pg = W.to_pages(inp, seed=C * 7 + P)
    got, guards = run_paged(cp, inp, pg)
    assert guards
    ref = oracle.prefill_paged(inp.q, pg.k_pages, pg.v_pages, pg.table, P)
    check(got, ref, f"paged C={C} P={P}")
    # and the same numbers as the contiguous cache
    check(got, oracle.prefill(inp), f"paged vs contiguous C={C} P={P}")


def test_paged_planted_and_lastkey(cp):
    for inp in (W.tiny(), W.edge(33, 1000, variant="lastkey"), W.edge(17, 31, variant="ramp")):
        pg = W.to_pages(inp, seed=11)
        got, _ = run_paged(cp, inp, pg)
        assert np.isfinite(got).all()
        check(got, oracle.prefill(inp), inp.name)


def test_paged_serving_chunk_full(cp):
    """Every element of the serving chunk on a shuffled, NaN-padded pool."""
    inp, ref = full_refs.serve()
    pg = W.to_pages(inp, seed=5, spare_pages=37)
    got, guards = run_paged(cp, inp, pg)
    assert guards
    check(got, ref, "paged serve")


def test_paged_long_prefix_full(cp):
    """Every element of the long prefix (C = 2048, P = 30720) on a shuffled,
    NaN-padded pool of 2,176 pages."""
    inp, ref = full_refs.long_prefix()
    pg = W.to_pages(inp, seed=6, spare_pages=11)
    got, guards = run_paged(cp, inp, pg)
    assert guards
    check(got, ref, "paged long prefix")


def test_shared_prefix_pages(cp):
    """Two logical pages may map to one physical page (prefix sharing): the
    oracle gathers through the same table."""
    inp = W.edge(20, 44)
    pg = W.to_pages(inp, seed=9)
    table = pg.table.copy()
    table[2] = table[0]           # tokens 32..47 now read the page of tokens 0..15
    got, _ = run_paged(cp, inp, pg, table)
    check(got, oracle.prefill_paged(inp.q, pg.k_pages, pg.v_pages, table, inp.P), "shared page")


def test_table_entry_out_of_range_is_reported(cp):
    inp = W.edge(17, 31)
    pg = W.to_pages(inp, seed=1)
    table = pg.table.copy()
    table[1] = pg.k_pages.shape[0] + 3
    assert cp.attn_get_device_error() == 0
    run_paged(cp, inp, pg, table)
    assert cp.attn_get_device_error() == cp.ATTN_EBOUNDS
    assert cp.attn_get_device_error() == 0
    got, _ = run_paged(cp, inp, pg)          # the context is still good
    check(got, oracle.prefill(inp), "after a bounds error")


def test_paged_argument_errors(cp):
    f = cp.raw("attn_prefill_paged")
    inp = W.edge(4, 3)
    q = torch.from_numpy(inp.q).cuda()
    pages = torch.zeros(2, 16, 8, 64, device="cuda")
    out = torch.empty_like(q)
    tb = torch.zeros(2, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert f(q.data_ptr(), pages.data_ptr(), pages.data_ptr(), None, out.data_ptr(), 4, 3, 2, s) == cp.ATTN_EINVAL
    assert f(q.data_ptr(), pages.data_ptr(), pages.data_ptr(), tb.data_ptr(), out.data_ptr(), 4, 3, 0, s) == cp.ATTN_EINVAL
    assert f(q.data_ptr(), pages.data_ptr(), pages.data_ptr(), tb.data_ptr() + 2, out.data_ptr(), 4, 3, 2, s) == cp.ATTN_EALIGN
    assert f(None, None, None, None, None, 0, 3, 0, s) == cp.ATTN_OK
