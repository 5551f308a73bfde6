"""The split-unit grids against the oracle, every element checked on a poisoned,
guarded output: chunks small enough that every unit is split (the longest unit
of 256 keys or more, 1024 for the bf16 kernels) over a cluster of twelve CTAs
(chunks of up to 32 rows against 8192 keys or more) or eight (against 1024
keys or more, 2048 for the bf16 kernels), of four or of three (at most as many units as the device holds such
clusters at once: chunks of up to 128 and 184 rows on 152 SMs) or over a CTA
pair (up to 304 rows), and chunks
whose last round of units goes to the pair grid (the tail), including a ragged
last query tile and a paged cache."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import GuardedOut  # noqa: E402


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


def run(cp, path, inp):
    g = GuardedOut(inp.C)
    q = torch.from_numpy(inp.q).cuda()
    if path == "attn_prefill_bf16kv":
        kv = W.to_bf16(inp)
        k = torch.from_numpy(kv.k.view(np.int16)).cuda()
        v = torch.from_numpy(kv.v.view(np.int16)).cuda()
        ref = oracle.prefill_bf16kv(inp.q, kv.k, kv.v, inp.P)
    else:
        k, v = torch.from_numpy(inp.k).cuda(), torch.from_numpy(inp.v).cuda()
        ref = oracle.prefill(inp)
    if path == "attn_prefill_paged":
        pg = W.to_pages(inp, seed=inp.C)
        cp.attn_prefill_paged(q, torch.from_numpy(pg.k_pages).cuda(), torch.from_numpy(pg.v_pages).cuda(),
                              torch.from_numpy(pg.table).cuda(), g.out, inp.P)
    else:
        getattr(cp, path)(q, k, v, g.out, inp.P)
    torch.cuda.synchronize()
    got = g.numpy()
    assert g.guards_intact(), "a value outside out was written"
    assert np.isfinite(got).all()
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{path} C={inp.C} P={inp.P}: {rep}"
    assert cp.attn_get_device_error() == 0


# Every unit split (at most 76 units, i.e. C <= 304 rows, on 152 SMs): over
# clusters of eight up to 32 rows, of four up to 128 rows, of three up to 184
# rows (on a GB300), over pairs beyond; and 77-92 units over threes in two
# waves when the units are long.
@pytest.mark.parametrize("path,C,P", [
    ("attn_prefill", 1, 2048), ("attn_prefill", 33, 2048), ("attn_prefill", 100, 3000),
    ("attn_prefill", 288, 2500), ("attn_prefill_paged", 100, 3000), ("attn_prefill_paged", 17, 4100),
    ("attn_prefill_bf16kv", 64, 8200), ("attn_prefill_bf16kv", 288, 8192), ("attn_prefill_bf16x3", 100, 8300),
    ("attn_prefill_bf16kv", 256, 2048), ("attn_prefill_bf16x3", 64, 3000), ("attn_prefill_bf16kv", 17, 4100),
    ("attn_prefill", 128, 700), ("attn_prefill", 33, 500), ("attn_prefill_paged", 64, 900),
    ("attn_prefill_bf16kv", 64, 1200), ("attn_prefill_bf16x3", 100, 1000),
    # pairs (more units than clusters of four)
    ("attn_prefill", 200, 1500), ("attn_prefill_paged", 160, 2000), ("attn_prefill_bf16x3", 250, 3000),
    # clusters of four at the thresholds: 257 and 384 keys (5 and 6 tiles of 64 over four CTAs),
    # 1032 keys (9 tiles of 128), a one-row chunk
    ("attn_prefill", 17, 240), ("attn_prefill", 128, 256), ("attn_prefill_bf16kv", 32, 1000),
    ("attn_prefill_bf16x3", 1, 1100), ("attn_prefill_paged", 3, 5000),
    # clusters of eight: 1025 keys (17 tiles of 64 over eight CTAs), 2048 keys (16 tiles of 128)
    ("attn_prefill", 32, 3000), ("attn_prefill", 1, 1024), ("attn_prefill_paged", 9, 2500),
    ("attn_prefill_bf16kv", 17, 3000), ("attn_prefill_bf16kv", 1, 2047), ("attn_prefill_bf16x3", 32, 2100),
    # clusters of three (33-46 units)
    ("attn_prefill", 160, 2000), ("attn_prefill", 129, 300), ("attn_prefill_paged", 136, 1500),
    ("attn_prefill_bf16kv", 150, 2500), ("attn_prefill_bf16x3", 129, 1100),
    # a partial round of 77-92 units over clusters of three in two waves
    ("attn_prefill", 320, 4000), ("attn_prefill_paged", 352, 4000), ("attn_prefill_bf16x3", 300, 8000),
    ("attn_prefill_bf16kv", 340, 8000),
    # clusters of twelve (a non-portable size: up to 32 rows against 8192 keys or more)
    ("attn_prefill", 32, 8200), ("attn_prefill", 1, 8191), ("attn_prefill_paged", 16, 9000),
    ("attn_prefill_bf16kv", 32, 8500), ("attn_prefill_bf16x3", 1, 8191),
    # 16 units against 16384 keys or more: twelves in two waves
    ("attn_prefill", 64, 16400), ("attn_prefill_bf16kv", 40, 17000),
])
def test_every_unit_split(cp, path, C, P):
    run(cp, path, W.edge(C, P, seed=C + P))


@pytest.mark.parametrize("variant", ["lastkey", "ramp"])
@pytest.mark.parametrize("path,C", [("attn_prefill", 64), ("attn_prefill", 32), ("attn_prefill_bf16kv", 32)])
def test_every_unit_split_max_in_last_tile(cp, variant, path, C):
    """A row's maximum in its final key tile: with the unit split, that tile
    belongs to the last rank of the cluster and the merge must carry it."""
    run(cp, path, W.edge(C, 3000, variant=variant))


# The tail: 512 units of which 56 go to the pair grid; C = 2040 leaves the last
# query tile 24 rows short.
@pytest.mark.parametrize("path,C,P", [
    ("attn_prefill", 2040, 100), ("attn_prefill_paged", 2040, 100), ("attn_prefill_bf16kv", 2040, 8200),
    ("attn_prefill_bf16kv", 2040, 1000), ("attn_prefill_bf16x3", 2040, 1000),
])
def test_tail_grid_ragged(cp, path, C, P):
    run(cp, path, W.edge(C, P, seed=7))


# A last round of 8, 16, 24 or 40 units goes to clusters of eight, four or
# three (on a GB300) instead of pairs, and one of 77-92 long units to threes
# in two waves.
@pytest.mark.parametrize("path,C,P", [
    ("attn_prefill", 640, 1500), ("attn_prefill", 660, 2000), ("attn_prefill", 768, 1100),
    ("attn_prefill_paged", 1280, 1500), ("attn_prefill_bf16kv", 1300, 3000), ("attn_prefill_bf16x3", 640, 2500),
    ("attn_prefill_bf16kv", 760, 1024),
    # a last round of 80 or 88 long units over threes in two waves
    ("attn_prefill", 928, 8500), ("attn_prefill_bf16kv", 960, 8200),
    # a last round of 8 long units over twelves
    ("attn_prefill", 640, 8200), ("attn_prefill_bf16kv", 640, 8200),
])
def test_tail_grid_clusters(cp, path, C, P):
    run(cp, path, W.edge(C, P, seed=11))
