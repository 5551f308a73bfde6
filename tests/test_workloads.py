"""The seeded input generator (CPU only)."""
import numpy as np
import pytest

import workloads as W


def test_splitmix64_published_vector():
    # The five first outputs for seed 1234567 that accompany the published
    # SplitMix64 reference code (Vigna, splitmix64.c test vector).
    assert W.splitmix64(1234567, 5).tolist() == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_uniform_range_and_exactness():
    u = W.uniform(7, 1 << 16)
    assert u.dtype == np.float32
    assert u.min() >= -1.0 and u.max() < 1.0
    # every value is a multiple of 2^-23 (24 kept bits mapped onto [-1, 1))
    assert np.all((u.astype(np.float64) * (1 << 23)) % 1 == 0)
    assert abs(float(u.mean())) < 0.02 and abs(float(u.var()) - 1 / 3) < 0.01


def test_normal_clipped_moments():
    z = W.normal_clipped(9, 1 << 16)
    assert z.min() >= -2.0 and z.max() <= 2.0
    assert abs(float(z.mean())) < 0.01 and abs(float(z.std()) - 0.5) < 0.01


def test_deterministic_and_seed_separated():
    a = W.make_inputs(3, 5, seed=1)
    b = W.make_inputs(3, 5, seed=1)
    c = W.make_inputs(3, 5, seed=2)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v)):
        np.testing.assert_array_equal(x, y)
    assert not np.array_equal(a.q, c.q)
    # q, k and v use seeds s, s+1, s+2: k of seed 1 is the stream q of seed 2 starts with
    np.testing.assert_array_equal(a.k.ravel()[:10], W.uniform(2, 10))


def test_shapes_and_pairs():
    inp = W.make_inputs(17, 31)
    assert inp.q.shape == (17, 32, 64) and inp.k.shape == (48, 8, 64) and inp.v.shape == (48, 8, 64)
    assert inp.pairs == sum(31 + i + 1 for i in range(17)) == 680
    assert W.serve().pairs == 6_292_480


def test_planting():
    inp = W.tiny()
    assert inp.planted.tolist() == list(W.TINY_PLANTED)
    for t in W.TINY_PLANTED:
        assert np.all(inp.k[t, 0] == 4.0) and np.all(inp.v[t, 0] == 4.0)
        if t >= inp.P:
            assert np.all(inp.q[t - inp.P, 0] == 4.0)
    # planted query meets planted key at score 64 * 16 / 8 = 128
    assert float(inp.q[0, 0] @ inp.k[0, 0]) / 8 == 128.0
    with pytest.raises(ValueError):
        W.make_inputs(2, 2, planted=[4])


def test_serve_planted_positions_distinct_and_seeded():
    a = W.distinct_positions(4, 64, 4096)
    b = W.distinct_positions(4, 64, 4096)
    assert len(set(a.tolist())) == 64 and np.array_equal(a, b)
    assert a.min() >= 0 and a.max() < 4096


def test_ramp_puts_row_max_on_diagonal():
    inp = W.edge(17, 31, variant="ramp")
    s = (inp.q[:, 0, :].astype(np.float64) @ inp.k[:, 0, :].astype(np.float64).T) / 8
    for i in range(inp.C):
        visible = s[i, : inp.P + i + 1]
        assert int(np.argmax(visible)) == inp.P + i


def test_lastkey_variant():
    inp = W.edge(33, 1000, variant="lastkey")
    assert inp.planted.tolist() == [1032]
    assert np.all(inp.q[32, 0] == 4.0)


def test_to_pages_layout():
    inp = W.edge(17, 31)
    pg = W.to_pages(inp, seed=3, spare_pages=4)
    assert pg.k_pages.shape == ((48 + 15) // 16 + 4, 16, 8, 64)
    assert len(set(pg.table.tolist())) == len(pg.table)        # distinct physical pages
    for t in (0, 15, 16, 31, 47):
        np.testing.assert_array_equal(pg.k_pages[pg.table[t // 16], t % 16], inp.k[t])
        np.testing.assert_array_equal(pg.v_pages[pg.table[t // 16], t % 16], inp.v[t])
    unused = np.setdiff1d(np.arange(pg.k_pages.shape[0]), pg.table)
    assert np.isnan(pg.k_pages[unused]).all() and np.isnan(pg.v_pages[unused]).all()
