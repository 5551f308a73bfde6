"""The oracle against facts fixed by the pages and by the mathematics (CPU only)."""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from conftest import read_golden
from oracle_pins import ALL_PINS
from online_model import online_rows


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.attention)


def test_worked_example_online_intermediates(golden_dir):
    """The tile update the kernels run, replayed on the page's worked example
    ("FlashAttention and inference kernels", Exercises 1) with tiles of two keys,
    reproduces every intermediate the page prints."""
    g = read_golden(f"{golden_dir}/online_softmax_worked_example.txt")
    s = [float(x) for x in g["scores_tile1"] + g["scores_tile2"]]
    vals = [[float(x)] for x in g["values_tile1"] + g["values_tile2"]]
    trace = []
    res = online_rows(s, vals, tile=2, trace=trace)

    def near(x, printed):
        decimals = len(printed.split(".")[1]) if "." in printed else 0
        return abs(x - float(printed)) <= 1.5 * 10.0 ** (-decimals)

    (m1, l1, o1), (m2, l2, o2) = trace
    assert near(m1, g["tile1_m"][0]) and near(l1, g["tile1_l"][0]) and near(o1[0], g["tile1_O"][0])
    assert near(m2, g["tile2_m"][0]) and near(l2, g["tile2_l"][0]) and near(o2[0], g["tile2_O"][0])
    assert near(math.exp(m1 - m2), g["tile2_correction"][0])
    assert near(res[0], g["result"][0])
    w = [math.exp(x) for x in s]
    for got, printed in zip(w, g["direct_weights"]):
        assert abs(got - float(printed)) <= 1.5 * 10.0 ** (-(len(printed.split(".")[1])))
    assert near(sum(w), g["direct_weight_sum"][0])


@pytest.mark.parametrize("tile", [1, 2, 3, 64, 128])
@pytest.mark.parametrize("stale", [None, 0.0, 8.0 * math.log(2.0)])
def test_online_model_matches_oracle(tile, stale):
    """Any tile width, with or without a stale reference maximum, gives the exact
    attention of the oracle (the update is exact, page 2: "mathematically
    identical to standard attention, not an approximation")."""
    inp = W.tiny()
    ref = oracle.prefill(inp, rows=[0, 8, 16])
    for r, i in enumerate([0, 8, 16]):
        for h in (0, 1, 5, 31):
            g = h // 4
            n = inp.P + i + 1
            s = [float(np.dot(inp.q[i, h].astype(np.float64), inp.k[j, g].astype(np.float64))) * 0.125
                 for j in range(n)]
            vals = [list(inp.v[j, g].astype(np.float64)) for j in range(n)]
            got = online_rows(s, vals, tile, stale_threshold=stale)
            np.testing.assert_allclose(got, ref[r, h], rtol=1e-11, atol=1e-12)


def test_online_model_fully_masked_tile():
    """A tile whose scores are all -inf before any visible key leaves m at -inf and
    produces no NaN (the teaching kernel's guard, page 2)."""
    s = [-math.inf, -math.inf, 1.0, 2.0]
    got = online_rows(s, [[1.0], [2.0], [3.0], [4.0]], tile=2)
    expect = (3.0 * math.e + 4.0 * math.e ** 2) / (math.e + math.e ** 2)
    assert abs(got[0] - expect) < 1e-12


def test_rows_subset_matches_full():
    inp = W.edge(33, 31)
    full = oracle.prefill(inp)
    rows = [32, 0, 17, 5]
    sub = oracle.prefill(inp, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])


def test_thread_count_does_not_change_result():
    inp = W.edge(17, 31)
    a = oracle.prefill(inp, threads=1)
    b = oracle.prefill(inp, threads=4)
    np.testing.assert_array_equal(a, b)


def test_bad_arguments_raise():
    inp = W.edge(4, 3)
    with pytest.raises(ValueError):
        oracle.attention(inp.q, inp.k, inp.v, 2)          # T != P + C
    with pytest.raises(RuntimeError):
        oracle.attention(inp.q, inp.k, inp.v, 3, rows=[4])  # row outside the chunk


def test_check_rule():
    ref = np.array([0.0, 1.0, -2.0, 10.0])
    tol = 1e-4 + 1e-3 * np.abs(ref)
    assert oracle.check(ref + 0.99 * tol, ref)["n_bad"] == 0
    assert oracle.check(ref + 1.01 * tol, ref)["n_bad"] == 4
    assert oracle.check(np.array([np.nan, 1.0, -2.0, 10.0]), ref)["n_bad"] == 1
    assert oracle.check(np.array([np.inf, 1.0, -2.0, 10.0]), ref)["n_bad"] == 1


def test_paged_oracle_equals_contiguous():
    """Gathering a paged cache through its block table (token t at slot t % 16 of
    page table[t // 16], "FlashAttention and inference kernels", PagedAttention)
    gives back the contiguous cache, so the paged oracle equals the oracle."""
    for C, P in ((17, 31), (1, 0), (33, 1000)):
        inp = W.edge(C, P)
        pg = W.to_pages(inp, seed=C + P)
        np.testing.assert_array_equal(oracle.gather_pages(pg.k_pages, pg.table, inp.T), inp.k)
        np.testing.assert_array_equal(oracle.gather_pages(pg.v_pages, pg.table, inp.T), inp.v)
        np.testing.assert_array_equal(oracle.prefill_paged(inp.q, pg.k_pages, pg.v_pages, pg.table, P),
                                      oracle.prefill(inp))


def test_paged_gather_follows_the_table():
    """A hand-made two-page cache with the pages swapped: token 0..15 live in
    physical page 1, tokens 16..19 in physical page 0."""
    pages = np.zeros((2, 16, 1, 1), np.float32)
    pages[1, :, 0, 0] = np.arange(16)
    pages[0, :4, 0, 0] = 16 + np.arange(4)
    got = oracle.gather_pages(pages, np.array([1, 0]), 20)
    np.testing.assert_array_equal(got[:, 0, 0], np.arange(20))


def test_score_matrix_by_brute_force():
    """Every entry of the oracle's score workspace is the plain dot product of
    its (position, head) query and (key, KV head h / 4) key, times 1/8, and -inf
    exactly where the key is past the row's position."""
    inp = W.edge(5, 3)
    S = oracle.score_matrix(inp.q, inp.k, inp.P)
    assert S.shape == (W.HQ, 5, 8)
    for h in (0, 3, 4, 17, 31):
        for i in range(5):
            for j in range(8):
                if j > inp.P + i:
                    assert S[h, i, j] == -math.inf
                else:
                    dot = sum(float(inp.q[i, h, d]) * float(inp.k[j, h // 4, d]) for d in range(W.D))
                    assert abs(S[h, i, j] - dot / 8.0) <= 1e-14


def test_probability_matrix_rows_and_pipeline_equal_the_oracle():
    """Rows of the probability workspace sum to 1, are exactly 0 above the
    diagonal and exactly 1 on a single-token row; multiplied by V they give the
    C oracle's attention, which is computed by a different route (two passes
    per row, no matrix)."""
    for inp in (W.edge(1, 0), W.edge(17, 31), W.edge(33, 0, variant="ramp"), W.tiny()):
        Pm = oracle.probability_matrix(oracle.score_matrix(inp.q, inp.k, inp.P))
        np.testing.assert_allclose(Pm.sum(axis=-1), 1.0, rtol=0, atol=1e-13)
        above = np.arange(inp.P + inp.C)[None, :] > (inp.P + np.arange(inp.C))[:, None]
        assert (Pm[:, above] == 0).all()
        if inp.C == 1 and inp.P == 0:
            assert (Pm[:, 0, 0] == 1.0).all()
        v = inp.v.astype(np.float64)
        out = np.stack([Pm[h] @ v[:, h // 4, :] for h in range(W.HQ)], axis=1)
        np.testing.assert_allclose(out, oracle.prefill(inp), rtol=1e-12, atol=1e-13)


def test_bf16_decoding_follows_the_format():
    """bf16 = sign, 8 exponent bits (bias 127), 7 fraction bits: values fixed by
    that definition, including a subnormal, the largest finite, infinity and -0."""
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x4080, 0x0001, 0x7F7F, 0x7F80, 0x8000, 0x3EAB], dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 4.0, 2.0 ** -133, (2.0 - 2.0 ** -7) * 2.0 ** 127, math.inf, -0.0,
            (1.0 + 43.0 / 128.0) * 2.0 ** -2]
    got = oracle.bf16_to_float(bits)
    for g, w in zip(got.tolist(), want):
        assert g == w and math.copysign(1.0, g) == math.copysign(1.0, w)


def test_bf16_inputs_are_truncations_and_oracle_uses_their_values():
    """The workload's bf16 bits keep the upper half of each fp32 value (the
    difference is below 2^-7 relative and never rounds up), and the bf16 oracle
    equals the fp32 oracle run on the decoded values."""
    inp = W.edge(17, 31)
    kv = W.to_bf16(inp)
    kd = oracle.bf16_to_float(kv.k).astype(np.float64)
    k = inp.k.astype(np.float64)
    assert (np.abs(kd) <= np.abs(k)).all() and (np.abs(k - kd) <= 2.0 ** -7 * np.abs(k)).all()
    ref = oracle.prefill_bf16kv(inp.q, kv.k, kv.v, inp.P)
    np.testing.assert_array_equal(
        ref, oracle.attention(inp.q, kd.astype(np.float32), oracle.bf16_to_float(kv.v), inp.P))
    # planted 4.0 survives exactly, so planted rows still score 128
    t = W.tiny()
    assert (oracle.bf16_to_float(W.to_bf16(t).k)[t.k == 4.0] == 4.0).all()
