"""Pins for the oracle: facts fixed by the pages and by the mathematics.

Each pin takes an ``attention(q, k, v, P, scale=..., rows=None)`` callable with
the oracle's signature and raises AssertionError when the callable disagrees
with the fact. The oracle must pass all of them; each deliberately broken copy
of the oracle (tests/test_oracle_mutants.py) must fail at least one.

None of these re-types the oracle's formula: the expected values are closed
forms, numbers printed on the pages, symmetries of attention, or a
differently-shaped computation (the materialised three-kernel pipeline).
"""
from __future__ import annotations

import math
import os

import numpy as np

import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden(name):
    from conftest import read_golden
    return read_golden(os.path.join(HERE, "golden", name))


def _close(a, b, rel=1e-12, abs_=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.abs(a - b)
    bad = ~(err <= abs_ + rel * np.abs(b))
    assert not bad.any(), f"{what}: {int(bad.sum())} mismatches, max err {err.max():.3e}"


# --- 1. The worked example ("FlashAttention and inference kernels", Exercises 1) ---------

def pin_worked_example(attention):
    """One query row, D = 1, scale 1: scores [1, 3, 2, 5], values [10, 20, 30, 40].

    The page prints the result as 36.88 (two decimals)."""
    g = _golden("online_softmax_worked_example.txt")
    s = [float(x) for x in g["scores_tile1"] + g["scores_tile2"]]
    vals = [float(x) for x in g["values_tile1"] + g["values_tile2"]]
    q = np.ones((1, 1, 1), np.float32)
    k = np.array(s, np.float32).reshape(4, 1, 1)
    v = np.array(vals, np.float32).reshape(4, 1, 1)
    out = attention(q, k, v, 3, scale=1.0)
    printed = float(g["result"][0])
    assert abs(out[0, 0, 0] - printed) <= 1.5 * 0.01, (out[0, 0, 0], printed)
    # The same data with the values paired to other keys gives another answer:
    # the oracle must weight each value by its own key's score.
    v2 = np.array(vals[::-1], np.float32).reshape(4, 1, 1)
    out2 = attention(q, k, v2, 3, scale=1.0)
    assert abs(out2[0, 0, 0] - printed) > 1.0


# --- 2. Closed forms ------------------------------------------------------------------

def pin_single_token(attention):
    """C = 1, P = 0: the only visible key has probability exactly 1, so the output
    is V[0] of the head's KV head, exactly ("Inference Attention 1", Lesson)."""
    inp = W.make_inputs(1, 0, seed=11)
    out = attention(inp.q, inp.k, inp.v, 0)
    for h in range(W.HQ):
        assert np.array_equal(out[0, h], inp.v[0, h // W.GROUP].astype(np.float64)), h


def pin_uniform_weights(attention):
    """q = 0 gives every visible key the same weight, so row i returns the mean of
    V over keys 0..P+i. With V[j][g][d] = (g + 1) j + d / 64 that mean is
    (g + 1)(P + i) / 2 + d / 64: it checks the causal bound, the prefix offset,
    the head-to-KV-head map and the d index at once (page 1, Lesson)."""
    for C, P in ((5, 0), (7, 9), (3, 40)):
        T = P + C
        q = np.zeros((C, W.HQ, W.D), np.float32)
        k = W.uniform(5, T * W.HKV * W.D).reshape(T, W.HKV, W.D)
        j = np.arange(T, dtype=np.float64)[:, None, None]
        g = np.arange(W.HKV, dtype=np.float64)[None, :, None]
        d = np.arange(W.D, dtype=np.float64)[None, None, :]
        v = ((g + 1) * j + d / 64.0).astype(np.float32)
        out = attention(q, k, v, P)
        i = np.arange(C, dtype=np.float64)[:, None, None]
        h = np.arange(W.HQ)[None, :, None]
        expect = (h // W.GROUP + 1) * (P + i) / 2.0 + d / 64.0
        _close(out, expect, rel=1e-13, abs_=1e-12, what=f"uniform weights C={C} P={P}")


def pin_head_map(attention):
    """V constant over keys within each KV head: any weights give that constant.
    Query head h must read KV head h / 4 (page 1, Lesson: 32 query heads, 8 KV
    heads, head h reading KV head h / 4)."""
    C, P = 6, 10
    inp = W.make_inputs(C, P, seed=21)
    g = np.arange(W.HKV, dtype=np.float32)[None, :, None]
    d = np.arange(W.D, dtype=np.float32)[None, None, :]
    v = np.broadcast_to(100.0 * g + d, inp.v.shape).astype(np.float32).copy()
    out = attention(inp.q, inp.k, v, P)
    for h in range(W.HQ):
        _close(out[:, h, :], np.broadcast_to(100.0 * (h // 4) + np.arange(W.D), (C, W.D)),
               rel=1e-14, abs_=1e-12, what=f"head {h}")


def pin_scale_two_keys(attention):
    """Two visible keys, k0 = 0 and k1 = 1 in every element, q = 1: the scores are 0
    and 64 / 8 = 8 (scale exactly 1/8, page 1, Lesson), so with values 3 and -1
    the output is (3 - e^8) / (1 + e^8)."""
    q = np.ones((1, W.HQ, W.D), np.float32)
    k = np.zeros((2, W.HKV, W.D), np.float32)
    k[1] = 1.0
    v = np.zeros((2, W.HKV, W.D), np.float32)
    v[0] = 3.0
    v[1] = -1.0
    out = attention(q, k, v, 1)
    expect = (3.0 - math.exp(8.0)) / (1.0 + math.exp(8.0))
    _close(out, np.full(out.shape, expect), rel=1e-14, abs_=1e-15, what="two keys")


def pin_dot_product_index(attention):
    """The score pairs element d of q with element d of k. Head h's query is 8 at
    d_h = (7 h + 3) mod 64 and 0 elsewhere; key 1 of every KV head is 1 at each
    d_h of its heads and 0 elsewhere, key 0 is zero. Scores are 0 and 8 * 1 / 8 = 1,
    so with values 2 and -1 each head returns (2 - e) / (1 + e)."""
    q = np.zeros((1, W.HQ, W.D), np.float32)
    k = np.zeros((2, W.HKV, W.D), np.float32)
    for h in range(W.HQ):
        dh = (7 * h + 3) % W.D
        q[0, h, dh] = 8.0
    for g in range(W.HKV):
        for h in range(W.GROUP * g, W.GROUP * (g + 1)):
            k[1, g, (7 * h + 3) % W.D] = 1.0
    # a head of the group must not pick up its neighbours' ones
    v = np.zeros((2, W.HKV, W.D), np.float32)
    v[0], v[1] = 2.0, -1.0
    out = attention(q, k, v, 1)
    expect = (2.0 - math.e) / (1.0 + math.e)
    _close(out, np.full(out.shape, expect), rel=1e-14, abs_=1e-15, what="dot index")


def pin_ramp_geometric(attention):
    """Ramp hazard (each row's maximum on its own diagonal key). Head 0: q = 1 and
    key j = (j + 1) / 16 in every element with T = 32, so scores are (j + 1) / 2
    and weights grow geometrically with ratio x = e^(1/2). With V[j][0][:] = j,
    row i (n = P + i + 1 visible keys) returns
        sum_j j x^j / sum_j x^j = x (1 - n x^(n-1) + (n-1) x^n) / ((1 - x)(x^n - 1))."""
    C, P = 17, 15
    inp = W.ramp(W.make_inputs(C, P, seed=3))
    assert inp.T == 32
    v = inp.v.copy()
    v[:, 0, :] = np.arange(inp.T, dtype=np.float32)[:, None]
    out = attention(inp.q, inp.k, v, P)
    x = math.exp(0.5)
    for i in range(C):
        n = P + i + 1
        s1 = x * (1.0 - n * x ** (n - 1) + (n - 1) * x ** n) / (1.0 - x) ** 2
        s0 = (x ** n - 1.0) / (x - 1.0)
        _close(out[i, 0, :], np.full(W.D, s1 / s0), rel=1e-12, abs_=1e-12, what=f"ramp row {i}")


# --- 3. Symmetries and invariants ----------------------------------------------------

def pin_chunk_consistency(attention):
    """A chunk at offset P returns the same rows as the whole prompt run causally
    from position 0 (page 1, Lesson: chunked prefill runs a chunk against
    everything already cached)."""
    C, P = 9, 23
    full = W.make_inputs(P + C, 0, seed=31)
    whole = attention(full.q, full.k, full.v, 0)
    part = attention(full.q[P:], full.k, full.v, P)
    _close(part, whole[P:], rel=1e-14, abs_=1e-15, what="chunk vs whole prompt")


def pin_prefix_permutation(attention):
    """Every chunk row sees the whole prefix, so permuting cached rows 0..P-1 of K
    and V together changes nothing."""
    C, P = 5, 40
    inp = W.make_inputs(C, P, seed=41)
    base = attention(inp.q, inp.k, inp.v, P)
    perm = np.random.default_rng(0).permutation(P)
    k2, v2 = inp.k.copy(), inp.v.copy()
    k2[:P], v2[:P] = inp.k[perm], inp.v[perm]
    out = attention(inp.q, k2, v2, P)
    _close(out, base, rel=1e-12, abs_=1e-14, what="prefix permutation")


def pin_affine_values(attention):
    """The weights of a row sum to one: V -> aV + b maps the output to a out + b."""
    C, P = 6, 12
    inp = W.make_inputs(C, P, seed=51)
    base = attention(inp.q, inp.k, inp.v, P)
    out = attention(inp.q, inp.k, (2.0 * inp.v + 0.5).astype(np.float32), P)
    _close(out, 2.0 * base + 0.5, rel=1e-12, abs_=1e-13, what="affine V")


def pin_gqa_equivalence(attention):
    """Grouped-query attention equals multi-head attention on KV heads replicated
    four times (head h reads KV head h / 4)."""
    C, P = 4, 9
    inp = W.make_inputs(C, P, seed=61)
    base = attention(inp.q, inp.k, inp.v, P)
    k32 = np.repeat(inp.k, W.GROUP, axis=1)
    v32 = np.repeat(inp.v, W.GROUP, axis=1)
    out = attention(inp.q, k32, v32, P)
    _close(out, base, rel=1e-14, abs_=1e-15, what="GQA vs replicated MHA")


def pin_planted_rows(attention):
    """Planted query rows (4.0 in head 0) meet planted keys at score 128 (page 1,
    Lesson). Those keys carry V = 4.0 and every other key trails by more than 100
    in score, so head 0 of a planted row returns 4.0 to within 1e-12; every
    output stays finite."""
    inp = W.tiny()
    out = attention(inp.q, inp.k, inp.v, inp.P)
    assert np.isfinite(out).all()
    for t in inp.planted:
        if t >= inp.P:
            _close(out[t - inp.P, 0, :], np.full(W.D, 4.0), rel=0, abs_=1e-12, what=f"planted row {t}")


def pin_last_key(attention):
    """Only the last key of the sequence is planted (page 1, Lesson). Row C-1 sees it
    and returns 4.0 in head 0; every other row cannot see it and is unchanged."""
    C, P = 17, 31
    plain = W.edge(C, P, seed=1, variant="plain")
    last = W.edge(C, P, seed=1, variant="lastkey")
    a = attention(plain.q, plain.k, plain.v, P)
    b = attention(last.q, last.k, last.v, P)
    _close(b[C - 1, 0, :], np.full(W.D, 4.0), rel=0, abs_=1e-12, what="last key row")
    np.testing.assert_array_equal(a[:C - 1], b[:C - 1])


# --- 4. Brute force: the three-kernel pipeline made literal ------------------------

def three_step(q, k, v, P, scale=0.125):
    """Scores matrix -> row softmax -> weighted sum, as the eager pipeline of
    "Inference Attention 1: The Full Score Matrix" (Lesson) runs it: -inf above
    the (offset) diagonal, 0 after the softmax. float64 numpy, tiny sizes only."""
    C, HQ, D = q.shape
    T, HKV, _ = k.shape
    group = HQ // HKV
    out = np.zeros((C, HQ, D))
    allowed = np.arange(T)[None, :] <= (P + np.arange(C))[:, None]
    for h in range(HQ):
        g = h // group
        S = (q[:, h, :].astype(np.float64) @ k[:, g, :].astype(np.float64).T) * scale
        S = np.where(allowed, S, -np.inf)
        S = S - S.max(axis=1, keepdims=True)
        Pm = np.exp(S)
        Pm = Pm / Pm.sum(axis=1, keepdims=True)
        out[:, h, :] = Pm @ v[:, g, :].astype(np.float64)
    return out


def pin_brute_force(attention):
    cases = [W.tiny(), W.edge(1, 0), W.edge(17, 31), W.edge(33, 0), W.edge(33, 31, variant="lastkey")]
    for inp in cases:
        _close(attention(inp.q, inp.k, inp.v, inp.P), three_step(inp.q, inp.k, inp.v, inp.P),
               rel=1e-12, abs_=1e-13, what=inp.name)


ALL_PINS = [pin_worked_example, pin_single_token, pin_uniform_weights, pin_head_map,
            pin_scale_two_keys, pin_dot_product_index, pin_ramp_geometric, pin_chunk_consistency,
            pin_prefix_permutation, pin_affine_values, pin_gqa_equivalence,
            pin_planted_rows, pin_last_key, pin_brute_force]
