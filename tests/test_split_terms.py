"""The split-term cases have the power to catch a lost hi or lo part.

The tolerance |err| <= 1e-4 + 1e-3 |ref| is loose next to split-TF32's own
error, so on ordinary inputs a product that lost one lo part (q, k, p or v
carried as tf32 alone, 2^-11 relative) can still pass: on the serving chunk
only a lost q lo leaves the tolerance. ``workloads.split_term_case`` builds
inputs where each lost part shows. This module checks that claim on the CPU
with a model of the split-precision arithmetic written here, in float64: the
products hi*hi + hi*lo + lo*hi of "Inference Attention 2: Flash Prefill
Against a Cached Prefix" (Lesson) carried on the tensor cores as tf32 pieces,
the probabilities unnormalised against the row maximum (optionally a stale one,
lowered by a few log2 units, as a running maximum can be), the sum l from the
full probabilities. The full model must meet the oracle's tolerance on every
case, and each model with one part dropped must miss it on most outputs of
its case. The GPU parity module runs the kernels on the same inputs.
"""
import numpy as np
import pytest

import oracle
import workloads as W


def tf32_hi(x):
    """x with its 13 low mantissa bits cleared (the tf32 part), as float64."""
    bits = np.asarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
    return bits.view(np.float32).astype(np.float64)


def split(x):
    hi = tf32_hi(x)
    return hi, np.asarray(x, dtype=np.float64) - hi


def split_model(inp, drop=None, stale_log2=0.0):
    """Attention with every contraction as hi*hi + hi*lo + lo*hi; ``drop`` names
    the operand ("q", "k", "p" or "v") whose lo part is lost."""
    C, P = inp.C, inp.P
    out = np.zeros((C, W.HQ, W.D))
    visible = np.arange(P + C)[None, :] <= (P + np.arange(C))[:, None]
    for h in range(W.HQ):
        g = h // W.GROUP
        qh, ql = split(inp.q[:, h])
        kh, kl = split(inp.k[:, g])
        vh, vl = split(inp.v[:, g])
        if drop == "q":
            ql = np.zeros_like(ql)
        if drop == "k":
            kl = np.zeros_like(kl)
        if drop == "v":
            vl = np.zeros_like(vl)
        s = np.where(visible, (qh @ kh.T + qh @ kl.T + ql @ kh.T) / 8.0, -np.inf)
        ref_max = s.max(axis=1, keepdims=True) - stale_log2 * np.log(2.0)
        p = np.exp(s - ref_max).astype(np.float32)
        ph, pl = split(p)
        if drop == "p":
            pl = np.zeros_like(pl)
        l = p.astype(np.float64).sum(axis=1, keepdims=True)
        out[:, h] = (ph @ vh + ph @ vl + pl @ vh) / l
    return out.astype(np.float32)


@pytest.fixture(scope="module")
def cases():
    return {t: (W.split_term_case(t), oracle.prefill(W.split_term_case(t))) for t in W.SPLIT_TERM_CASES}


@pytest.mark.parametrize("term", W.SPLIT_TERM_CASES)
def test_full_split_model_meets_the_tolerance(cases, term):
    inp, ref = cases[term]
    for stale in (0.0, 3.3):
        rep = oracle.check(split_model(inp, None, stale), ref)
        assert rep["n_bad"] == 0 and rep["worst_ratio"] < 0.1, (term, stale, rep)


@pytest.mark.parametrize("term,drop", [("q", "q"), ("k", "k"), ("pv", "p"), ("pv", "v")])
def test_a_lost_lo_part_leaves_the_tolerance(cases, term, drop):
    inp, ref = cases[term]
    for stale in (0.0, 3.3):
        rep = oracle.check(split_model(inp, drop, stale), ref)
        assert rep["n_bad"] >= rep["n"] // 4 and rep["worst_ratio"] > 5.0, (term, drop, stale, rep)
