"""The three-kernel score-matrix pipeline ("Inference Attention 1: The Full
Score Matrix", Lesson) against the oracle: the output on the page's checked
prompt lengths (1, 17, 33, 257, 512 tokens) and on chunks with a cached
prefix, and each step's workspace against the oracle's score and probability
matrices."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import GuardedOut, device_inputs, sample_rows  # noqa: E402


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


def workspace(cp, C, P):
    n = cp.attn_naive_workspace_bytes(C, P) // 4
    ws = torch.empty(n + 4, dtype=torch.float32, device="cuda")
    ws.view(torch.int32).fill_(-1)
    return ws


def check(got, ref, what):
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{what}: {rep}"


def run_pipeline(cp, inp):
    q, k, v = device_inputs(inp)
    g = GuardedOut(inp.C)
    ws = workspace(cp, inp.C, inp.P)
    cp.attn_naive_prefill(q, k, v, g.out, ws, inp.P)
    torch.cuda.synchronize()
    return g.numpy(), g.guards_intact()


@pytest.mark.parametrize("T", [1, 17, 33, 257, 512])
def test_full_prompt_matches_oracle(cp, T):
    inp = W.edge(T, 0, seed=T)
    got, guards = run_pipeline(cp, inp)
    assert guards
    check(got, oracle.prefill(inp), f"T={T}")
    if T == 1:  # the single-token row: the value itself
        np.testing.assert_array_equal(got[0], np.repeat(inp.v[0], 4, axis=0))


@pytest.mark.parametrize("C,P", [(100, 77), (64, 1000), (3, 61)])
def test_chunk_with_prefix_matches_oracle(cp, C, P):
    inp = W.edge(C, P, seed=C + P)
    got, guards = run_pipeline(cp, inp)
    assert guards
    check(got, oracle.prefill(inp), f"C={C} P={P}")


def test_planted_scores_do_not_overflow(cp):
    """Planted rows score 128 against each other; without the row maximum the
    exponential overflows."""
    inp = W.tiny()
    got, _ = run_pipeline(cp, inp)
    assert np.isfinite(got).all()
    check(got, oracle.prefill(inp), "tiny planted")


def test_each_step_against_the_oracle_matrices(cp):
    inp = W.edge(45, 19, seed=4)
    C, P, T = inp.C, inp.P, inp.P + inp.C
    q, k, v = device_inputs(inp)
    ws = workspace(cp, C, P)
    S = ws[:32 * C * T].view(32, C, T)
    cp.attn_naive_scores(q, k, ws, P)
    torch.cuda.synchronize()
    got_s = S.cpu().numpy()
    ref_s = oracle.score_matrix(inp.q, inp.k, P)
    above = np.isinf(ref_s)
    assert (got_s[above] == -np.inf).all()
    check(got_s[~above], ref_s[~above], "scores")
    cp.attn_naive_softmax(ws, C, P)
    torch.cuda.synchronize()
    got_p = S.cpu().numpy()
    assert (got_p[above] == 0).all()
    np.testing.assert_allclose(got_p, oracle.probability_matrix(ref_s), rtol=1e-5, atol=1e-7)
    g = GuardedOut(C)
    cp.attn_naive_weighted_sum(ws, v, g.out, P)
    torch.cuda.synchronize()
    check(g.numpy(), oracle.prefill(inp), "weighted sum")
    assert g.guards_intact()
    # nothing past the matrix was touched
    assert (ws[32 * C * T:].view(torch.int32) == -1).all()


def test_page_sizes_sampled_and_equal_to_flash(cp):
    """T = 2048, the largest size the page measures: sampled rows against the
    oracle, and the whole output against the flash kernel within tolerance."""
    inp = W.full_causal(2048)
    got, guards = run_pipeline(cp, inp)
    assert guards
    rows = sample_rows(inp.C, n_random=12, seed=3)
    check(got[rows], oracle.prefill(inp, rows=rows), "T=2048 sampled")
    q, k, v = device_inputs(inp)
    flash = torch.empty_like(q)
    cp.attn_prefill(q, k, v, flash, 0)
    torch.cuda.synchronize()
    check(got, flash.cpu().numpy().astype(np.float64), "pipeline vs flash")


def test_workspace_and_argument_errors(cp):
    inp = W.edge(17, 5)
    q, k, v = device_inputs(inp)
    out = torch.empty_like(q)
    small = torch.empty(cp.attn_naive_workspace_bytes(17, 5) // 4 - 1, dtype=torch.float32, device="cuda")
    f = cp.raw("attn_naive_prefill")
    s = torch.cuda.current_stream().cuda_stream
    assert f(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), small.data_ptr(), small.numel() * 4,
             17, 5, s) == cp.ATTN_ESPACE
    assert f(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), None, 0, 17, 5, s) == cp.ATTN_ESPACE
    assert f(None, None, None, None, None, 0, 0, 5, s) == cp.ATTN_OK
    assert cp.raw("attn_naive_softmax")(small.data_ptr() + 4, 17, 5, s) == cp.ATTN_EALIGN
    assert cp.attn_naive_workspace_bytes(2048, 0) == 32 * 2048 * 2048 * 4
