"""Every GPU path against the double-precision oracle, element by element, on
poisoned, guard-banded outputs: |err| <= 1e-4 + 1e-3 |ref| on every value (the
attention-v1 rule, "Inference Attention 2: Flash Prefill Against a Cached
Prefix", Lesson)."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import full_refs  # noqa: E402
from gpu_util import run_entry, sample_rows  # noqa: E402


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


PATHS = ["attn_prefill", "attn_prefill_bf16x3", "attn_prefill_ffma", "attn_reference_prefill"]


def _check(got, ref, what):
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{what}: {rep}"
    return rep


def _edge_cases():
    out = []
    for C in W.EDGE_C:
        for P in W.EDGE_P:
            for variant in ("plain", "lastkey", "ramp"):
                out.append((C, P, variant))
    return out


@pytest.mark.parametrize("path", PATHS)
def test_tiny_planted(cp, path):
    inp = W.tiny()
    got, guards = run_entry(getattr(cp, path), inp)
    assert guards
    _check(got, oracle.prefill(inp), f"{path} tiny")
    for t in inp.planted:
        if t >= inp.P:
            assert np.all(np.isfinite(got[t - inp.P]))


@pytest.mark.parametrize("C,P,variant", _edge_cases())
@pytest.mark.parametrize("path", PATHS)
def test_edge_sweep(cp, path, C, P, variant):
    inp = W.edge(C, P, variant=variant)
    got, guards = run_entry(getattr(cp, path), inp)
    assert guards
    _check(got, oracle.prefill(inp), f"{path} {inp.name}")


@pytest.mark.parametrize("term", W.SPLIT_TERM_CASES)
@pytest.mark.parametrize("path", ["attn_prefill", "attn_prefill_paged", "attn_prefill_ffma"])
def test_split_term_cases(cp, path, term):
    """Inputs on which a product that lost one lo part (of q, k, p or v) misses
    the tolerance on most outputs (shown on the CPU by test_split_terms.py), so
    passing them shows that the split-TF32 kernel carries every part; the FFMA
    path computes in fp32 and must pass them too."""
    inp = W.split_term_case(term)
    if path == "attn_prefill_paged":
        pg = W.to_pages(inp, seed=5)
        kp, vp = torch.from_numpy(pg.k_pages).cuda(), torch.from_numpy(pg.v_pages).cuda()
        tb = torch.from_numpy(pg.table).cuda()
        fn = lambda q, k, v, out, P, stream: cp.attn_prefill_paged(q, kp, vp, tb, out, P, stream)
    else:
        fn = getattr(cp, path)
    got, guards = run_entry(fn, inp)
    assert guards
    rep = _check(got, oracle.prefill(inp), f"{path} {inp.name}")
    print(f"{path} {inp.name}: worst err/tol {rep['worst_ratio']:.3g}")


@pytest.mark.parametrize("term", W.BF16_SPLIT_TERM_CASES)
def test_bf16x3_split_term_cases(cp, term):
    """attn_prefill_bf16x3 on inputs where a lost second bf16 term of q, k, p or
    v misses the tolerance on most outputs (shown on the CPU by
    test_split_terms_bf16.py): passing them shows that every x2 is carried."""
    inp = W.split_term_case(term)
    got, guards = run_entry(cp.attn_prefill_bf16x3, inp)
    assert guards
    rep = _check(got, oracle.prefill(inp), f"bf16x3 {inp.name}")
    print(f"attn_prefill_bf16x3 {inp.name}: worst err/tol {rep['worst_ratio']:.3g}")


@pytest.mark.parametrize("T", W.FULL_T_SMALL + W.FULL_T)
@pytest.mark.parametrize("path", ["attn_prefill", "attn_prefill_bf16x3", "attn_prefill_ffma"])
def test_full_causal(cp, path, T):
    inp = W.full_causal(T)
    if path == "attn_prefill":
        fn = lambda q, k, v, out, P, stream: cp.attn_full_causal(q, k, v, out, stream)
    else:
        fn = getattr(cp, path)
    got, guards = run_entry(fn, inp)
    assert guards
    _check(got, oracle.prefill(inp), f"{path} T={T}")
    if T == 1:
        # the single-token row has probability exactly 1 ("Inference Attention 1", Lesson),
        # so the output is V[0] as the path carries it: exact for the split-TF32 and
        # FFMA paths, V as two bf16 terms (16 significant bits, |err| <= 2^-16 |v|)
        # on the bf16x3 path
        rtol = 2.0 ** -16 if path == "attn_prefill_bf16x3" else 1e-6
        np.testing.assert_allclose(got[0], np.repeat(inp.v[0], 4, axis=0), rtol=rtol, atol=1e-7)


@pytest.mark.parametrize("path", ["attn_prefill", "attn_prefill_bf16x3", "attn_prefill_ffma"])
def test_serving_chunk_full_check(cp, path):
    """C = P = 2048 with 64 planted positions, every element against the oracle."""
    inp, ref = full_refs.serve()
    got, guards = run_entry(getattr(cp, path), inp)
    assert guards
    rep = _check(got, ref, f"{path} serve")
    print(f"{path} serve: worst err/tol {rep['worst_ratio']:.3g}")


@pytest.mark.parametrize("path", ["attn_prefill", "attn_prefill_bf16x3", "attn_prefill_ffma"])
def test_long_prefix_full_check(cp, path):
    """C = 2048 against P = 30720 (32,768 visible keys), normal(0, 0.5) inputs
    clipped to [-2, 2]: every one of the 4,194,304 outputs against the oracle,
    including the rows the split tail grid computes."""
    inp, ref = full_refs.long_prefix()
    got, guards = run_entry(getattr(cp, path), inp)
    assert guards
    rep = _check(got, ref, f"{path} long")
    print(f"{path} long prefix: worst err/tol {rep['worst_ratio']:.3g}")


def test_reference_serving_sampled(cp):
    """The starter-design reference at the timing configuration (sampled rows)."""
    inp = W.serve()
    got, guards = run_entry(cp.attn_reference_prefill, inp)
    assert guards
    rows = sample_rows(inp.C, n_random=16, seed=9)
    _check(got[rows], oracle.prefill(inp, rows=rows), "reference serve")


def test_chunk_equals_rows_of_full_prompt(cp):
    """A chunk at offset P returns the rows P.. of the whole prompt run from 0."""
    C, P = 200, 333
    full = W.full_causal(P + C, seed=4)
    part = W.Inputs(q=full.q[P:].copy(), k=full.k, v=full.v, C=C, P=P)
    a, _ = run_entry(cp.attn_prefill, part)
    b, _ = run_entry(lambda q, k, v, out, P_, s: cp.attn_full_causal(q, k, v, out, s), full)
    ref = oracle.prefill(part)
    _check(a, ref, "chunk")
    _check(b[P:], ref, "full rows")


def test_deterministic(cp):
    inp = W.edge(64, 1000)
    a, _ = run_entry(cp.attn_prefill, inp)
    b, _ = run_entry(cp.attn_prefill, inp)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_side_stream(cp):
    inp = W.edge(33, 31)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got, _ = run_entry(cp.attn_prefill, inp, stream=s)
    _check(got, oracle.prefill(inp), "side stream")


def test_no_device_error_after_runs(cp):
    run_entry(cp.attn_prefill, W.tiny())
    assert cp.attn_get_device_error() == 0


def test_argument_errors_on_device(cp):
    inp = W.edge(17, 31)
    q = torch.from_numpy(inp.q).cuda()
    k = torch.from_numpy(inp.k).cuda()
    v = torch.from_numpy(inp.v).cuda()
    out = torch.empty_like(q)
    f = cp.raw("attn_prefill")
    stream = torch.cuda.current_stream().cuda_stream
    assert f(q.data_ptr() + 4, k.data_ptr(), v.data_ptr(), out.data_ptr(), 17, 31, stream) == cp.ATTN_EALIGN
    assert f(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), -1, 31, stream) == cp.ATTN_EINVAL
    assert f(None, None, None, None, 0, 31, stream) == cp.ATTN_OK
    with pytest.raises(TypeError):
        cp.attn_prefill(q.double(), k, v, out, 31)
    with pytest.raises(ValueError):
        cp.attn_prefill(q, k[:-1], v[:-1], out, 31)
    with pytest.raises(ValueError):
        cp.attn_prefill(q.cpu(), k, v, out, 31)
