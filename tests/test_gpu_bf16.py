"""attn_prefill_bf16kv against the oracle on the values the bf16 cache holds,
with the fp32 contract's tolerance (1e-4 + 1e-3 |ref|): the tile edges, the
planted and last-key cases, the serving chunk and the long prefix sampled."""
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


def run_bf16(cp, inp, kv=None):
    kv = W.to_bf16(inp) if kv is None else kv
    q = torch.from_numpy(inp.q).cuda()
    k = torch.from_numpy(kv.k.view(np.int16)).cuda().view(torch.bfloat16)
    v = torch.from_numpy(kv.v.view(np.int16)).cuda().view(torch.bfloat16)
    g = GuardedOut(inp.C)
    cp.attn_prefill_bf16kv(q, k, v, g.out, inp.P)
    torch.cuda.synchronize()
    return g.numpy(), g.guards_intact(), kv


def check(got, ref, what):
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{what}: {rep}"


@pytest.mark.parametrize("C,P", [(1, 0), (2, 0), (17, 31), (33, 0), (64, 1000), (100, 77), (129, 127),
                                 (257, 0), (31, 4097)])
def test_matches_oracle_at_tile_edges(cp, C, P):
    inp = W.edge(C, P, seed=C * 3 + P)
    got, guards, kv = run_bf16(cp, inp)
    assert guards
    check(got, oracle.prefill_bf16kv(inp.q, kv.k, kv.v, P), f"C={C} P={P}")


@pytest.mark.parametrize("variant", ["lastkey", "ramp"])
def test_variants(cp, variant):
    inp = W.edge(33, 1000, variant=variant)
    got, _, kv = run_bf16(cp, inp)
    assert np.isfinite(got).all()
    check(got, oracle.prefill_bf16kv(inp.q, kv.k, kv.v, inp.P), variant)


def test_planted_tiny(cp):
    inp = W.tiny()
    got, guards, kv = run_bf16(cp, inp)
    assert guards and np.isfinite(got).all()
    check(got, oracle.prefill_bf16kv(inp.q, kv.k, kv.v, inp.P), "tiny planted")


def test_full_prompts(cp):
    for T in (257, 512):
        inp = W.full_causal(T, seed=T)
        got, _, kv = run_bf16(cp, inp)
        check(got, oracle.prefill_bf16kv(inp.q, kv.k, kv.v, 0), f"T={T}")


def test_serving_chunk_full(cp):
    """Every element of the serving chunk against the oracle on the stored values."""
    inp, kv, ref = full_refs.serve_bf16()
    got, guards, _ = run_bf16(cp, inp, kv)
    assert guards
    check(got, ref, "serve")


def test_long_prefix_full(cp):
    """Every element of the long prefix (C = 2048, P = 30720) against the oracle."""
    inp, kv, ref = full_refs.long_prefix_bf16()
    got, guards, _ = run_bf16(cp, inp, kv)
    assert guards
    check(got, ref, "long prefix")


@pytest.mark.parametrize("term", ["q", "pv1"])
def test_split_term_cases(cp, term):
    """Inputs on which a lost second bf16 term of q or of the probabilities
    misses the tolerance on most outputs (shown on the CPU by
    test_split_terms_bf16.py); K and V are used as stored, so they have none."""
    inp = W.split_term_case(term)
    got, guards, kv = run_bf16(cp, inp)
    assert guards
    rep = oracle.check(got, oracle.prefill_bf16kv(inp.q, kv.k, kv.v, inp.P))
    assert rep["n_bad"] == 0, f"{inp.name}: {rep}"
    print(f"attn_prefill_bf16kv {inp.name}: worst err/tol {rep['worst_ratio']:.3g}")


def test_agrees_with_the_fp32_kernel_on_the_same_values(cp):
    """attn_prefill on the decoded fp32 cache computes the same attention."""
    inp = W.edge(200, 300, seed=9)
    got, _, kv = run_bf16(cp, inp)
    q = torch.from_numpy(inp.q).cuda()
    k = torch.from_numpy(oracle.bf16_to_float(kv.k)).cuda()
    v = torch.from_numpy(oracle.bf16_to_float(kv.v)).cuda()
    out = torch.empty_like(q)
    cp.attn_prefill(q, k, v, out, inp.P)
    torch.cuda.synchronize()
    check(got, out.cpu().numpy().astype(np.float64), "bf16 kernel vs fp32 kernel")


def test_argument_checks(cp):
    inp = W.edge(4, 3)
    q = torch.from_numpy(inp.q).cuda()
    k32 = torch.from_numpy(inp.k).cuda()
    out = torch.empty_like(q)
    with pytest.raises(ValueError):
        cp.attn_prefill_bf16kv(q, k32, k32, out, 3)  # fp32 cache where bf16 is required
    f = cp.raw("attn_prefill_bf16kv")
    kb = torch.zeros(7, 8, 64, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert f(q.data_ptr(), kb.data_ptr() + 2, kb.data_ptr(), out.data_ptr(), 4, 3, s) == cp.ATTN_EALIGN
    assert f(None, None, None, None, 0, 3, s) == cp.ATTN_OK
    assert f(q.data_ptr(), None, kb.data_ptr(), out.data_ptr(), 4, 3, s) == cp.ATTN_EINVAL
