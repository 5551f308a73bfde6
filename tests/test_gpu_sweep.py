"""A seeded random sweep of (C, P) shapes for every prefill path and of
context-length mixes for decode, each output checked in full against the
oracle: shapes nobody picked by hand (ragged tails, prefixes that are not tile
multiples, chunks shorter than a tile)."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_util import GuardedOut, device_inputs  # noqa: E402


def _shapes(n=10, seed=2024):
    r = W.splitmix64(seed, 2 * n)
    return [(1 + int(r[2 * i] % np.uint64(300)), int(r[2 * i + 1] % np.uint64(2500))) for i in range(n)]


SHAPES = _shapes()


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


def check(got, ref, what):
    rep = oracle.check(got, ref)
    assert rep["n_bad"] == 0, f"{what}: {rep}"


@pytest.mark.parametrize("C,P", SHAPES)
def test_sweep_all_prefill_paths(cp, C, P):
    inp = W.edge(C, P, seed=C * 131 + P)
    ref = oracle.prefill(inp)
    q, k, v = device_inputs(inp)
    for path in ("attn_prefill", "attn_prefill_bf16x3", "attn_prefill_ffma"):
        g = GuardedOut(C)
        getattr(cp, path)(q, k, v, g.out, P)
        torch.cuda.synchronize()
        assert g.guards_intact(), path
        check(g.numpy(), ref, f"{path} C={C} P={P}")
    # paged
    pg = W.to_pages(inp, seed=C + P)
    g = GuardedOut(C)
    cp.attn_prefill_paged(q, torch.from_numpy(pg.k_pages).cuda(), torch.from_numpy(pg.v_pages).cuda(),
                          torch.from_numpy(pg.table).cuda(), g.out, P)
    torch.cuda.synchronize()
    check(g.numpy(), ref, f"paged C={C} P={P}")
    # bf16 cache
    kv = W.to_bf16(inp)
    g = GuardedOut(C)
    cp.attn_prefill_bf16kv(q, torch.from_numpy(kv.k.view(np.int16)).cuda().view(torch.bfloat16),
                           torch.from_numpy(kv.v.view(np.int16)).cuda().view(torch.bfloat16), g.out, P)
    torch.cuda.synchronize()
    check(g.numpy(), oracle.prefill_bf16kv(inp.q, kv.k, kv.v, P), f"bf16kv C={C} P={P}")
    # score-matrix pipeline (its workspace is 32 C (P + C) floats: at most ~360 MB here)
    ws = torch.empty(cp.attn_naive_workspace_bytes(C, P) // 4, dtype=torch.float32, device="cuda")
    g = GuardedOut(C)
    cp.attn_naive_prefill(q, k, v, g.out, ws, P)
    torch.cuda.synchronize()
    check(g.numpy(), ref, f"naive C={C} P={P}")
    assert cp.attn_get_device_error() == 0


@pytest.mark.parametrize("seed", [5, 6, 7])
def test_sweep_decode_mixes(cp, seed):
    r = W.splitmix64(seed, 24)
    lens = [int(x % np.uint64(5000)) for x in r[:12]]
    batch = W.decode_batch(lens, seed=seed)
    q = torch.from_numpy(batch.q).cuda()
    args = (torch.from_numpy(batch.k_pages).cuda(), torch.from_numpy(batch.v_pages).cuda(),
            torch.from_numpy(batch.table).cuda(), torch.from_numpy(batch.ctx).cuda())
    ref = np.zeros(batch.q.shape)
    for b, T in enumerate(batch.ctx.tolist()):
        if T:
            ref[b] = oracle.attention(batch.q[b:b + 1], oracle.gather_pages(batch.k_pages, batch.table[b], T),
                                      oracle.gather_pages(batch.v_pages, batch.table[b], T), T - 1)[0]
    for splits in (0, 1, 5):
        out = torch.full_like(q, float("nan"))
        nbytes = cp.attn_decode_workspace_bytes(len(lens), batch.max_context, splits)
        ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device="cuda")
        cp.attn_decode_paged(q, *args, out, batch.max_context, splits, ws)
        torch.cuda.synchronize()
        check(out.cpu().numpy(), ref, f"decode seed={seed} splits={splits}")
    assert cp.attn_get_device_error() == 0


def _large_shapes(n=5, seed=77):
    """Chunks of 19 k + m query tiles of 32 rows (m in 1..9, the last tile
    ragged) against 1000..6000 cached keys: on 152 SMs their last round holds
    8 m <= 72 units of at least 1024 keys, so a pair grid splits them."""
    r = W.splitmix64(seed, 4 * n)
    out = []
    for i in range(n):
        tiles = 19 * (1 + int(r[4 * i] % np.uint64(4))) + 1 + int(r[4 * i + 1] % np.uint64(9))
        C = 32 * tiles - int(r[4 * i + 2] % np.uint64(32))
        P = 1000 + int(r[4 * i + 3] % np.uint64(5000))
        out.append((C, P))
    return out


@pytest.mark.parametrize("C,P", _large_shapes())
def test_sweep_large_chunks(cp, C, P):
    """Chunks of several rounds of units, where the whole-unit grid and the
    split-unit pair grid share the work (the pair grid merging its two halves
    through distributed shared memory): every output of the four paths that
    have a pair grid (contiguous and paged split-TF32, bf16x3, bf16 cache)
    against the oracle."""
    inp = W.edge(C, P, seed=C * 7 + P)
    ref = oracle.prefill(inp)
    q, k, v = device_inputs(inp)
    for path in ("attn_prefill", "attn_prefill_bf16x3"):
        g = GuardedOut(C)
        getattr(cp, path)(q, k, v, g.out, P)
        torch.cuda.synchronize()
        assert g.guards_intact(), path
        check(g.numpy(), ref, f"{path} C={C} P={P}")
    pg = W.to_pages(inp, seed=C + 3 * P)
    g = GuardedOut(C)
    cp.attn_prefill_paged(q, torch.from_numpy(pg.k_pages).cuda(), torch.from_numpy(pg.v_pages).cuda(),
                          torch.from_numpy(pg.table).cuda(), g.out, P)
    torch.cuda.synchronize()
    assert g.guards_intact()
    check(g.numpy(), ref, f"paged C={C} P={P}")
    kv = W.to_bf16(inp)
    g = GuardedOut(C)
    cp.attn_prefill_bf16kv(q, torch.from_numpy(kv.k.view(np.int16)).cuda().view(torch.bfloat16),
                           torch.from_numpy(kv.v.view(np.int16)).cuda().view(torch.bfloat16), g.out, P)
    torch.cuda.synchronize()
    assert g.guards_intact()
    check(g.numpy(), oracle.prefill_bf16kv(inp.q, kv.k, kv.v, P), f"bf16kv C={C} P={P}")
    assert cp.attn_get_device_error() == 0
