"""Seeded synthetic inputs for chunked-prefill grouped-query attention.

This module only makes numbers: it holds none of the attention arithmetic.
Both the double-precision oracle (``oracle/``) and the CUDA path receive the
arrays made here, so neither side ever generates its own inputs.

Tensor shapes follow the attention-v1 contract of "Inference Attention 2:
Flash Prefill Against a Cached Prefix" (Lesson): q is [C][32][64], kCache and
vCache are [P + C][8][64], all fp32, row-major.

Generator. Each tensor draws from its own SplitMix64 stream (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014): the
n-th output is mix64(seed + (n + 1) * 0x9E3779B97F4A7C15) with the published
mixing constants. A uniform draw keeps the top 24 bits, so every value in
[-1, 1) is exact in fp32. Normal draws use the Box-Muller transform in double
precision. Seeds follow the teaching program of "FlashAttention and inference
kernels" (A working FlashAttention forward kernel): q, k and v get seeds
s, s + 1 and s + 2; planted positions come from seed s + 3.

Hazards (page 1, Lesson): a planted position t carries 4.0 in every element of
KV head 0 of kCache and vCache, and, when t lies inside the chunk, in query
head 0 of chunk row t - P, so a planted query meets a planted key with score
64 * 16 / 8 = 128.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HQ = 32          # query heads
HKV = 8          # KV heads
D = 64           # head dimension
GROUP = HQ // HKV

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int) -> np.ndarray:
    """The first ``n`` outputs of the SplitMix64 stream started at ``seed``."""
    with np.errstate(over="ignore"):
        idx = np.arange(1, n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform(seed: int, n: int) -> np.ndarray:
    """``n`` fp32 values uniform on [-1, 1), each exactly representable."""
    top24 = (splitmix64(seed, n) >> np.uint64(40)).astype(np.float64)
    return (top24 * (2.0 / (1 << 24)) - 1.0).astype(np.float32)


def normal_clipped(seed: int, n: int, sigma: float = 0.5, clip: float = 2.0) -> np.ndarray:
    """``n`` fp32 values, normal(0, sigma) by Box-Muller, clipped to [-clip, clip]."""
    m = (n + 1) // 2
    raw = splitmix64(seed, 2 * m)
    u1 = ((raw[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / (1 << 53))  # (0, 1]
    u2 = (raw[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))          # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return np.clip(z[:n] * sigma, -clip, clip).astype(np.float32)


def distinct_positions(seed: int, count: int, upper: int) -> np.ndarray:
    """``count`` distinct positions in [0, upper), drawn in order from one stream."""
    if count > upper:
        raise ValueError("more planted positions than positions")
    chosen: list[int] = []
    seen: set[int] = set()
    block = 0
    while len(chosen) < count:
        draws = splitmix64(seed + 0x1000 * block, 4 * count + 16)
        for x in (draws % np.uint64(upper)).tolist():
            if x not in seen:
                seen.add(x)
                chosen.append(int(x))
                if len(chosen) == count:
                    break
        block += 1
    return np.array(sorted(chosen), dtype=np.int64)


@dataclass
class Inputs:
    """One attention call's inputs: q [C][32][64], k/v [P+C][8][64], fp32."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    C: int
    P: int
    planted: np.ndarray = field(default_factory=lambda: np.zeros(0, dtype=np.int64))
    name: str = ""

    @property
    def T(self) -> int:
        return self.P + self.C

    @property
    def pairs(self) -> int:
        """Visible (row, key) pairs: sum over chunk rows i of P + i + 1."""
        return self.C * self.P + self.C * (self.C + 1) // 2


def make_inputs(C: int, P: int, seed: int = 1, dist: str = "uniform",
                planted=None, name: str = "") -> Inputs:
    """Fresh inputs for a chunk of ``C`` rows at offset ``P``.

    ``dist`` is "uniform" (uniform[-1, 1)) or "normal" (normal(0, 0.5) clipped
    to [-2, 2]). ``planted`` is an iterable of positions in [0, P + C).
    """
    if C < 0 or P < 0:
        raise ValueError("C and P must be non-negative")
    T = P + C
    draw = uniform if dist == "uniform" else normal_clipped
    if dist not in ("uniform", "normal"):
        raise ValueError(f"unknown distribution {dist!r}")
    q = draw(seed, C * HQ * D).reshape(C, HQ, D)
    k = draw(seed + 1, T * HKV * D).reshape(T, HKV, D)
    v = draw(seed + 2, T * HKV * D).reshape(T, HKV, D)
    pos = np.array(sorted(set(int(t) for t in (planted if planted is not None else []))), dtype=np.int64)
    plant(q, k, v, P, pos)
    return Inputs(q=q, k=k, v=v, C=C, P=P, planted=pos, name=name)


def plant(q: np.ndarray, k: np.ndarray, v: np.ndarray, P: int, positions) -> None:
    """Write 4.0 into KV head 0 (K and V) at each position, and into query head 0
    of the chunk row at that position when it lies inside the chunk."""
    T = k.shape[0]
    for t in positions:
        t = int(t)
        if not 0 <= t < T:
            raise ValueError(f"planted position {t} outside [0, {T})")
        k[t, 0, :] = 4.0
        v[t, 0, :] = 4.0
        if t >= P:
            q[t - P, 0, :] = 4.0


def ramp(inp: Inputs) -> Inputs:
    """Make every chunk row's largest score sit on its own diagonal key.

    Query head 0 is all ones and key j of KV head 0 is 2 (j + 1) / T in every
    element, so scores rise with j and row i's maximum is key P + i, which lies
    in that row's last K/V tile whatever the tile width.
    """
    T = inp.T
    inp.q[:, 0, :] = 1.0
    inp.k[:, 0, :] = (2.0 * (np.arange(T, dtype=np.float64) + 1.0) / T).astype(np.float32)[:, None]
    return inp


# ---------------------------------------------------------------------------
# The named workloads. Sizes come from the page-1 hazards and the serving
# shapes; the recipe is stated once here and used by tests and bench alike.
# ---------------------------------------------------------------------------

TINY_PLANTED = (0, 13, 31, 39, 47)


def tiny(seed: int = 1) -> Inputs:
    """C=17, P=31, uniform, planted at prefix and chunk positions incl. the last key."""
    return make_inputs(17, 31, seed, "uniform", TINY_PLANTED, name="tiny C=17 P=31")


def edge(C: int, P: int, seed: int = 1, variant: str = "plain") -> Inputs:
    """Tile-edge sweep case; ``variant`` is "plain", "lastkey" or "ramp"."""
    if variant == "plain":
        return make_inputs(C, P, seed, "uniform", name=f"edge C={C} P={P}")
    if variant == "lastkey":
        return make_inputs(C, P, seed, "uniform", [P + C - 1], name=f"edge-lastkey C={C} P={P}")
    if variant == "ramp":
        return ramp(make_inputs(C, P, seed, "uniform", name=f"edge-ramp C={C} P={P}"))
    raise ValueError(variant)


def full_causal(T: int, seed: int = 1) -> Inputs:
    """A whole prompt of T tokens with no cached prefix (P = 0)."""
    return make_inputs(T, 0, seed, "uniform", name=f"full-causal T={T}")


def serve(seed: int = 1, C: int = 2048, P: int = 2048, n_planted: int = 64) -> Inputs:
    """Serving chunk C=2048 against P=2048 cached keys, 64 planted positions."""
    pos = distinct_positions(seed + 3, n_planted, P + C)
    return make_inputs(C, P, seed, "uniform", pos, name=f"serve C={C} P={P}")


def long_prefix(seed: int = 1, C: int = 2048, P: int = 30720) -> Inputs:
    """C=2048 against a 30720-token cached prefix, normal(0, 0.5) clipped to [-2, 2]."""
    return make_inputs(C, P, seed, "normal", name=f"long C={C} P={P}")


SPLIT_TERM_CASES = ("q", "k", "pv")
# The cases for the bf16-piece paths (x = x1 + x2, two bf16 terms, 16
# significant bits together): "q" and "k" as above, and "pv1", the "pv" case
# with value rows of about +1 and -1 instead of +8 and -8 (at |v| = 8 a 16-bit
# split is itself at the tolerance's absolute floor).
BF16_SPLIT_TERM_CASES = ("q", "k", "pv1")


def split_term_case(term: str, seed: int = 11) -> Inputs:
    """Inputs on which each part of an error-compensated split-precision product
    matters: an operand x carried as hi + lo (hi = x with its 13 low mantissa
    bits cleared, tf32) must keep both parts, and these cases are built so that
    dropping the lo part of one operand moves most outputs outside the oracle's
    tolerance while the scores keep a moderate spread.

    "q": q = 1 + u/16 (full 24-bit mantissas), k = +-32 with the signs of dims
    32..63 the negation of dims 0..31, so q.k is small but the lo part of q
    moves every score by about 1e-2. C = P = 64.
    "k": the roles swapped: q = +-32, k = 1 + u/16. C = P = 64.
    "pv": one chunk row at P = 1 against two keys of nearly equal score (key 0
    is key 1 plus u/64) whose value rows are 8 (1 + u/16) and -8 (1 + u'/16):
    the output nearly cancels, so the lo parts of the probabilities and of V
    each show at the scale of |v| = 8.
    "pv1": the same with value rows 1 + u/16 and -(1 + u'/16).
    """
    if term == "q":
        inp = make_inputs(64, 64, seed)
        q = (1.0 + inp.q.astype(np.float64) / 16.0).astype(np.float32)
        sign = np.where(inp.k[:, :, :32] >= 0, 32.0, -32.0)
        k = np.concatenate([sign, -sign], axis=2).astype(np.float32)
        return Inputs(q=q, k=k, v=inp.v, C=64, P=64, name="split-term q")
    if term == "k":
        inp = make_inputs(64, 64, seed)
        q = np.where(inp.q >= 0, 32.0, -32.0).astype(np.float32)
        k = (1.0 + inp.k.astype(np.float64) / 16.0).astype(np.float32)
        return Inputs(q=q, k=k, v=inp.v, C=64, P=64, name="split-term k")
    if term in ("pv", "pv1"):
        scale = 8.0 if term == "pv" else 1.0
        inp = make_inputs(1, 1, seed)
        k = inp.k.copy()
        k[0] = (k[1].astype(np.float64) + uniform(seed + 7, HKV * D).reshape(HKV, D) / 64.0).astype(np.float32)
        v = np.empty_like(inp.v)
        v[0] = (scale * (1.0 + inp.v[0].astype(np.float64) / 16.0)).astype(np.float32)
        v[1] = (-scale * (1.0 + inp.v[1].astype(np.float64) / 16.0)).astype(np.float32)
        return Inputs(q=inp.q, k=k, v=v, C=1, P=1, name=f"split-term {term}")
    raise ValueError(term)


EDGE_C = (1, 17, 33, 64)
EDGE_P = (0, 31, 1000)
FULL_T = (512, 1024, 2048)
FULL_T_SMALL = (1, 17, 33, 257)


PAGE = 16  # tokens per page of a paged cache


@dataclass
class Paged:
    """A paged copy of a cache: k_pages / v_pages [num_pages][16][8][64] and an
    int32 block table; token t is slot t % 16 of physical page table[t // 16]
    ("FlashAttention and inference kernels", PagedAttention)."""
    k_pages: np.ndarray
    v_pages: np.ndarray
    table: np.ndarray


def to_pages(inp: Inputs, seed: int = 7, spare_pages: int = 5) -> Paged:
    """Scatter ``inp``'s K/V into shuffled physical pages.

    Physical pages are a seeded permutation (``spare_pages`` extra pages that no
    token uses are included). Unused pool content -- the spare pages and the
    slots of the last page past P + C - 1 -- is NaN, so a kernel that gives any
    weight to it, or multiplies it by a zero weight, fails.
    """
    T = inp.T
    n_logical = (T + PAGE - 1) // PAGE
    n_pages = n_logical + spare_pages
    perm = np.argsort(uniform(seed, n_pages), kind="stable")
    table = perm[:n_logical].astype(np.int32)
    k_pages = np.full((n_pages, PAGE, HKV, D), np.nan, dtype=np.float32)
    v_pages = np.full((n_pages, PAGE, HKV, D), np.nan, dtype=np.float32)
    t = np.arange(T)
    k_pages[table[t // PAGE], t % PAGE] = inp.k
    v_pages[table[t // PAGE], t % PAGE] = inp.v
    return Paged(k_pages=k_pages, v_pages=v_pages, table=table)


@dataclass
class DecodeBatch:
    """One decode step for B sequences against a paged cache.

    q [B][32][64]; k_pages / v_pages [num_pages][16][8][64] (unused slots and
    spare pages NaN); table int32 [B][max_blocks] (entries past a sequence's
    pages are -1 and must never be read); ctx int32 [B]."""
    q: np.ndarray
    k_pages: np.ndarray
    v_pages: np.ndarray
    table: np.ndarray
    ctx: np.ndarray

    @property
    def max_context(self) -> int:
        return int(self.ctx.max()) if self.ctx.size else 0


def decode_batch(ctx_lens, seed: int = 1, spare_pages: int = 3, planted=()) -> DecodeBatch:
    """Sequences of the given context lengths (the decode teaching program of
    "FlashAttention and inference kernels" uses 1, 17, 1000 and 4096), pages
    shuffled over one pool. ``planted`` = positions t: each sequence with
    ctx > t gets 4.0 in KV head 0 at t, and query head 0 of every sequence is 4.0."""
    ctx = np.asarray(ctx_lens, dtype=np.int32)
    B = ctx.size
    pages_per = (ctx + PAGE - 1) // PAGE
    max_blocks = max(1, int(pages_per.max()) if B else 1)
    n_pages = int(pages_per.sum()) + spare_pages
    perm = np.argsort(uniform(seed + 7, n_pages), kind="stable").astype(np.int32)
    q = uniform(seed, B * HQ * D).reshape(B, HQ, D)
    k_pages = np.full((n_pages, PAGE, HKV, D), np.nan, dtype=np.float32)
    v_pages = np.full((n_pages, PAGE, HKV, D), np.nan, dtype=np.float32)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    nxt = 0
    for b in range(B):
        T = int(ctx[b])
        k = uniform(seed + 1 + 2 * b + 1000, T * HKV * D).reshape(T, HKV, D)
        v = uniform(seed + 2 + 2 * b + 1000, T * HKV * D).reshape(T, HKV, D)
        if planted:
            q[b, 0, :] = 4.0
            for t in planted:
                if t < T:
                    k[t, 0, :] = 4.0
                    v[t, 0, :] = 4.0
        for lp in range(int(pages_per[b])):
            table[b, lp] = perm[nxt]
            nxt += 1
        t = np.arange(T)
        k_pages[table[b, t // PAGE], t % PAGE] = k
        v_pages[table[b, t // PAGE], t % PAGE] = v
    return DecodeBatch(q=q, k_pages=k_pages, v_pages=v_pages, table=table, ctx=ctx)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The bf16 bit patterns of fp32 values by truncation: the upper 16 bits of
    each value (sign, exponent, 7 fraction bits). An encoding of the inputs,
    not part of the method; both sides receive the same bits."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@dataclass
class Bf16KV:
    """A workload's K/V cache as bf16 bit patterns [P + C][8][64] (uint16)."""
    k: np.ndarray
    v: np.ndarray


def to_bf16(inp: Inputs) -> Bf16KV:
    return Bf16KV(k=bf16_bits(inp.k), v=bf16_bits(inp.v))
