"""A host-side model of the tiled online-softmax update the kernels run.

Test infrastructure. It is not the oracle (the oracle is two-pass and never
tiles); it replays, in float64 Python, the per-tile update of "Inference
Attention 2: Flash Prefill Against a Cached Prefix" (Lesson): for each tile
with maximum m_tile, m_new = max(m_old, m_tile), alpha = exp(m_old - m_new),
l = alpha * l + sum exp(s_j - m_new), acc = alpha * acc + sum exp(s_j - m_new) V_j,
and one division by l at the very end. A tile whose scores are all -inf leaves
m at -inf and computes no alpha ("FlashAttention and inference kernels", the
three places to read in the teaching kernel).

Two optional behaviours match what the tensor-core kernel does and are checked
here to be exact reorderings of the same arithmetic:
- ``stale_threshold``: keep the old maximum while the tile maximum exceeds it by
  at most this amount; l and acc keep sharing one reference maximum, so acc / l
  is unchanged.
"""
from __future__ import annotations

import math


def online_rows(scores, values, tile, stale_threshold=None, trace=None):
    """Run the tile update over one row.

    scores: list of floats (already scaled; -inf for masked keys)
    values: list of vectors (lists) of equal length
    tile:   keys per tile
    Returns acc / l as a list. If ``trace`` is a list, (m, l, acc) after each
    tile is appended to it.
    """
    d = len(values[0])
    m = -math.inf
    l = 0.0
    acc = [0.0] * d
    for t0 in range(0, len(scores), tile):
        s = scores[t0:t0 + tile]
        vs = values[t0:t0 + tile]
        m_tile = max(s)
        m_new = max(m, m_tile)
        if m_new == -math.inf:          # the whole tile masked and nothing seen yet
            if trace is not None:
                trace.append((m, l, list(acc)))
            continue
        if stale_threshold is not None and m != -math.inf and m_new - m <= stale_threshold:
            m_new = m                    # keep the stale reference maximum
        alpha = 0.0 if m == -math.inf else math.exp(m - m_new)
        p = [0.0 if x == -math.inf else math.exp(x - m_new) for x in s]
        l = alpha * l + sum(p)
        acc = [alpha * a + sum(pj * vj[c] for pj, vj in zip(p, vs)) for c, a in enumerate(acc)]
        m = m_new
        if trace is not None:
            trace.append((m, l, list(acc)))
    return [a / l for a in acc]
