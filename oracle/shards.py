"""Context partitions, visiting orders and the sharded forward, float64.
TEST INFRASTRUCTURE ONLY (see the package docstring).

* Contiguous partition: shard r owns positions [r S/P, (r+1) S/P).
* Zigzag partition (TSP page, "Zyphra presenta el paralelismo de secuencia y
  tensor (TSP)", section "Lo que realmente significa plegar": K/V are
  reordered in zigzag before FlashAttention so that causal work is balanced):
  the sequence is cut into 2P chunks of c = S/(2P) positions; shard r owns
  chunk r followed by chunk 2P-1-r.
* Ring order ("Avances en la capacitacion de LLMs de secuencia larga",
  section "Limitaciones de los Enfoques Existentes": context parallelism
  passes key/value blocks between peers): at step t shard r holds the key
  block of shard (r - t) mod P.
* Double ring (same page, section "Mejorando la Eficiencia de Comunicacion
  con la Atencion de Doble Anillo"): the page names a two-level ring but not
  its layout; the reading here is P = outer x inner shards, an inner ring
  inside each group and an outer ring between groups, so only the visiting
  order changes.
"""
from __future__ import annotations

import numpy as np

from .attention import attention, merge_lse, _f64


def chunk_len(S: int, P: int, layout: str) -> int:
    if layout == "zigzag":
        if S % (2 * P):
            raise ValueError(f"zigzag needs S % 2P == 0 (S={S}, P={P})")
        return S // (2 * P)
    if layout == "contiguous":
        if S % P:
            raise ValueError(f"contiguous needs S % P == 0 (S={S}, P={P})")
        return S // P
    raise ValueError(f"unknown layout {layout!r}")


def zigzag_order(S: int, P: int) -> np.ndarray:
    """order[x] = natural position held at shard-major row x (chunks r, 2P-1-r)."""
    c = chunk_len(S, P, "zigzag")
    parts = []
    for r in range(P):
        parts.append(np.arange(r * c, (r + 1) * c))
        parts.append(np.arange((2 * P - 1 - r) * c, (2 * P - r) * c))
    return np.concatenate(parts)


def contiguous_order(S: int, P: int) -> np.ndarray:
    chunk_len(S, P, "contiguous")
    return np.arange(S)


def shard_order(S: int, P: int, layout: str) -> np.ndarray:
    return zigzag_order(S, P) if layout == "zigzag" else contiguous_order(S, P)


def shard_positions(S: int, P: int, layout: str):
    """List of P arrays: the global positions owned by each shard, in row order."""
    order = shard_order(S, P, layout)
    n = S // P
    return [order[r * n:(r + 1) * n] for r in range(P)]


def permute_rows(x, order, inverse=False):
    """Reorder the sequence axis (-2) of x: y[.., i, :] = x[.., order[i], :];
    the inverse puts row i back at position order[i]."""
    x = np.asarray(x)
    if not inverse:
        return x[..., order, :].copy()
    y = np.empty_like(x)
    y[..., order, :] = x
    return y


def ring_visit_order(P: int, r: int):
    return [(r - t) % P for t in range(P)]


def double_ring_visit_order(P: int, r: int, inner: int):
    if P % inner:
        raise ValueError("inner ring size must divide P")
    outer = P // inner
    g, i = divmod(r, inner)
    return [((g - u) % outer) * inner + ((i - v) % inner)
            for u in range(outer) for v in range(inner)]


def visible_pairs(q_pos, k_pos) -> int:
    """Number of (query, key) pairs with pos(key) <= pos(query)."""
    q_pos = np.asarray(q_pos)
    k_sorted = np.sort(np.asarray(k_pos))
    return int(np.searchsorted(k_sorted, q_pos, side="right").sum())


def sharded_attention(q, k, v, scale, P, layout, visit="ring", inner=None,
                      causal=True, return_partials=False):
    """Causal attention over P context shards, each merged from per-block partials.

    Shard r's queries see every key block j in its visiting order; each
    (shard, block) pair gives an (o, lse) partial over that block's keys at
    their global positions, and the partials are merged by ``merge_lse``.
    Returns (o, lse) in natural row order.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    S = q.shape[-2]
    pos = shard_positions(S, P, layout)
    o = np.zeros(q.shape[:-1] + (v.shape[-1],))
    lse = np.zeros(q.shape[:-1])
    partials = {}
    for r in range(P):
        if visit == "ring":
            order = ring_visit_order(P, r)
        elif visit == "double_ring":
            order = double_ring_visit_order(P, r, inner)
        elif isinstance(visit, (list, tuple)):
            order = visit[r]
        else:
            raise ValueError(visit)
        ops, lps = [], []
        for j in order:
            po, pl = attention(q[..., pos[r], :], k[..., pos[j], :], v[..., pos[j], :],
                               scale, causal=causal, q_pos=pos[r], k_pos=pos[j])
            ops.append(po)
            lps.append(pl)
            partials[(r, j)] = (po, pl)
        mo, ml = merge_lse(np.stack(ops), np.stack(lps))
        o[..., pos[r], :] = mo
        lse[..., pos[r]] = ml
    if return_partials:
        return o, lse, partials
    return o, lse
