"""fp64 causal linear attention and its sequence-parallel form.  TEST
INFRASTRUCTURE ONLY (see the package docstring).

"Effiziente Parallelisierung linearer Aufmerksamkeitssequenzen fuer
skalierbare Sprachmodelle" (a summary of Linear Attention Sequence
Parallelism, LASP) states that LASP exchanges intermediate states between
GPUs point to point in the forward and the backward pass and exploits the
right-product trick of linear attention; it prints no formula.  Readings
taken (the plainest the page supports):

* linear attention: identity feature map, no normalisation, no decay, the
  causal mask of a language model, a score scale:
      o_t = scale * sum_{s <= t} (q_t . k_s) v_s               (left product)
          = scale * q_t . KV_t,  KV_t = sum_{s <= t} k_s^T v_s   (right product)
* the sequence is cut into P contiguous shards (linear attention costs the
  same per row everywhere, so no zigzag is needed); shard r receives
  KV_in(r) = sum of k^T v over the shards before it, point to point from
  shard r-1, adds its own rows' sum and passes it on;
* inside a shard, rows are taken in blocks: a block's output is the masked
  left product within the block plus the right product of its queries with
  the state of everything before the block;
* backward:
      dq_t = scale * sum_{s <= t} (dO_t . v_s) k_s
      dk_s = scale * sum_{t >= s} (dO_t . v_s) q_t
      dv_s = scale * sum_{t >= s} (q_t . k_s) dO_t
  and the state that travels backwards, from later shards to earlier ones,
  is dKV_in(r) = sum of q^T dO over the shards after r.
"""
from __future__ import annotations

import numpy as np

from .attention import _f64


def _row_blocks(n, step=512):
    for r0 in range(0, n, step):
        yield r0, min(n, r0 + step)


def linear_attention(q, k, v, scale):
    """o [..., S, D] of causal linear attention (left product, by row blocks)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead, S = q.shape[:-2], q.shape[-2]
    q2, k2, v2 = (x.reshape(-1, S, x.shape[-1]) for x in (q, k, v))
    o = np.zeros(q2.shape[:2] + (v.shape[-1],))
    for n in range(q2.shape[0]):
        for r0, r1 in _row_blocks(S):
            s = q2[n, r0:r1] @ k2[n, :r1].T
            s *= np.arange(r1)[None, :] <= np.arange(r0, r1)[:, None]   # causal mask
            o[n, r0:r1] = scale * (s @ v2[n, :r1])
    return o.reshape(*lead, S, v.shape[-1])


def linear_attention_backward(q, k, v, do, scale):
    """(dq, dk, dv) of causal linear attention, float64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    lead, S = q.shape[:-2], q.shape[-2]
    q2, k2, v2, do2 = (x.reshape(-1, S, x.shape[-1]) for x in (q, k, v, do))
    dq, dk, dv = np.zeros_like(q2), np.zeros_like(k2), np.zeros_like(v2)
    for n in range(q2.shape[0]):
        for r0, r1 in _row_blocks(S):
            mask = np.arange(r1)[None, :] <= np.arange(r0, r1)[:, None]   # rows t, columns s
            ds = (do2[n, r0:r1] @ v2[n, :r1].T) * mask                     # dO_t . v_s
            ps = (q2[n, r0:r1] @ k2[n, :r1].T) * mask                      # q_t . k_s
            dq[n, r0:r1] = scale * (ds @ k2[n, :r1])
            dk[n, :r1] += scale * (ds.T @ q2[n, r0:r1])
            dv[n, :r1] += scale * (ps.T @ do2[n, r0:r1])
    shape = lambda x: x.reshape(*lead, S, x.shape[-1])
    return shape(dq), shape(dk), shape(dv)


def shard_bounds(S: int, P: int):
    """Row range [a, b) of each of P contiguous shards."""
    if S % P:
        raise ValueError(f"S={S} not divisible into {P} shards")
    n = S // P
    return [(r * n, (r + 1) * n) for r in range(P)]


def lasp_forward(q, k, v, scale, P, block):
    """The sequence-parallel forward, step by step: per shard the local
    state, the point-to-point pass of states from shard to shard, then per
    block of the shard the intra-block left product plus the right product
    with the state before the block.  One head: q, k, v [S, D].  Returns o
    and the state each shard received."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    S, D = q.shape
    bounds = shard_bounds(S, P)
    local = [k[a:b].T @ v[a:b] for a, b in bounds]          # each shard's own sum of k^T v
    received = [np.zeros((D, v.shape[1]))]                  # shard 0 receives nothing
    for r in range(1, P):                                   # the ring of sends r-1 -> r
        received.append(received[r - 1] + local[r - 1])
    o = np.zeros((S, v.shape[1]))
    for r, (a, b) in enumerate(bounds):
        state = received[r].copy()
        for r0 in range(a, b, block):
            r1 = min(b, r0 + block)
            qb, kb, vb = q[r0:r1], k[r0:r1], v[r0:r1]
            intra = np.tril(qb @ kb.T) @ vb
            o[r0:r1] = scale * (qb @ state + intra)
            state = state + kb.T @ vb
    return o, received


def lasp_backward(q, k, v, do, scale, P, block):
    """The sequence-parallel backward: the forward states again for dq, and
    the states of q^T dO passed from later shards to earlier ones for dk and
    dv.  One head.  Returns (dq, dk, dv) and the backward state each shard
    received."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    S, D = q.shape
    bounds = shard_bounds(S, P)
    _, fwd_in = lasp_forward(q, k, v, scale, P, block)
    local = [q[a:b].T @ do[a:b] for a, b in bounds]
    received = [None] * P
    received[P - 1] = np.zeros((D, do.shape[1]))
    for r in range(P - 2, -1, -1):                          # the ring of sends r+1 -> r
        received[r] = received[r + 1] + local[r + 1]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for r, (a, b) in enumerate(bounds):
        state_f = fwd_in[r].copy()                          # k^T v of everything before the block
        starts = list(range(a, b, block))
        for r0 in starts:
            r1 = min(b, r0 + block)
            qb, kb, vb, dob = q[r0:r1], k[r0:r1], v[r0:r1], do[r0:r1]
            dm = np.tril(dob @ vb.T)
            dq[r0:r1] = scale * (dob @ state_f.T + dm @ kb)
            state_f = state_f + kb.T @ vb
        state_b = received[r].copy()                        # q^T dO of everything after the block
        for r0 in reversed(starts):
            r1 = min(b, r0 + block)
            qb, kb, vb, dob = q[r0:r1], k[r0:r1], v[r0:r1], do[r0:r1]
            dm = np.tril(dob @ vb.T)
            pm = np.tril(qb @ kb.T)
            dk[r0:r1] = scale * (vb @ state_b.T + dm.T @ qb)
            dv[r0:r1] = scale * (kb @ state_b + pm.T @ dob)
            state_b = state_b + qb.T @ dob
    return (dq, dk, dv), received


def linear_attention_rows(q, k, v, scale, rows):
    """o of the given query rows of one head [S, D] (left product per row)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    return np.stack([scale * ((k[:t + 1] @ q[t]) @ v[:t + 1]) for t in rows])


def linear_dq_rows(q, k, v, do, scale, rows):
    """dq of the given query rows of one head."""
    k, v, do = _f64(k), _f64(v), _f64(do)
    return np.stack([scale * ((v[:t + 1] @ do[t]) @ k[:t + 1]) for t in rows])


def linear_dkv_rows(q, k, v, do, scale, cols):
    """(dk, dv) of the given key rows of one head (every later query)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dk = np.stack([scale * ((do[s:] @ v[s]) @ q[s:]) for s in cols])
    dv = np.stack([scale * ((q[s:] @ k[s]) @ do[s:]) for s in cols])
    return dk, dv
