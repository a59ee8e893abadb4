"""fp64 causal softmax attention, its (o, lse) partials, their merge and the
backward pass.  TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition written out (the METP abstract's unit O = f(A B) C with A B = Q K^T,
f = causal row softmax of the scaled scores, C = V):

    s_ij  = scale * q_i . k_j     if pos(k_j) <= pos(q_i)   else -inf
    m_i   = max_j s_ij
    lse_i = m_i + ln sum_j exp(s_ij - m_i)          (natural log)
    P_ij  = exp(s_ij - lse_i)
    O_i   = sum_j P_ij v_j

A row with no visible key is the empty partial: O_i = 0, lse_i = -inf.  A
partial over a key subset is the same formula with j restricted to it.

Backward (textbook, P recomputed from the saved lse):

    Delta_i = dO_i . O_i
    dP_ij = dO_i . v_j
    dS_ij = P_ij (dP_ij - Delta_i)
    dQ_i  = scale sum_j dS_ij k_j
    dK_j  = scale sum_i dS_ij q_i
    dV_j  = sum_i P_ij dO_i

Rows are processed in blocks only to bound memory; keys a block cannot see
(position above the block's last query position) are left out because their
exp(-inf) terms are exactly zero.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf
_SCORE_BUDGET = 1 << 23     # fp64 score elements held at once (64 MB)


def _f64(x) -> np.ndarray:
    """Convert a torch tensor (any dtype, e.g. bf16) or array to float64."""
    if hasattr(x, "detach"):
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _positions(pos, n):
    return np.arange(n, dtype=np.int64) if pos is None else np.asarray(pos, dtype=np.int64)


def _row_blocks(n_rows, n_keys):
    step = max(1, min(512, _SCORE_BUDGET // max(1, n_keys)))
    for r0 in range(0, n_rows, step):
        yield r0, min(n_rows, r0 + step)


def _scores(qb, k, scale, qp, kp, causal):
    """s = scale q k^T with invisible pairs at -inf; returns (s, key slice end)."""
    if causal:
        # keys beyond the last visible position contribute exp(-inf) = 0
        kend = int(np.searchsorted(kp, qp.max(), side="right")) if np.all(np.diff(kp) >= 0) else len(kp)
    else:
        kend = len(kp)
    s = scale * (qb @ k[:kend].T)
    if causal:
        s = np.where(kp[None, :kend] <= qp[:, None], s, NEG_INF)
    return s, kend


def _lse_rows(s):
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], NEG_INF)
    empty = m == NEG_INF
    m0 = np.where(empty, 0.0, m)
    with np.errstate(divide="ignore"):
        lse = m0 + np.log(np.exp(s - m0[:, None]).sum(axis=1))
    return np.where(empty, NEG_INF, lse)


def _probs(s, lse):
    empty = lse == NEG_INF
    lse0 = np.where(empty, 0.0, lse)
    p = np.exp(s - lse0[:, None])
    p[empty] = 0.0
    return p


def _attention_2d(q, k, v, scale, causal, qp, kp):
    Sq, D = q.shape
    o = np.zeros((Sq, v.shape[1]))
    lse = np.full(Sq, NEG_INF)
    for r0, r1 in _row_blocks(Sq, k.shape[0]):
        s, kend = _scores(q[r0:r1], k, scale, qp[r0:r1], kp, causal)
        lse[r0:r1] = _lse_rows(s)
        p = _probs(s, lse[r0:r1])
        o[r0:r1] = p @ v[:kend]
    return o, lse


def attention(q, k, v, scale, causal=True, q_pos=None, k_pos=None):
    """(o, lse) of causal softmax attention, float64.

    q: [..., Sq, D]; k, v: [..., Sk, D] (same leading dims).  q_pos / k_pos
    give each row's global sequence position (default 0..n-1); a key is
    visible to a query iff its position is <= the query's.  With a key
    subset this is the (o, lse) partial of that block.  Returns
    o [..., Sq, D] and lse [..., Sq]; rows with no visible key give o = 0,
    lse = -inf.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead = q.shape[:-2]
    Sq, Sk = q.shape[-2], k.shape[-2]
    qp, kp = _positions(q_pos, Sq), _positions(k_pos, Sk)
    q2 = q.reshape(-1, Sq, q.shape[-1])
    k2 = k.reshape(-1, Sk, k.shape[-1])
    v2 = v.reshape(-1, Sk, v.shape[-1])
    o = np.zeros((q2.shape[0], Sq, v.shape[-1]))
    lse = np.full((q2.shape[0], Sq), NEG_INF)
    for n in range(q2.shape[0]):
        o[n], lse[n] = _attention_2d(q2[n], k2[n], v2[n], scale, causal, qp, kp)
    return o.reshape(*lead, Sq, v.shape[-1]), lse.reshape(*lead, Sq)


def softmax_matrix(q, k, scale, causal=True, q_pos=None, k_pos=None):
    """The full P matrix [Sq, Sk] of one head (small cases only)."""
    q, k = _f64(q), _f64(k)
    qp, kp = _positions(q_pos, q.shape[0]), _positions(k_pos, k.shape[0])
    s = scale * (q @ k.T)
    if causal:
        s = np.where(kp[None, :] <= qp[:, None], s, NEG_INF)
    return _probs(s, _lse_rows(s))


def attention_rows(q, k, v, scale, rows, causal=True):
    """(o, lse) of the query rows ``rows`` [B,H,n] of full-sequence attention.

    q, k, v: [B,H,S,D] in natural order; each sampled row attends to its own
    visible prefix.  Returns o [B,H,n,D], lse [B,H,n].
    """
    rows = np.asarray(rows)
    B, H, n = rows.shape
    D = q.shape[-1]
    o = np.zeros((B, H, n, D))
    lse = np.zeros((B, H, n))
    for b in range(B):
        for h in range(H):
            r = rows[b, h]
            o[b, h], lse[b, h] = attention(q[b, h][r], k[b, h], v[b, h], scale,
                                           causal=causal, q_pos=r)
    return o, lse


def merge_lse(o_parts, lse_parts):
    """Exact merge of n (o, lse) partials of the same rows.

    o_parts [n, ..., D], lse_parts [n, ...].  With M = max_i lse_i,
    w_i = exp(lse_i - M): lse = M + ln sum_i w_i, o = sum_i w_i o_i / sum_i w_i.
    Rows whose partials are all empty (lse = -inf) stay empty: o = 0, lse = -inf.
    """
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    M = lse_parts.max(axis=0)
    empty = M == NEG_INF
    M0 = np.where(empty, 0.0, M)
    w = np.exp(lse_parts - M0[None])
    wsum = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(empty, NEG_INF, M0 + np.log(wsum))
        o = (w[..., None] * o_parts).sum(axis=0) / np.where(empty, 1.0, wsum)[..., None]
    o[empty] = 0.0
    return o, lse


def attention_backward(q, k, v, do, scale, causal=True, o=None, lse=None):
    """(dq, dk, dv) of causal attention for [..., S, D] inputs, float64.

    P is recomputed from the lse of the forward (computed here if not given).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    if o is None or lse is None:
        o, lse = attention(q, k, v, scale, causal=causal)
    o, lse = _f64(o), _f64(lse)
    lead = q.shape[:-2]
    S, D = q.shape[-2], q.shape[-1]
    flat = lambda x, d: x.reshape(-1, S, d) if d else x.reshape(-1, S)
    q2, k2, v2, do2, o2, l2 = flat(q, D), flat(k, D), flat(v, D), flat(do, D), flat(o, D), flat(lse, 0)
    dq = np.zeros_like(q2)
    dk = np.zeros_like(k2)
    dv = np.zeros_like(v2)
    pos = np.arange(S)
    for n in range(q2.shape[0]):
        delta = (do2[n] * o2[n]).sum(axis=1)
        for r0, r1 in _row_blocks(S, S):
            qb = q2[n, r0:r1]
            s, kend = _scores(qb, k2[n], scale, pos[r0:r1], pos, causal)
            p = _probs(s, l2[n, r0:r1])
            dp = do2[n, r0:r1] @ v2[n, :kend].T
            ds = p * (dp - delta[r0:r1, None])
            dq[n, r0:r1] = scale * (ds @ k2[n, :kend])
            dk[n, :kend] += scale * (ds.T @ qb)
            dv[n, :kend] += p.T @ do2[n, r0:r1]
    return dq.reshape(*lead, S, D), dk.reshape(*lead, S, D), dv.reshape(*lead, S, D)


def backward_query_rows(q, k, v, do, o_rows, lse_rows, scale, rows):
    """dQ of sampled query rows of one head.

    q, k, v, do: [S, D] of one head (natural order); o_rows / lse_rows: the
    forward output of those rows; rows: sorted positions.  Returns [n, D].
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    rows = np.asarray(rows)
    delta = (do[rows] * _f64(o_rows)).sum(axis=1)
    pos = np.arange(k.shape[0])
    dq = np.zeros((len(rows), q.shape[1]))
    for r0, r1 in _row_blocks(len(rows), k.shape[0]):
        rr = rows[r0:r1]
        s, kend = _scores(q[rr], k, scale, rr, pos, True)
        p = _probs(s, _f64(lse_rows)[r0:r1])
        dp = do[rr] @ v[:kend].T
        ds = p * (dp - delta[r0:r1, None])
        dq[r0:r1] = scale * (ds @ k[:kend])
    return dq


def backward_key_columns(q, k, v, do, o, lse, scale, cols):
    """dK, dV of sampled key rows of one head.

    Needs the forward o [S, D] and lse [S] of every query row of the head
    (every later query sees the key).  Returns (dk [n, D], dv [n, D]).
    """
    q, k, v, do, o, lse = map(_f64, (q, k, v, do, o, lse))
    cols = np.asarray(cols)
    S = q.shape[0]
    delta = (do * o).sum(axis=1)
    dk = np.zeros((len(cols), q.shape[1]))
    dv = np.zeros((len(cols), v.shape[1]))
    for c, j in enumerate(cols):
        i = np.arange(j, S)                       # queries that see key j
        s = scale * (q[i] @ k[j])
        p = np.exp(s - lse[i])
        dp = do[i] @ v[j]
        ds = p * (dp - delta[i])
        dk[c] = scale * (ds @ q[i])
        dv[c] = p @ do[i]
    return dk, dv


def attention_backward_block(q, k, v, do, lse, delta, scale, causal=True, q_pos=None, k_pos=None):
    """Gradient contributions of one (query slab, key block) pair, float64.

    With the FINAL lse_i and delta_i = dO_i . O_i of the query rows (over
    the whole sequence), the pair contributes, over its visible (i, j):
        P_ij = exp(s_ij - lse_i),  dS_ij = P_ij (dO_i . v_j - delta_i)
        dq_i += scale sum_j dS_ij k_j,  dk_j += scale sum_i dS_ij q_i,
        dv_j += sum_i P_ij dO_i
    q, do: [Sq, D]; k, v: [Sk, D] (one head).  Summing the contributions of
    every block of a partition gives the full gradients.
    """
    q, k, v, do, lse, delta = map(_f64, (q, k, v, do, lse, delta))
    qp, kp = _positions(q_pos, q.shape[0]), _positions(k_pos, k.shape[0])
    s = scale * (q @ k.T)
    if causal:
        s = np.where(kp[None, :] <= qp[:, None], s, NEG_INF)
    p = _probs(s, lse)
    ds = p * (do @ v.T - delta[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), p.T @ do


# -------------------------------------------- grouped-query attention ----
#
# "Avances en la capacitacion de LLMs de secuencia larga", section
# "Comprendiendo la Arquitectura de los LLMs": grouped-query attention groups
# the query heads so that each group shares one key/value head (the 7B-GQA
# model of section "Evaluacion y Comparacion con Sistemas Existentes").  The
# page does not say which query heads form a group; the reading here is
# consecutive groups: with H query heads and Hkv key/value heads, query head
# h reads key/value head h // (H / Hkv).

def kv_head_of(h: int, n_heads: int, n_kv_heads: int) -> int:
    """Key/value head that query head h reads."""
    if n_heads % n_kv_heads:
        raise ValueError(f"{n_heads} query heads are not a multiple of {n_kv_heads} key/value heads")
    return h // (n_heads // n_kv_heads)


def attention_gqa(q, k, v, scale, causal=True):
    """(o, lse) of grouped-query causal attention, float64.

    q: [B, H, S, D]; k, v: [B, Hkv, S, D] with H a multiple of Hkv.  Each
    query head is the single-head attention of its rows against the
    key/value head of its group.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, S, _ = q.shape
    Hkv = k.shape[1]
    o = np.zeros(q.shape[:3] + (v.shape[-1],))
    lse = np.zeros(q.shape[:3])
    for b in range(B):
        for h in range(H):
            hk = kv_head_of(h, H, Hkv)
            o[b, h], lse[b, h] = attention(q[b, h], k[b, hk], v[b, hk], scale, causal=causal)
    return o, lse


def attention_backward_gqa(q, k, v, do, scale, causal=True, o=None, lse=None):
    """(dq, dk, dv) of grouped-query causal attention, float64.

    dq per query head; the dk, dv of a key/value head are the sums of the
    single-head gradients of every query head that reads it (the head is
    one input of all of them).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    if o is None or lse is None:
        o, lse = attention_gqa(q, k, v, scale, causal=causal)
    o, lse = _f64(o), _f64(lse)
    B, H = q.shape[:2]
    Hkv = k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            hk = kv_head_of(h, H, Hkv)
            gq, gk, gv = attention_backward(q[b, h], k[b, hk], v[b, hk], do[b, h], scale, causal=causal,
                                            o=o[b, h], lse=lse[b, h])
            dq[b, h] = gq
            dk[b, hk] += gk
            dv[b, hk] += gv
    return dq, dk, dv
