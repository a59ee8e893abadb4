"""Pins for the fp64 oracle: brute force, library special cases, closed forms,
invariants and the shard/merge algebra.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
import importlib
oatt = importlib.import_module("oracle.attention")

RNG = np.random.default_rng(1234)


def brute_attention(q, k, v, scale, causal, qpos, kpos):
    """Pure-Python loops, softmax as exp(s)/sum exp(s) (no max shift)."""
    Sq, D = len(q), len(q[0])
    o = [[0.0] * len(v[0]) for _ in range(Sq)]
    lse = [-math.inf] * Sq
    for i in range(Sq):
        scores = {}
        for j in range(len(k)):
            if causal and kpos[j] > qpos[i]:
                continue
            scores[j] = scale * sum(q[i][d] * k[j][d] for d in range(D))
        if not scores:
            continue
        z = sum(math.exp(s) for s in scores.values())
        lse[i] = math.log(z)
        for j, s in scores.items():
            for d in range(len(v[0])):
                o[i][d] += math.exp(s) / z * v[j][d]
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("S,D", [(1, 3), (5, 4), (16, 8), (13, 2)])
def test_forward_brute_force(causal, S, D):
    q, k, v = (RNG.standard_normal((S, D)) for _ in range(3))
    scale = 1 / math.sqrt(D)
    o, lse = oracle.attention(q, k, v, scale, causal=causal)
    ob, lb = brute_attention(q.tolist(), k.tolist(), v.tolist(), scale, causal,
                             list(range(S)), list(range(S)))
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-13)


def test_partial_brute_force_with_positions():
    # a zigzag shard (positions 2,3,12,13 of 16) against another shard's block
    q, k, v = (RNG.standard_normal((4, 6)) for _ in range(3))
    qpos, kpos = [2, 3, 12, 13], [4, 5, 10, 11]
    o, lse = oracle.attention(q, k, v, 0.3, q_pos=qpos, k_pos=kpos)
    ob, lb = brute_attention(q.tolist(), k.tolist(), v.tolist(), 0.3, True, qpos, kpos)
    # rows 2,3 see no key of this block: empty partial
    assert np.all(lse[:2] == -np.inf) and np.all(o[:2] == 0)
    np.testing.assert_allclose(o, ob, atol=1e-13)
    np.testing.assert_array_equal(lse[:2], lb[:2])
    np.testing.assert_allclose(lse[2:], lb[2:], atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_forward_matches_torch_sdpa_fp64(causal):
    B, H, S, D = 2, 3, 300, 16
    q, k, v = (torch.randn(B, H, S, D, dtype=torch.float64) for _ in range(3))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
    o, _ = oracle.attention(q, k, v, 1 / math.sqrt(D), causal=causal)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)


def test_lse_matches_torch_logsumexp():
    S, D = 70, 8
    q, k = torch.randn(S, D, dtype=torch.float64), torch.randn(S, D, dtype=torch.float64)
    s = (q @ k.T) * 0.5
    s = s.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), -math.inf)
    _, lse = oracle.attention(q, k, torch.zeros(S, 2, dtype=torch.float64), 0.5)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=1).numpy(), atol=1e-12)


def test_softmax_rows_sum_to_one():
    S, D = 40, 8
    q, k = RNG.standard_normal((S, D)) * 3, RNG.standard_normal((S, D))
    for causal in (True, False):
        p = oracle.softmax_matrix(q, k, 1 / math.sqrt(D), causal=causal)
        assert np.all(p >= 0)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-13)
        if causal:
            assert np.all(np.triu(p, 1) == 0)


def test_closed_form_q_zero_no_mask():
    S, D = 37, 5
    v = RNG.standard_normal((S, D))
    o, lse = oracle.attention(np.zeros((S, D)), RNG.standard_normal((S, D)), v, 0.7, causal=False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(S), atol=1e-13)


def test_closed_form_q_zero_causal():
    S, D = 37, 5
    v = RNG.standard_normal((S, D))
    o, lse = oracle.attention(np.zeros((S, D)), RNG.standard_normal((S, D)), v, 0.7)
    cum = np.cumsum(v, axis=0) / np.arange(1, S + 1)[:, None]
    np.testing.assert_allclose(o, cum, atol=1e-13)
    np.testing.assert_allclose(lse, np.log(np.arange(1, S + 1)), atol=1e-13)


def test_first_row_sees_only_itself():
    S, D = 9, 4
    q, k, v = (RNG.standard_normal((S, D)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, 0.5)
    assert np.array_equal(o[0], v[0])
    assert lse[0] == 0.5 * (q[0] @ k[0])


def test_key_shift_moves_lse_only():
    S, D = 50, 6
    q, k, v = (RNG.standard_normal((S, D)) for _ in range(3))
    u = RNG.standard_normal(D)
    o1, l1 = oracle.attention(q, k, v, 0.4)
    o2, l2 = oracle.attention(q, k + u, v, 0.4)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 0.4 * (q @ u), atol=1e-12)


def test_row_blocking_is_invisible(monkeypatch):
    S, D = 200, 4
    q, k, v = (RNG.standard_normal((S, D)) for _ in range(3))
    o1, l1 = oracle.attention(q, k, v, 0.5)
    monkeypatch.setattr(oatt, "_SCORE_BUDGET", 7 * S)
    o2, l2 = oracle.attention(q, k, v, 0.5)
    np.testing.assert_allclose(o2, o1, atol=1e-14)
    np.testing.assert_allclose(l2, l1, atol=1e-14)


# ----------------------------------------------------------------- merge ----

@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_sharded_equals_unsharded(layout, P):
    S = 48 if layout == "zigzag" or P != 3 else 48
    B, H, D = 1, 2, 8
    q, k, v = (RNG.standard_normal((B, H, S, D)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, 0.35)
    os_, ls_ = oracle.sharded_attention(q, k, v, 0.35, P, layout)
    np.testing.assert_allclose(os_, o, atol=1e-12)
    np.testing.assert_allclose(ls_, lse, atol=1e-12)


def test_merge_any_visiting_order_and_double_ring():
    S, P, D = 64, 4, 5
    q, k, v = (RNG.standard_normal((S, D)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, 0.5)
    for visit in ("double_ring", [list(RNG.permutation(P)) for _ in range(P)]):
        os_, ls_ = oracle.sharded_attention(q, k, v, 0.5, P, "zigzag", visit=visit, inner=2)
        np.testing.assert_allclose(os_, o, atol=1e-12)
        np.testing.assert_allclose(ls_, lse, atol=1e-12)


# Double ring, P = outer x inner shards, shard r = (group g, place i) with
# r = g*inner + i.  Written out by hand from the reading of the 2D page's
# double ring ("Mejorando la Eficiencia de Comunicacion con la Atencion de
# Doble Anillo"): for `inner` steps the blocks go round the inner ring of
# the group whose blocks are being visited (place i, then i-1, ...); then
# the outer ring moves every shard on to the blocks of the group before it.
DOUBLE_RING_ORDERS = {
    (4, 2): [[0, 1, 2, 3], [1, 0, 3, 2], [2, 3, 0, 1], [3, 2, 1, 0]],
    (8, 4): [[0, 3, 2, 1, 4, 7, 6, 5], [1, 0, 3, 2, 5, 4, 7, 6], [2, 1, 0, 3, 6, 5, 4, 7],
             [3, 2, 1, 0, 7, 6, 5, 4], [4, 7, 6, 5, 0, 3, 2, 1], [5, 4, 7, 6, 1, 0, 3, 2],
             [6, 5, 4, 7, 2, 1, 0, 3], [7, 6, 5, 4, 3, 2, 1, 0]],
    (6, 2): [[0, 1, 4, 5, 2, 3], [1, 0, 5, 4, 3, 2], [2, 3, 0, 1, 4, 5], [3, 2, 1, 0, 5, 4],
             [4, 5, 2, 3, 0, 1], [5, 4, 3, 2, 1, 0]],
}


@pytest.mark.parametrize("P,inner", sorted(DOUBLE_RING_ORDERS))
def test_double_ring_matches_hand_derived_orders(P, inner):
    for r in range(P):
        assert oracle.double_ring_visit_order(P, r, inner) == DOUBLE_RING_ORDERS[(P, inner)][r], r


@pytest.mark.parametrize("P,inner", [(4, 2), (8, 4), (8, 2), (6, 3), (6, 2), (12, 4), (4, 1), (4, 4)])
def test_double_ring_structure(P, inner):
    """The two levels of the order, independently of the literal tables:
    every shard visits every block once, starting with its own; step block
    u*inner + v lies in group (g - u) mod outer; inside that segment the
    place steps down by one each step (the inner ring); at every step the
    blocks held form a one-to-one map, so each hand-off is a permutation in
    which an inner hop moves a block to the next shard of the same group."""
    outer = P // inner
    orders = [oracle.double_ring_visit_order(P, r, inner) for r in range(P)]
    for r, order in enumerate(orders):
        g, i = divmod(r, inner)
        assert sorted(order) == list(range(P)) and order[0] == r
        for u in range(outer):
            seg = order[u * inner:(u + 1) * inner]
            assert all(b // inner == (g - u) % outer for b in seg), (r, u, seg)
            assert [b % inner for b in seg] == [(i - v) % inner for v in range(inner)], (r, u, seg)
    for t in range(P):
        held = [orders[r][t] for r in range(P)]
        assert sorted(held) == list(range(P))
        if t + 1 < P and (t + 1) % inner:                 # inner hop: from the previous place in the group
            for r in range(P):
                sender = held.index(orders[r][t + 1])
                assert sender // inner == r // inner and sender % inner == (r % inner - 1) % inner
    # inner = P is the single ring, inner = 1 the ring over groups of one
    if inner in (1, P):
        assert orders == [oracle.ring_visit_order(P, r) for r in range(P)]


def test_merge_identity_and_permutation():
    n, R, D = 4, 30, 7
    o = RNG.standard_normal((n, R, D))
    lse = RNG.standard_normal((n, R)) * 3
    lse[1, :5] = -np.inf
    mo, ml = oracle.merge_lse(o, lse)
    perm = RNG.permutation(n)
    po, pl = oracle.merge_lse(o[perm], lse[perm])
    np.testing.assert_allclose(po, mo, atol=1e-13)
    np.testing.assert_allclose(pl, ml, atol=1e-13)
    # merging with an empty partial is the identity
    eo, el = oracle.merge_lse(np.stack([o[0], np.full((R, D), 9.0)]),
                              np.stack([lse[0], np.full(R, -np.inf)]))
    np.testing.assert_allclose(eo, o[0], atol=1e-15)
    np.testing.assert_allclose(el, lse[0], atol=1e-15)
    # all empty stays empty
    zo, zl = oracle.merge_lse(o[:2], np.full((2, R), -np.inf))
    assert np.all(zo == 0) and np.all(zl == -np.inf)


def test_merge_two_halves_closed_form():
    # two disjoint key halves of one row: merge must give the full softmax
    D = 3
    q, k, v = RNG.standard_normal((1, D)), RNG.standard_normal((10, D)), RNG.standard_normal((10, D))
    o, lse = oracle.attention(q, k, v, 1.0, causal=False)
    a = oracle.attention(q, k[:4], v[:4], 1.0, causal=False)
    b = oracle.attention(q, k[4:], v[4:], 1.0, causal=False)
    mo, ml = oracle.merge_lse(np.stack([a[0], b[0]]), np.stack([a[1], b[1]]))
    np.testing.assert_allclose(mo, o, atol=1e-14)
    np.testing.assert_allclose(ml, lse, atol=1e-14)
    # and lse of the whole is ln(e^lse_a + e^lse_b)
    np.testing.assert_allclose(ml, np.logaddexp(a[1], b[1]), atol=1e-14)


# ---------------------------------------------------------------- zigzag ----

def _golden_chunks():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "zigzag_chunks.txt")
    rows = [list(map(int, l.split())) for l in open(path) if l.strip() and not l.startswith("#")]
    return rows


def test_zigzag_matches_golden_chunk_map():
    rows = _golden_chunks()
    assert len(rows) == 2 + 4 + 8
    for P, r, c0, c1 in rows:
        S = 2 * P * 3
        c = S // (2 * P)
        pos = oracle.shard_positions(S, P, "zigzag")[r]
        np.testing.assert_array_equal(pos[:c] // c, c0)
        np.testing.assert_array_equal(pos[c:] // c, c1)


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_zigzag_permute_roundtrip_is_exact(P):
    S = 2 * P * 5
    x = RNG.standard_normal((2, 3, S, 4))
    order = oracle.zigzag_order(S, P)
    assert sorted(order.tolist()) == list(range(S))
    y = oracle.permute_rows(x, order)
    assert np.array_equal(oracle.permute_rows(y, order, inverse=True), x)
    # shard r's rows are one contiguous slab of 2c rows after the permute
    for r, pos in enumerate(oracle.shard_positions(S, P, "zigzag")):
        assert np.array_equal(y[..., r * S // P:(r + 1) * S // P, :], x[..., pos, :])


@pytest.mark.parametrize("P,c", [(2, 3), (4, 5), (8, 2), (4, 1024)])
def test_zigzag_balances_causal_work(P, c):
    S = 2 * P * c
    pos = oracle.shard_positions(S, P, "zigzag")
    allpos = np.arange(S)
    for r in range(P):
        assert oracle.visible_pairs(pos[r], allpos) == 2 * P * c * c + c
        for t, j in enumerate(oracle.ring_visit_order(P, r)):
            n = oracle.visible_pairs(pos[r], pos[j])
            assert n == (2 * c * c + c if t == 0 else 2 * c * c)


def test_contiguous_is_unbalanced():
    # the reason for zigzag: the last contiguous shard sees far more pairs
    S, P = 64, 4
    pos = oracle.shard_positions(S, P, "contiguous")
    work = [oracle.visible_pairs(p, np.arange(S)) for p in pos]
    assert work[0] < work[-1]


# -------------------------------------------------------------- backward ----

def _loss_grads_fd(q, k, v, do, scale, h=1e-6):
    def loss(q_, k_, v_):
        o, _ = oracle.attention(q_, k_, v_, scale)
        return float((o * do).sum())
    grads = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(base[which])
        for idx in np.ndindex(g.shape):
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            g[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        grads.append(g)
    return grads


def test_backward_finite_differences():
    S, D = 7, 3
    q, k, v, do = (RNG.standard_normal((S, D)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.6)
    fq, fk, fv = _loss_grads_fd(q, k, v, do, 0.6)
    for a, b in ((dq, fq), (dk, fk), (dv, fv)):
        np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-8)


def test_backward_matches_torch_autograd():
    B, H, S, D = 1, 2, 90, 8
    q, k, v, do = (torch.randn(B, H, S, D, dtype=torch.float64) for _ in range(4))
    qq, kk, vv = (x.clone().requires_grad_() for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True)
    o.backward(do)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 1 / math.sqrt(D))
    np.testing.assert_allclose(dq, qq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, kk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, vv.grad.numpy(), atol=1e-11)


def test_backward_invariants():
    S, D = 60, 5
    q, k, v, do = (RNG.standard_normal((S, D)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5)
    # sum_j dS_ij = 0 for every row  =>  sum_j dK_j = 0
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    # rows of P sum to one  =>  sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)
    # the last key is seen only by the last query: dV_last = P_last,last dO_last
    p = oracle.softmax_matrix(q, k, 0.5)
    np.testing.assert_allclose(dv[-1], p[-1, -1] * do[-1], atol=1e-14)


def test_sampled_rows_match_full():
    B, H, S, D = 1, 2, 130, 4
    q, k, v, do = (RNG.standard_normal((B, H, S, D)) for _ in range(4))
    rows = np.sort(np.stack([[RNG.permutation(S)[:17] for _ in range(H)]]), axis=-1)
    o, lse = oracle.attention(q, k, v, 0.5)
    so, sl = oracle.attention_rows(q, k, v, 0.5, rows)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5)
    for h in range(H):
        r = rows[0, h]
        np.testing.assert_allclose(so[0, h], o[0, h][r], atol=1e-13)
        np.testing.assert_allclose(sl[0, h], lse[0, h][r], atol=1e-13)
        sdq = oracle.backward_query_rows(q[0, h], k[0, h], v[0, h], do[0, h],
                                         so[0, h], sl[0, h], 0.5, r)
        np.testing.assert_allclose(sdq, dq[0, h][r], atol=1e-12)
        sdk, sdv = oracle.backward_key_columns(q[0, h], k[0, h], v[0, h], do[0, h],
                                               o[0, h], lse[0, h], 0.5, r)
        np.testing.assert_allclose(sdk, dk[0, h][r], atol=1e-12)
        np.testing.assert_allclose(sdv, dv[0, h][r], atol=1e-12)


@pytest.mark.parametrize("layout,P", [("zigzag", 2), ("zigzag", 4), ("contiguous", 3)])
def test_block_backward_contributions_sum_to_full(layout, P):
    S, D = 48, 5
    q, k, v, do = (RNG.standard_normal((S, D)) for _ in range(4))
    o, lse = oracle.attention(q, k, v, 0.45)
    delta = (do * o).sum(axis=1)
    dq, dk, dv = np.zeros((S, D)), np.zeros((S, D)), np.zeros((S, D))
    pos = oracle.shard_positions(S, P, layout)
    for r in range(P):
        for j in range(P):
            gq, gk, gv = oracle.attention_backward_block(q[pos[r]], k[pos[j]], v[pos[j]], do[pos[r]],
                                                         lse[pos[r]], delta[pos[r]], 0.45,
                                                         q_pos=pos[r], k_pos=pos[j])
            dq[pos[r]] += gq
            dk[pos[j]] += gk
            dv[pos[j]] += gv
    fq, fk, fv = oracle.attention_backward(q, k, v, do, 0.45)
    np.testing.assert_allclose(dq, fq, atol=1e-12)
    np.testing.assert_allclose(dk, fk, atol=1e-12)
    np.testing.assert_allclose(dv, fv, atol=1e-12)


# ---------------------------------------------- grouped-query attention ----

def _rep(x, group):
    """Key/value heads expanded to one per query head (torch's repeat_interleave)."""
    return torch.repeat_interleave(x, group, dim=1)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (6, 1), (8, 2)])
def test_gqa_forward_matches_torch_sdpa_on_repeated_kv(H, Hkv):
    B, S, D = 2, 40, 8
    g = torch.Generator().manual_seed(H * 10 + Hkv)
    q = torch.randn(B, H, S, D, dtype=torch.float64, generator=g)
    k, v = (torch.randn(B, Hkv, S, D, dtype=torch.float64, generator=g) for _ in range(2))
    o, lse = oracle.attention_gqa(q, k, v, 1 / math.sqrt(D))
    kr, vr = _rep(k, H // Hkv), _rep(v, H // Hkv)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kr, vr, is_causal=True)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)
    s = (q @ kr.transpose(-1, -2)) / math.sqrt(D)
    s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


def test_gqa_with_one_query_head_per_group_is_mha():
    B, H, S, D = 1, 3, 30, 4
    q, k, v = (RNG.standard_normal((B, H, S, D)) for _ in range(3))
    o, lse = oracle.attention_gqa(q, k, v, 0.5)
    ro, rl = oracle.attention(q, k, v, 0.5)
    np.testing.assert_array_equal(o, ro)
    np.testing.assert_array_equal(lse, rl)


@pytest.mark.parametrize("H,Hkv", [(4, 2), (6, 3), (4, 1)])
def test_gqa_backward_matches_torch_autograd(H, Hkv):
    # autograd through repeat_interleave sums each key/value head's gradient
    # over the query heads that read it
    B, S, D = 1, 50, 8
    g = torch.Generator().manual_seed(H + Hkv)
    q, do = (torch.randn(B, H, S, D, dtype=torch.float64, generator=g) for _ in range(2))
    k, v = (torch.randn(B, Hkv, S, D, dtype=torch.float64, generator=g) for _ in range(2))
    qq, kk, vv = (x.clone().requires_grad_() for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qq, _rep(kk, H // Hkv), _rep(vv, H // Hkv), is_causal=True)
    o.backward(do)
    dq, dk, dv = oracle.attention_backward_gqa(q, k, v, do, 1 / math.sqrt(D))
    np.testing.assert_allclose(dq, qq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, kk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, vv.grad.numpy(), atol=1e-11)


def test_gqa_backward_finite_differences():
    B, H, Hkv, S, D, h = 1, 4, 2, 5, 2, 1e-6
    q, do = (RNG.standard_normal((B, H, S, D)) for _ in range(2))
    k, v = (RNG.standard_normal((B, Hkv, S, D)) for _ in range(2))
    dq, dk, dv = oracle.attention_backward_gqa(q, k, v, do, 0.7)

    def loss(k_, v_):
        return float((oracle.attention_gqa(q, k_, v_, 0.7)[0] * do).sum())

    for which, ref in ((0, dk), (1, dv)):
        fd = np.zeros_like(k)
        for idx in np.ndindex(fd.shape):
            plus, minus = [k.copy(), v.copy()], [k.copy(), v.copy()]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        np.testing.assert_allclose(ref, fd, rtol=1e-6, atol=1e-8)
