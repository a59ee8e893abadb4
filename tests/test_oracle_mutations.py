"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch each one.  Each mutation swaps one internal step for a wrong variant."""
import importlib

import numpy as np
import pytest

import oracle
import tests.test_oracle_pins as pins

oatt = importlib.import_module("oracle.attention")
oshd = importlib.import_module("oracle.shards")


def _scores_exclusive(qb, k, scale, qp, kp, causal):
    s = scale * (qb @ k.T)
    if causal:
        s = np.where(kp[None, :] < qp[:, None], s, -np.inf)
    return s, len(kp)


def _scores_unscaled(qb, k, scale, qp, kp, causal):
    s = qb @ k.T
    if causal:
        s = np.where(kp[None, :] <= qp[:, None], s, -np.inf)
    return s, len(kp)


def _lse_without_max(s):
    m = s.max(axis=1)
    m0 = np.where(m == -np.inf, 0.0, m)
    with np.errstate(divide="ignore"):
        return np.log(np.exp(s - m0[:, None]).sum(axis=1))


def _merge_no_normalise(o_parts, lse_parts):
    o_parts, lse_parts = np.asarray(o_parts, float), np.asarray(lse_parts, float)
    M = lse_parts.max(axis=0)
    w = np.exp(lse_parts - M[None])
    return (w[..., None] * o_parts).sum(axis=0), M + np.log(w.sum(axis=0))


def _zigzag_off_by_one(S, P):
    c = S // (2 * P)
    parts = []
    for r in range(P):
        parts.append(np.arange(r * c, (r + 1) * c))
        parts.append(np.arange(((2 * P - 2 - r) % (2 * P)) * c, ((2 * P - 2 - r) % (2 * P) + 1) * c))
    return np.concatenate(parts)


def _backward_transposed(q, k, v, do, scale, causal=True, o=None, lse=None):
    dq, dk, dv = _orig_backward(q, k, v, do, scale, causal, o, lse)
    # classic slip: dK built from dS instead of dS^T (i.e. query-indexed)
    q64, k64 = oatt._f64(q), oatt._f64(k)
    p = oracle.softmax_matrix(q64, k64, scale) if q64.ndim == 2 else None
    if p is None:
        return dq, dk, dv
    v64, do64 = oatt._f64(v), oatt._f64(do)
    o_, _ = oracle.attention(q64, k64, v64, scale)
    ds = p * (do64 @ v64.T - (do64 * o_).sum(1)[:, None])
    return dq, scale * (ds @ q64), dv


def _backward_no_delta(q, k, v, do, scale, causal=True, o=None, lse=None):
    dq, dk, dv = _orig_backward(q, k, v, do, scale, causal, o, lse)
    q64, k64, v64, do64 = map(oatt._f64, (q, k, v, do))
    if q64.ndim != 2:
        return dq, dk, dv
    p = oracle.softmax_matrix(q64, k64, scale)
    ds = p * (do64 @ v64.T)
    return scale * ds @ k64, scale * ds.T @ q64, dv


_orig_backward = oatt.attention_backward


def _double_ring_outer_first(P, r, inner):
    # slip: the loops swapped, the outer ring turning fastest
    outer = P // inner
    g, i = divmod(r, inner)
    return [((g - u) % outer) * inner + ((i - v) % inner) for v in range(inner) for u in range(outer)]


def _double_ring_inner_up(P, r, inner):
    # slip: the inner ring turning the other way (place i + v)
    outer = P // inner
    g, i = divmod(r, inner)
    return [((g - u) % outer) * inner + ((i + v) % inner) for u in range(outer) for v in range(inner)]


def _kv_head_interleaved(h, n_heads, n_kv_heads):
    # wrong grouping: query heads dealt round-robin over the key/value heads
    return h % n_kv_heads


def _backward_gqa_last_head_wins(q, k, v, do, scale, causal=True, o=None, lse=None):
    # slip: the key/value gradient of a group is overwritten, not summed
    q, k, v, do = map(oatt._f64, (q, k, v, do))
    B, H = q.shape[:2]
    Hkv = k.shape[1]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hkv)
            dq[b, h], dk[b, hk], dv[b, hk] = oatt.attention_backward(q[b, h], k[b, hk], v[b, hk], do[b, h], scale)
    return dq, dk, dv

FORWARD_PINS = [pins.test_first_row_sees_only_itself, pins.test_closed_form_q_zero_causal,
                pins.test_softmax_rows_sum_to_one, pins.test_lse_matches_torch_logsumexp,
                lambda: pins.test_forward_matches_torch_sdpa_fp64(True),
                lambda: pins.test_forward_brute_force(True, 16, 8)]
MERGE_PINS = [pins.test_merge_two_halves_closed_form,
              lambda: pins.test_sharded_equals_unsharded("zigzag", 4)]
ZIGZAG_PINS = [pins.test_zigzag_matches_golden_chunk_map,
               lambda: pins.test_zigzag_balances_causal_work(4, 5)]
DOUBLE_RING_PINS = [lambda: pins.test_double_ring_matches_hand_derived_orders(8, 4),
                    lambda: pins.test_double_ring_structure(8, 2)]
BACKWARD_PINS = [pins.test_backward_finite_differences, pins.test_backward_invariants]
GQA_PINS = [lambda: pins.test_gqa_forward_matches_torch_sdpa_on_repeated_kv(4, 2),
            lambda: pins.test_gqa_backward_matches_torch_autograd(4, 2), pins.test_gqa_backward_finite_differences]


def _some_pin_fails(pin_list):
    for pin in pin_list:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            return True
    return False


@pytest.mark.parametrize("target,attr,bad,pin_list", [
    ("att", "_scores", _scores_exclusive, FORWARD_PINS),
    ("att", "_scores", _scores_unscaled, FORWARD_PINS),
    ("att", "_lse_rows", _lse_without_max, FORWARD_PINS),
    ("shd", "merge_lse", _merge_no_normalise, MERGE_PINS),
    ("shd", "zigzag_order", _zigzag_off_by_one, ZIGZAG_PINS),
])
def test_planted_forward_mistake_is_caught(monkeypatch, target, attr, bad, pin_list):
    mod = oatt if target == "att" else oshd
    monkeypatch.setattr(mod, attr, bad)
    if attr == "merge_lse":
        monkeypatch.setattr(oracle, "merge_lse", bad)
    assert _some_pin_fails(pin_list), f"no pin caught mutation {bad.__name__}"


@pytest.mark.parametrize("bad", [_backward_transposed, _backward_no_delta])
def test_planted_backward_mistake_is_caught(monkeypatch, bad):
    monkeypatch.setattr(oatt, "attention_backward", bad)
    monkeypatch.setattr(oracle, "attention_backward", bad)
    assert _some_pin_fails(BACKWARD_PINS), f"no pin caught mutation {bad.__name__}"


def test_planted_gqa_grouping_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "kv_head_of", _kv_head_interleaved)
    assert _some_pin_fails(GQA_PINS[:1]), "no pin caught the interleaved grouping"


def test_planted_gqa_backward_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(oatt, "attention_backward_gqa", _backward_gqa_last_head_wins)
    monkeypatch.setattr(oracle, "attention_backward_gqa", _backward_gqa_last_head_wins)
    assert _some_pin_fails(GQA_PINS[1:]), "no pin caught the unsummed key/value gradient"


@pytest.mark.parametrize("bad", [_double_ring_outer_first, _double_ring_inner_up])
def test_planted_double_ring_mistake_is_caught(monkeypatch, bad):
    monkeypatch.setattr(oshd, "double_ring_visit_order", bad)
    monkeypatch.setattr(oracle, "double_ring_visit_order", bad)
    assert _some_pin_fails(DOUBLE_RING_PINS), f"no pin caught mutation {bad.__name__}"


def test_unmutated_oracle_passes_every_listed_pin():
    for lst in (FORWARD_PINS, MERGE_PINS, ZIGZAG_PINS, BACKWARD_PINS, GQA_PINS, DOUBLE_RING_PINS):
        assert not _some_pin_fails(lst)
