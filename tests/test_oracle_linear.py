"""Pins for the fp64 oracle of causal linear attention and its
sequence-parallel (LASP) form: brute force, the recurrent right-product
form, torch autograd, finite differences, a closed form, and planted
mistakes that the pins catch.  CPU only."""
import importlib
import math

import numpy as np
import pytest
import torch

import oracle

olin = importlib.import_module("oracle.linear")
RNG = np.random.default_rng(99)


def brute(q, k, v, scale):
    S = q.shape[0]
    o = np.zeros((S, v.shape[1]))
    for t in range(S):
        for s in range(t + 1):
            o[t] += scale * float(np.dot(q[t], k[s])) * v[s]
    return o


def recurrent(q, k, v, scale):
    """The right product as a recurrence over the rows: a running k^T v."""
    S, D = q.shape
    state = np.zeros((D, v.shape[1]))
    o = np.zeros((S, v.shape[1]))
    for t in range(S):
        state += np.outer(k[t], v[t])
        o[t] = scale * q[t] @ state
    return o


@pytest.mark.parametrize("S,D", [(1, 3), (9, 4), (17, 6)])
def test_forward_brute_force(S, D):
    q, k, v = (RNG.standard_normal((S, D)) for _ in range(3))
    np.testing.assert_allclose(oracle.linear_attention(q, k, v, 0.7), brute(q, k, v, 0.7), atol=1e-12)


def test_forward_matches_recurrence_and_row_blocking():
    S, D = 1100, 8     # more than two row blocks
    q, k, v = (RNG.standard_normal((S, D)) for _ in range(3))
    np.testing.assert_allclose(oracle.linear_attention(q, k, v, 0.3), recurrent(q, k, v, 0.3), atol=1e-9)


def test_closed_form_prefix_sum():
    # q = k = e_0 and scale 1: every score is 1, so o_t is the prefix sum of v
    S, D = 50, 5
    e0 = np.zeros((S, D))
    e0[:, 0] = 1.0
    v = RNG.standard_normal((S, D))
    np.testing.assert_allclose(oracle.linear_attention(e0, e0, v, 1.0), np.cumsum(v, axis=0), atol=1e-12)


def test_backward_matches_torch_autograd():
    B, H, S, D = 1, 2, 70, 8
    q, k, v, do = (torch.randn(B, H, S, D, dtype=torch.float64) for _ in range(4))
    qq, kk, vv = (x.clone().requires_grad_() for x in (q, k, v))
    scale = 1 / math.sqrt(D)
    o = scale * torch.tril(qq @ kk.transpose(-1, -2)) @ vv
    o.backward(do)
    dq, dk, dv = oracle.linear_attention_backward(q, k, v, do, scale)
    for a, b in ((dq, qq.grad), (dk, kk.grad), (dv, vv.grad)):
        np.testing.assert_allclose(a, b.numpy(), atol=1e-10)


def test_backward_finite_differences():
    S, D, h = 6, 3, 1e-6
    q, k, v, do = (RNG.standard_normal((S, D)) for _ in range(4))
    grads = oracle.linear_attention_backward(q, k, v, do, 0.8)
    base = [q, k, v]
    for which in range(3):
        fd = np.zeros_like(base[which])
        for idx in np.ndindex(fd.shape):
            plus, minus = [x.copy() for x in base], [x.copy() for x in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd[idx] = ((oracle.linear_attention(*plus, 0.8) * do).sum()
                       - (oracle.linear_attention(*minus, 0.8) * do).sum()) / (2 * h)
        np.testing.assert_allclose(grads[which], fd, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("P,block", [(1, 64), (2, 16), (4, 8), (4, 7), (8, 5)])
def test_lasp_forward_equals_direct(P, block):
    S, D = 96, 6
    q, k, v = (RNG.standard_normal((S, D)) for _ in range(3))
    o, received = oracle.lasp_forward(q, k, v, 0.5, P, block)
    np.testing.assert_allclose(o, oracle.linear_attention(q, k, v, 0.5), atol=1e-10)
    # the state shard r receives is the k^T v of every earlier row
    for r, (a, _) in enumerate(oracle.shard_bounds(S, P)):
        np.testing.assert_allclose(received[r], k[:a].T @ v[:a], atol=1e-10)


@pytest.mark.parametrize("P,block", [(1, 32), (2, 16), (4, 5), (3, 8)])
def test_lasp_backward_equals_direct(P, block):
    S, D = 48, 4
    q, k, v, do = (RNG.standard_normal((S, D)) for _ in range(4))
    (dq, dk, dv), received = oracle.lasp_backward(q, k, v, do, 0.6, P, block)
    rq, rk, rv = oracle.linear_attention_backward(q, k, v, do, 0.6)
    for a, b in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(a, b, atol=1e-10)
    for r, (_, b) in enumerate(oracle.shard_bounds(S, P)):
        np.testing.assert_allclose(received[r], q[b:].T @ do[b:], atol=1e-10)


# ------------------------------------------------------ planted mistakes ----

def _lasp_inclusive_state(q, k, v, scale, P, block):
    # slip: a shard receives the state including its own rows
    q, k, v = (np.asarray(x, float) for x in (q, k, v))
    o, received = _orig_forward(q, k, v, scale, P, block)
    bounds = oracle.shard_bounds(q.shape[0], P)
    bad = [k[:b].T @ v[:b] for a, b in bounds]
    o2 = o.copy()
    for r, (a, b) in enumerate(bounds):
        o2[a:b] += scale * q[a:b] @ (bad[r] - received[r])
    return o2, bad


def _linear_strict_mask(q, k, v, scale):
    # slip: the diagonal left out of the causal mask
    q, k, v = (np.asarray(x, float) for x in (q, k, v))
    return scale * np.tril(q @ k.T, -1) @ v


_orig_forward = olin.lasp_forward


def test_planted_lasp_mistakes_are_caught(monkeypatch):
    monkeypatch.setattr(oracle, "lasp_forward", _lasp_inclusive_state)
    with pytest.raises(AssertionError):
        test_lasp_forward_equals_direct(4, 8)
    monkeypatch.undo()
    monkeypatch.setattr(oracle, "linear_attention", _linear_strict_mask)
    with pytest.raises(AssertionError):
        test_forward_brute_force(9, 4)


def test_row_helpers_match_full_functions():
    S, D = 130, 5
    q, k, v, do = (RNG.standard_normal((S, D)) for _ in range(4))
    rows = np.array([0, 1, 63, 64, 129])
    o = oracle.linear_attention(q, k, v, 0.4)
    dq, dk, dv = oracle.linear_attention_backward(q, k, v, do, 0.4)
    np.testing.assert_allclose(oracle.linear_attention_rows(q, k, v, 0.4, rows), o[rows], atol=1e-11)
    np.testing.assert_allclose(oracle.linear_dq_rows(q, k, v, do, 0.4, rows), dq[rows], atol=1e-11)
    rk, rv = oracle.linear_dkv_rows(q, k, v, do, 0.4, rows)
    np.testing.assert_allclose(rk, dk[rows], atol=1e-11)
    np.testing.assert_allclose(rv, dv[rows], atol=1e-11)
