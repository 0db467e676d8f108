"""Pins of the oracle's backward (gradients of the plain definition).

Expected values come from torch fp64 autograd (a library routine), central
finite differences (brute force on tiny inputs) and identities the gradient
formulas imply -- never from the oracle itself.
"""

import math

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(99)


def _loss_grads_torch(q, k, v, do, scale, causal):
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = (q @ k.T) * scale
    if causal:
        s = s.masked_fill(torch.ones(q.shape[0], k.shape[0], dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ v
    (o * torch.tensor(do)).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_autograd(causal):
    n, d = 23, 8
    q, k, v, do = (RNG.standard_normal((n, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, scale, causal)
    tq, tk, tv = _loss_grads_torch(q, k, v, do, scale, causal)
    np.testing.assert_allclose(dq, tq, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_central_finite_differences(causal):
    n, d = 3, 2
    q, k, v, do = (RNG.standard_normal((n, d)) for _ in range(4))
    scale = 0.7

    def loss(qq, kk, vv):
        o, _ = oracle.attention_head(qq, kk, vv, scale, causal)
        return float((o * do).sum())

    grads = oracle.attention_backward_head(q, k, v, do, scale, causal)
    eps = 1e-6
    for which, g in zip(range(3), grads):
        for idx in np.ndindex(n, d):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += eps
            args_m[which][idx] -= eps
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert g[idx] == pytest.approx(fd, rel=1e-6, abs=1e-8)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_identities(causal):
    n, d = 17, 6
    q, k, v, do = (RNG.standard_normal((n, d)) for _ in range(4))
    scale = 0.4
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, scale, causal)
    # every row of P sums to 1, so the rows of dV = P^T dO sum to the rows of dO
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), rtol=1e-12, atol=1e-12)
    # every row of dS sums to 0, so dK summed over keys is 0 (sum_j dS_ij = 0 for each i)
    np.testing.assert_allclose(dk.sum(axis=0), np.zeros(d), atol=1e-12)
    # D_i = rowsum(O_i * dO_i) equals rowsum(P_i * dP_i)
    o, _ = oracle.attention_head(q, k, v, scale, causal)
    s = scale * q @ k.T
    if causal:
        s = np.where(np.arange(n)[None, :] > np.arange(n)[:, None], -np.inf, s)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(oracle.backward_delta(o, do), ((do @ v.T) * p).sum(axis=1), rtol=1e-12, atol=1e-12)


def test_uniform_attention_value_gradient():
    """Q = 0: P = 1/N everywhere (non-causal), so dV_j = mean over rows of dO and dQ, dK from dS = 0."""
    n, d = 9, 4
    q = np.zeros((n, d))
    k, v, do = (RNG.standard_normal((n, d)) for _ in range(3))
    dq, dk, dv = oracle.attention_backward_head(q, k, v, do, 0.5, False)
    np.testing.assert_allclose(dv, np.tile(do.sum(axis=0) / n, (n, 1)), rtol=1e-12)
    np.testing.assert_allclose(dk, np.zeros_like(dk), atol=1e-14)


def test_batched_wrapper():
    q, k, v, do = (RNG.standard_normal((2, 3, 5, 4)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.3, True)
    dq1, dk1, dv1 = oracle.attention_backward_head(q[1, 2], k[1, 2], v[1, 2], do[1, 2], 0.3, True)
    np.testing.assert_allclose(dq[1, 2], dq1)
    np.testing.assert_allclose(dk[1, 2], dk1)
    np.testing.assert_allclose(dv[1, 2], dv1)


@pytest.mark.parametrize("causal", [False, True])
def test_row_restricted_gradients_match_torch_autograd(causal):
    """attention_backward_rows at seeded query and key rows equals torch fp64 autograd's full
    gradients at those rows; with a block smaller than N the row statistics span several blocks."""
    n, d = 53, 8
    q, k, v, do = (RNG.standard_normal((n, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    tq, tk, tv = _loss_grads_torch(q, k, v, do, scale, causal)
    qr = np.array([0, 1, 17, 30, 52])
    kr = np.array([0, 5, 26, 51, 52])
    for block in (7, 512):
        dq, dk, dv = oracle.attention_backward_rows(q, k, v, do, scale, causal, q_rows=qr, k_rows=kr, block=block)
        np.testing.assert_allclose(dq, tq[qr], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dk, tk[kr], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dv, tv[kr], rtol=1e-11, atol=1e-12)


def test_row_restricted_last_key_closed_form():
    """Causal, last key j = N-1: only row N-1 attends it, so dV_j = P_{N-1,j} dO_{N-1} and
    dK_j = scale * dS_{N-1,j} q_{N-1} (a closed form from one explicit softmax row)."""
    n, d = 12, 4
    q, k, v, do = (RNG.standard_normal((n, d)) for _ in range(4))
    scale = 0.6
    s = scale * q[-1] @ k.T
    p = np.exp(s - s.max())
    p /= p.sum()
    dp = v @ do[-1]
    ds = p * (dp - (p * dp).sum())
    _, dk, dv = oracle.attention_backward_rows(q, k, v, do, scale, True, k_rows=[n - 1])
    np.testing.assert_allclose(dv[0], p[-1] * do[-1], rtol=1e-12)
    np.testing.assert_allclose(dk[0], scale * ds[-1] * q[-1], rtol=1e-12, atol=1e-14)
