"""Pins of the oracle's analytic backward pass.

The pages print no gradient formulas (the notes' "Backward Pass:
Recomputation" only says S and P are recomputed), so the oracle's
gradients are pinned to the derivative itself: central finite differences of
the forward definition in float64, torch's float64 autograd on its own
attention, and identities every exact gradient of softmax attention obeys.
"""

import numpy as np
import pytest

import oracle


def _loss(q, k, v, do, scale, window):
    o, _ = oracle.dense_forward(q, k, v, scale, window)
    return float(np.sum(o * do))


@pytest.mark.parametrize("n,d,window", [(1, 1, 0), (3, 2, 0), (5, 3, 0), (5, 3, 3), (4, 2, 1)])
def test_finite_differences(n, d, window):
    rng = np.random.default_rng(n * 10 + d + window)
    q, k, v, do = (rng.standard_normal((1, 2, n, d)) for _ in range(4))
    scale = 0.7
    grads = oracle.dense_backward(q, k, v, do, scale, window)
    h = 1e-6
    for which, g in zip(range(3), grads):
        base = [q, k, v]
        for idx in np.ndindex(*g.shape):
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd = (_loss(*plus, do, scale, window) - _loss(*minus, do, scale, window)) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, g[idx])


@pytest.mark.parametrize("window", [0, 5])
def test_against_torch_autograd(window):
    torch = pytest.importorskip("torch")
    gen = torch.Generator().manual_seed(21)
    q, k, v, do = (torch.randn(2, 2, 19, 6, generator=gen, dtype=torch.float64) for _ in range(4))
    qs, ks, vs = (x.clone().requires_grad_(True) for x in (q, k, v))
    mask = None
    if window > 0:
        i = torch.arange(19)
        mask = (i[:, None] - i[None, :]).abs() <= (window - 1) // 2
    out = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=0.45)
    out.backward(do)
    dq, dk, dv = oracle.dense_backward(q.numpy(), k.numpy(), v.numpy(), do.numpy(), 0.45, window)
    for mine, ref in ((dq, qs.grad), (dk, ks.grad), (dv, vs.grad)):
        assert np.max(np.abs(mine - ref.numpy())) <= 1e-12


def test_gradient_identities():
    """Identities of the exact gradient, for any inputs:
    * adding one vector to every key leaves each softmax row unchanged, so the
      key gradients sum to zero over the keys;
    * the rows of P sum to one, so the value gradients sum to the sum of dO;
    * with all keys equal every score row is constant, so dQ vanishes."""
    rng = np.random.default_rng(4)
    q, k, v, do = (rng.standard_normal((2, 3, 23, 8)) for _ in range(4))
    for window in (0, 7):
        dq, dk, dv = oracle.dense_backward(q, k, v, do, 0.3, window)
        assert np.max(np.abs(dk.sum(-2))) <= 1e-12
        assert np.max(np.abs(dv.sum(-2) - do.sum(-2))) <= 1e-12
    k_eq = np.broadcast_to(rng.standard_normal(8), k.shape)
    dq, _, _ = oracle.dense_backward(q, k_eq, v, do, 0.3)
    assert np.max(np.abs(dq)) <= 1e-13


def test_mutant_backward_is_caught():
    """Dropping the D term of the softmax Jacobian (a plausible mistake) breaks
    the key-gradient identity; the real oracle satisfies it."""
    rng = np.random.default_rng(5)
    q, k, v, do = (rng.standard_normal((1, 1, 9, 4)) for _ in range(4))
    s = q[0, 0] @ k[0, 0].T * 0.5
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    dp = do[0, 0] @ v[0, 0].T
    dk_bad = 0.5 * (p * dp).T @ q[0, 0]
    assert np.max(np.abs(dk_bad.sum(0))) > 1e-3
    _, dk, _ = oracle.dense_backward(q, k, v, do, 0.5)
    assert np.max(np.abs(dk.sum(-2))) <= 1e-13
