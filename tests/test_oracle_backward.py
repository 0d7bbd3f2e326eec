"""Pins of the oracle's training backward of the two projections (FlashOverlap technical
summary: the title's training setting; section 2's decomposed all-gather and
reduce-scatter serve the backward with their roles swapped).  The gradients are fixed
by torch autograd on the undecomposed fp64 forward (a library routine, independent of
the oracle's formulas) and by exactness of the ring decompositions on integers."""
import numpy as np
import pytest
import torch

from oracle import bf16, ops


def _ints(rng, shape):
    return rng.integers(-2, 3, shape).astype(np.float64)


@pytest.mark.parametrize("P", [1, 2, 3])
def test_column_parallel_backward_matches_autograd(P):
    rng = np.random.default_rng(P)
    m, K, Nr = 3, 5, 4
    X = [_ints(rng, (m, K)) for _ in range(P)]
    W = [_ints(rng, (Nr, K)) for _ in range(P)]
    dY = [_ints(rng, (P * m, Nr)) for _ in range(P)]
    dX, dW = ops.col_linear_backward(X, W, dY)
    xt = torch.tensor(np.concatenate(X), requires_grad=True)
    wt = [torch.tensor(w, requires_grad=True) for w in W]
    ys = [xt @ w.T for w in wt]  # forward: every rank multiplies the gathered X
    torch.autograd.backward(ys, [torch.tensor(d) for d in dY])
    gx = xt.grad.numpy()
    for d in range(P):
        assert np.array_equal(dX[d], bf16.round_f64(gx[d * m:(d + 1) * m]))
    for r in range(P):
        assert np.array_equal(dW[r], bf16.round_f64(wt[r].grad.numpy()))


@pytest.mark.parametrize("P", [1, 2, 3])
def test_row_parallel_backward_matches_autograd(P):
    rng = np.random.default_rng(10 + P)
    m, Fr, N = 2, 4, 6
    H = [_ints(rng, (P * m, Fr)) for _ in range(P)]
    W = [_ints(rng, (N, Fr)) for _ in range(P)]
    dZ = [_ints(rng, (m, N)) for _ in range(P)]
    dH, dW = ops.row_linear_backward(H, W, dZ)
    ht = [torch.tensor(h, requires_grad=True) for h in H]
    wt = [torch.tensor(w, requires_grad=True) for w in W]
    z = sum(h @ w.T for h, w in zip(ht, wt))  # forward before the scatter: rows d*m.. go to rank d
    torch.autograd.backward([z], [torch.tensor(np.concatenate(dZ))])
    for r in range(P):
        assert np.array_equal(dH[r], bf16.round_f64(ht[r].grad.numpy()))
        assert np.array_equal(dW[r], bf16.round_f64(wt[r].grad.numpy()))


def test_ring_decompositions_equal_the_definitions_on_integers():
    rng = np.random.default_rng(30)
    P, m, K, Nr, Fr, N = 4, 2, 8, 4, 6, 4
    X = [_ints(rng, (m, K)) for _ in range(P)]
    W = [_ints(rng, (Nr, K)) for _ in range(P)]
    dY = [_ints(rng, (P * m, Nr)) for _ in range(P)]
    a, b = ops.col_linear_backward(X, W, dY), ops.col_linear_backward(X, W, dY, decomposed=False)
    assert all(np.array_equal(u, v) for x, y in zip(a, b) for u, v in zip(x, y))
    H = [_ints(rng, (P * m, Fr)) for _ in range(P)]
    W2 = [_ints(rng, (N, Fr)) for _ in range(P)]
    dZ = [_ints(rng, (m, N)) for _ in range(P)]
    a, b = ops.row_linear_backward(H, W2, dZ), ops.row_linear_backward(H, W2, dZ, decomposed=False)
    assert all(np.array_equal(u, v) for x, y in zip(a, b) for u, v in zip(x, y))
