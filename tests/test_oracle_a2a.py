"""Pins of the oracle's decomposed all-to-all (FlashOverlap technical summary, section
2, "Flash All-to-All": the all-to-all of Ulysses parallelism decomposed into P2P steps):
the ownership routing against block-identity weights, exactness on integer inputs, the
step-order invariants, and message tagging."""
import numpy as np
import pytest

from oracle import ops, schedule
from oracle.ring import RingError


def _ints(rng, shape):
    return rng.integers(-2, 3, shape).astype(np.float64)


@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_producer_routes_every_rank_block_to_its_owner(P):
    # W_r = P stacked identities: block d of rank r's output is X_r itself, so Y_d must
    # hold X_0, X_1, ... in source order
    rng = np.random.default_rng(P)
    m, K = 3, 4
    X = [_ints(rng, (m, K)) for _ in range(P)]
    W = [np.concatenate([np.eye(K)] * P) for _ in range(P)]
    for Y in (ops.gemm_a2a_definition(X, W), ops.gemm_a2a_ring(X, W)[0]):
        for d in range(P):
            assert np.array_equal(Y[d], np.concatenate(X))


@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_consumer_routes_every_source_chunk(P):
    # W_d selects source s's chunk (identity at K block s): Y_d = rows d*m.. of C_s
    rng = np.random.default_rng(10 + P)
    m, Kc = 2, 3
    C = [_ints(rng, (P * m, Kc)) for _ in range(P)]
    for s in range(P):
        W = [np.zeros((Kc, P * Kc)) for _ in range(P)]
        for w in W:
            w[:, s * Kc:(s + 1) * Kc] = np.eye(Kc)
        for Y in (ops.a2a_gemm_definition(C, W), ops.a2a_gemm_ring(C, W)[0]):
            for d in range(P):
                assert np.array_equal(Y[d], C[s][d * m:(d + 1) * m])


@pytest.mark.parametrize("P", [2, 3, 4, 5])
@pytest.mark.parametrize("order", ["flash", "naive"])
def test_decomposed_equals_undecomposed_on_integers(P, order):
    rng = np.random.default_rng(20 + P)
    m, K, Nb, Kc, N = 3, 8, 2, 4, 5
    X = [_ints(rng, (m, K)) for _ in range(P)]
    W = [_ints(rng, (P * Nb, K)) for _ in range(P)]
    a = ops.gemm_a2a_definition(X, W)
    b, _ = ops.gemm_a2a_ring(X, W, order)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    C = [_ints(rng, (P * m, Kc)) for _ in range(P)]
    W2 = [_ints(rng, (N, P * Kc)) for _ in range(P)]
    a = ops.a2a_gemm_definition(C, W2)
    b, _ = ops.a2a_gemm_ring(C, W2, order)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_step_orders(P):
    for r in range(P):
        blocks = [schedule.a2a_block(r, t, P) for t in range(P)]
        sources = [schedule.a2a_source(r, t, P) for t in range(P)]
        assert sorted(blocks) == list(range(P)) and blocks[-1] == r   # own block last
        assert sorted(sources) == list(range(P)) and sources[0] == r  # own chunk first
        for t in range(1, P):  # the chunk folded at step t is the one sent to r at hop t
            assert (schedule.a2a_source(r, t, P) + t) % P == r


def test_logs_follow_the_step_orders():
    P, m, K, Nb = 4, 2, 4, 2
    rng = np.random.default_rng(30)
    X = [_ints(rng, (m, K)) for _ in range(P)]
    W = [_ints(rng, (P * Nb, K)) for _ in range(P)]
    _, log = ops.gemm_a2a_ring(X, W)
    assert all(d == schedule.a2a_block(r, t, P) for r, t, d in log)
    C = [_ints(rng, (P * m, 4)) for _ in range(P)]
    _, log = ops.a2a_gemm_ring(C, [_ints(rng, (3, P * 4)) for _ in range(P)])
    assert all(s == schedule.a2a_source(r, t, P) for r, t, s in log)


def test_dropped_message_is_detected():
    P, m, Kc = 3, 2, 4
    rng = np.random.default_rng(31)
    C = [_ints(rng, (P * m, Kc)) for _ in range(P)]
    W = [_ints(rng, (3, P * Kc)) for _ in range(P)]
    drop_first = {"done": False}

    def fault(src, dst, msg):
        if not drop_first["done"]:
            drop_first["done"] = True
            return []
        return [msg]
    with pytest.raises(RingError):
        ops.a2a_gemm_ring(C, W, fault=fault)
