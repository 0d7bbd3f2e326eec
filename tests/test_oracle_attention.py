"""Pins of the oracle's attention (FlashOverlap technical summary, section 2,
"Query Split Attention"): closed forms, scalar brute force, and the ring
decomposition against the two-pass definition."""
import math

import numpy as np
import pytest

from oracle import ops


def _brute_attention(Q, K, V, causal=True):
    """Scalar-loop softmax attention with math.exp (independent of numpy matmul)."""
    S, H, D = K.shape
    out = np.zeros((Q.shape[0], H, D))
    for h in range(H):
        for i in range(Q.shape[0]):
            keys = [j for j in range(S) if not (causal and j > i)]
            sc = [sum(Q[i, h, d] * K[j, h, d] for d in range(D)) / math.sqrt(D) for j in keys]
            mx = max(sc)
            w = [math.exp(s - mx) for s in sc]
            tot = sum(w)
            for d in range(D):
                out[i, h, d] = sum(wj * V[j, h, d] for wj, j in zip(w, keys)) / tot
    return out


@pytest.mark.parametrize("causal", [True, False])
def test_definition_matches_scalar_brute_force(causal):
    rng = np.random.default_rng(1)
    Q, K, V = (rng.standard_normal((6, 2, 4)) for _ in range(3))
    assert np.allclose(ops.attention_definition(Q, K, V, causal), _brute_attention(Q, K, V, causal),
                       rtol=1e-12, atol=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(2)
    S, H, D = 9, 3, 8
    Q = rng.standard_normal((S, H, D))
    K = rng.standard_normal((S, H, D))
    # constant V -> output equals that constant
    c = rng.standard_normal((1, H, D))
    O = ops.attention_definition(Q, K, np.repeat(c, S, axis=0))
    assert np.allclose(O, np.repeat(c, S, axis=0), rtol=0, atol=1e-14)
    # K = 0 -> equal scores -> running mean of V over visible keys
    V = rng.standard_normal((S, H, D))
    O = ops.attention_definition(Q, np.zeros_like(K), V)
    mean = np.cumsum(V, axis=0) / np.arange(1, S + 1)[:, None, None]
    assert np.allclose(O, mean, rtol=1e-12, atol=1e-12)
    # the first query sees only the first key
    O = ops.attention_definition(Q, K, V)
    assert np.allclose(O[0], V[0], rtol=0, atol=1e-15)
    # one dominant key: query i attends only to key j* <= i
    Kd = np.zeros_like(K)
    Kd[3] = 200.0 * Q.mean(axis=0)
    Qd = np.repeat(Q.mean(axis=0, keepdims=True), S, axis=0)
    O = ops.attention_definition(Qd, Kd, V)
    assert np.allclose(O[3:], np.repeat(V[3:4], S - 3, axis=0), atol=1e-9)


@pytest.mark.parametrize("P", [1, 2, 3, 4])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("prune", [False, True])
def test_ring_equals_definition(P, causal, prune):
    rng = np.random.default_rng(10 + P)
    m, H, D = 5, 2, 8
    Q, K, V = ([rng.standard_normal((m, H, D)) for _ in range(P)] for _ in range(3))
    O, log = ops.qsplit_attention_ring(Q, K, V, causal=causal, prune=prune)
    ref = ops.attention_definition(np.concatenate(Q), np.concatenate(K), np.concatenate(V), causal)
    assert np.allclose(np.concatenate(O), ref, rtol=1e-12, atol=1e-12)
    for r in range(P):
        used = sorted(s for (rr, t, s, u) in log if rr == r and u)
        assert used == (list(range(r + 1)) if causal else list(range(P)))
        first = [(t, s, u) for (rr, t, s, u) in log if rr == r and t == 0]
        assert first == [(0, r, True)], "local slice first"


def test_ring_sampled_rows_match_definition():
    rng = np.random.default_rng(3)
    P, m, H, D = 3, 6, 2, 4
    Q, K, V = ([rng.standard_normal((m, H, D)) for _ in range(P)] for _ in range(3))
    rows = [np.array([0, 5]), np.array([2]), np.array([0, 1, 5])]
    O, _ = ops.qsplit_attention_ring(Q, K, V, q_rows=rows)
    Kc, Vc, Qc = np.concatenate(K), np.concatenate(V), np.concatenate(Q)
    for r in range(P):
        ref = ops.attention_definition(Qc, Kc, Vc, q_rows=r * m + rows[r])
        assert np.allclose(O[r], ref, rtol=1e-12, atol=1e-12)


def test_planted_mistakes_are_caught(monkeypatch):
    rng = np.random.default_rng(4)
    Q, K, V = (rng.standard_normal((5, 1, 4)) for _ in range(3))
    brute = _brute_attention(Q, K, V)
    with monkeypatch.context() as mp:   # scale dropped
        mp.setattr(ops.math, "sqrt", lambda x: 1.0)
        assert not np.allclose(ops.attention_definition(Q, K, V), brute, atol=1e-9)
    # a diagonal-exclusive mask would leave query 0 with no key (NaN), caught by the row-0 pin
    s = (Q[:, 0] @ K[:, 0].T) / 2.0
    s = np.where(np.arange(5)[None, :] >= np.arange(5)[:, None], -np.inf, s)
    with np.errstate(invalid="ignore"):
        p = np.exp(s - s.max(axis=1, keepdims=True))
    assert np.isnan(p[0]).all()
