"""Pins of the oracle's AG-GEMM / GEMM-RS (FlashOverlap technical summary, section 2).

Every pin compares the oracle against something other than itself: pure-Python
integer brute force, the exactness the method claims (decomposed == undecomposed),
schedule-order independence over all permutations, P=1 collapsing to a plain GEMM,
and the step-order rules (local slice first, kept slice last).
"""
import itertools

import numpy as np
import pytest

from oracle import ops, schedule
from oracle.ring import RingError


def _ints(rng, shape):
    return rng.integers(-2, 3, shape).astype(np.float64)


def _brute_gemm(A, B):
    """Pure-Python integer C = A @ B^T (no numpy arithmetic)."""
    A = [[int(v) for v in row] for row in np.asarray(A)]
    B = [[int(v) for v in row] for row in np.asarray(B)]
    return [[sum(a * b for a, b in zip(ra, rb)) for rb in B] for ra in A]


def _as_int(Y):
    return [[int(v) for v in row] for row in np.asarray(Y)]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("direction", [1, -1])
def test_ag_ring_equals_brute_force(P, direction):
    rng = np.random.default_rng(10 + P)
    m, K, N = 3, 7, 5
    X = [_ints(rng, (m, K)) for _ in range(P)]
    W = [_ints(rng, (N, K)) for _ in range(P)]
    Y, log = ops.ag_gemm_ring(X, W, direction=direction)
    full = [list(row) for x in X for row in np.asarray(x)]
    for r in range(P):
        assert _as_int(Y[r]) == _brute_gemm(full, W[r])
    # schedule: local slice first, every slice exactly once per rank
    for r in range(P):
        steps = sorted((t, s) for (rr, t, s) in log if rr == r)
        assert steps[0] == (0, r)
        assert sorted(s for _, s in steps) == list(range(P))


@pytest.mark.parametrize("P", [2, 3, 4])
def test_ag_every_compute_order_gives_identical_result(P):
    rng = np.random.default_rng(20 + P)
    X = [_ints(rng, (2, 6)) for _ in range(P)]
    W = [_ints(rng, (3, 6)) for _ in range(P)]
    ref, _ = ops.ag_gemm_ring(X, W)
    for perm in itertools.permutations(range(P)):
        orders = [list(perm)] * P
        Y, _ = ops.ag_gemm_ring(X, W, compute_order=orders)
        for r in range(P):
            assert np.array_equal(Y[r], ref[r])


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("direction", [1, -1])
@pytest.mark.parametrize("order", ["flash", "naive"])
def test_rs_ring_equals_brute_force(P, direction, order):
    if order == "naive" and direction == -1:
        pytest.skip("naive order is defined on the +1 ring")
    rng = np.random.default_rng(30 + P)
    m, Kp, N = 2, 5, 4
    Xfull = [_ints(rng, (P * m, Kp)) for _ in range(P)]
    W = [_ints(rng, (N, Kp)) for _ in range(P)]
    chunks = [ops.split_chunks(x, P) for x in Xfull]
    Y, log = ops.gemm_rs_ring(chunks, W, order=order, direction=direction)
    # brute force: Y = sum_r X_r W_r^T over the concatenated K dimension, row chunk d to rank d
    Xcat = np.concatenate(Xfull, axis=1)
    Wcat = np.concatenate(W, axis=1)
    full = _brute_gemm(Xcat, Wcat)
    for d in range(P):
        assert _as_int(Y[d]) == full[d * m:(d + 1) * m]
    for r in range(P):
        steps = sorted((t, c) for (rr, t, c) in log if rr == r)
        assert sorted(c for _, c in steps) == list(range(P))
        if order == "flash":
            assert steps[-1] == (P - 1, r), "kept slice must be computed last"
        else:
            assert [c for _, c in steps] == list(range(P))


@pytest.mark.parametrize("P", [2, 3, 4, 6, 8])
def test_rs_definition_equals_ring_and_p1_is_plain_gemm(P):
    rng = np.random.default_rng(40 + P)
    Xfull = [_ints(rng, (P * 4, 8)) for _ in range(P)]
    W = [_ints(rng, (6, 8)) for _ in range(P)]
    chunks = [ops.split_chunks(x, P) for x in Xfull]
    Yd = ops.gemm_rs_definition(chunks, W)
    Yr, _ = ops.gemm_rs_ring(chunks, W)
    for d in range(P):
        assert np.array_equal(Yd[d], Yr[d])
    # P = 1: reduce-scatter of one rank is the identity
    Y1, _ = ops.gemm_rs_ring([[Xfull[0]]], [W[0]])
    assert _as_int(Y1[0]) == _brute_gemm(Xfull[0], W[0])
    Ya, _ = ops.ag_gemm_ring([Xfull[0]], [W[0]])
    assert _as_int(Ya[0]) == _brute_gemm(Xfull[0], W[0])


def test_schedule_formulas_local_first_kept_last():
    for P in range(1, 9):
        for r in range(P):
            ag = [schedule.ag_slice(r, t, P) for t in range(P)]
            rs = [schedule.rs_chunk(r, t, P) for t in range(P)]
            assert ag[0] == r and sorted(ag) == list(range(P))
            assert rs[-1] == r and sorted(rs) == list(range(P))
            for t in range(P - 1):
                # what rank r forwards at hop t+1 is what its successor needs at step t+1
                assert schedule.ag_slice((r + 1) % P, t + 1, P) == ag[t]
                assert schedule.rs_chunk((r + 1) % P, t + 1, P) == rs[t]
            for c in range(P):
                assert schedule.rs_hop(c, c, P) == P - 1


def _drop_first(target_seq):
    state = {"done": False}

    def fault(src, dst, msg):
        if not state["done"] and msg.seq == target_seq:
            state["done"] = True
            return []
        return [msg]
    return fault


def _duplicate(src, dst, msg):
    return [msg, msg] if (src, msg.seq) == (0, 1) else [msg]


def _reorder():
    held = {}

    def fault(src, dst, msg):
        if src == 0 and msg.seq == 1:
            held["m"] = msg
            return []
        if src == 0 and "m" in held:
            return [msg, held.pop("m")]
        return [msg]
    return fault


@pytest.mark.parametrize("make_fault", [lambda: _drop_first(1), lambda: _drop_first(2),
                                        lambda: _duplicate, _reorder])
def test_ring_faults_are_detected(make_fault):
    P = 4
    rng = np.random.default_rng(5)
    X = [_ints(rng, (2, 3)) for _ in range(P)]
    W = [_ints(rng, (2, 3)) for _ in range(P)]
    with pytest.raises(RingError):
        ops.ag_gemm_ring(X, W, fault=make_fault())
    chunks = [ops.split_chunks(_ints(rng, (P * 2, 3)), P) for _ in range(P)]
    with pytest.raises(RingError):
        ops.gemm_rs_ring(chunks, W, fault=make_fault())


# ----------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the pins above
# ----------------------------------------------------------------------------

def _rs_pins_pass(P=4):
    try:
        test_rs_ring_equals_brute_force(P, 1, "flash")
        return True
    except (AssertionError, RingError, ValueError, TypeError, KeyError):
        return False


def _ag_pins_pass(P=3):
    try:
        test_ag_ring_equals_brute_force(P, 1)
        return True
    except (AssertionError, RingError, ValueError, KeyError):
        return False


def test_planted_mistakes_are_caught(monkeypatch):
    assert _rs_pins_pass() and _ag_pins_pass()
    with monkeypatch.context() as mp:      # kept slice not last (off-by-one chunk order)
        mp.setattr(ops, "rs_chunk", lambda r, t, P, d=1: (r - d * t) % P)
        assert not _rs_pins_pass()
    with monkeypatch.context() as mp:      # accumulator dropped (no add of the incoming partial)
        real = ops.rs_hop
        mp.setattr(ops, "rs_hop", lambda r, c, P, d=1: 0 if real(r, c, P, d) < P - 1 else P - 1)
        assert not _rs_pins_pass()
    with monkeypatch.context() as mp:      # weight rows taken in the wrong order
        mp.setattr(ops, "gemm", lambda A, B: np.asarray(A, float) @ np.asarray(B, float)[::-1].T)
        assert not _ag_pins_pass()
    with monkeypatch.context() as mp:      # a dropped term of the contraction
        mp.setattr(ops, "gemm", lambda A, B: np.asarray(A, float)[:, 1:] @ np.asarray(B, float)[:, 1:].T)
        assert not _ag_pins_pass()
    with monkeypatch.context() as mp:      # a slice computed from the wrong rank's buffer
        mp.setattr(ops, "ag_slice", lambda r, t, P, d=1: (r - d * t) % P if t < 2 else (r - d * (t - 1)) % P)
        assert not _ag_pins_pass(P=4)
