"""Pins of the oracle's MLP chain and of the timeline model (FlashOverlap technical
summary: section 1 on the last chunk's exposed communication, section 2 on local-first
and kept-last scheduling, section 4 on the MLP layer)."""
import math

import numpy as np
import pytest

import fo_workloads as wl
from oracle import bf16, ops, schedule


def test_silu_mul_closed_forms_and_brute_force():
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0, 2.5, -700.0])
    u = np.array([3.0, 2.0, 2.0, 1.0, 1.0, -4.0, 1.0])
    out = ops.silu_mul(g, u)
    brute = [gi / (1.0 + math.exp(-gi)) * ui if gi > -700 else 0.0 for gi, ui in zip(g, u)]
    assert np.allclose(out, brute, rtol=1e-15, atol=1e-300)
    assert out[0] == 0.0
    assert abs(out[3] - 30.0) < 1e-10 and abs(out[4]) < 1e-11


def _brute_chain(X, Wc, Wr, P):
    """Integer MLP chain with pure-Python ints and the oracle's bf16 rounding."""
    Xfull = [[int(v) for v in row] for x in X for row in np.asarray(bf16.to_f64(x))]
    out_rows = []
    Wc_i = [[[int(v) for v in row] for row in bf16.to_f64(w)] for w in Wc]
    Wr_i = [[[int(v) for v in row] for row in bf16.to_f64(w)] for w in Wr]
    H = []
    for r in range(P):
        Yr = [[sum(a * b for a, b in zip(xr, wr)) for wr in Wc_i[r]] for xr in Xfull]
        H.append(bf16.round_f64(np.array(Yr, dtype=np.float64)))
    for i in range(len(Xfull)):
        row = []
        for n in range(len(Wr_i[0])):
            row.append(sum(int(H[r][i, k]) * Wr_i[r][n][k] for r in range(P) for k in range(len(Wr_i[r][n]))))
        out_rows.append(row)
    return np.array(out_rows, dtype=np.float64)


def test_integer_chain_matches_brute_force_small():
    cfg = wl.MLPConfig("t", 0, P=2, tokens=8, hidden=6, ffn=8, gated=False, integer=True)
    inp = wl.mlp_inputs(cfg)
    X = [bf16.to_f64(x) for x in inp["X_shards"]]
    Wc = [bf16.to_f64(w) for w in inp["W_col"]]
    Wr = [bf16.to_f64(w) for w in inp["W_row"]]
    _, _, Z = ops.mlp_layer(X, Wc, Wr, gated=False)
    brute = bf16.round_f64(_brute_chain(inp["X_shards"], inp["W_col"], inp["W_row"], cfg.P))
    assert np.array_equal(np.concatenate(Z), brute)


def test_tiny_config_decomposed_equals_definition_bitwise():
    cfg = wl.TINY
    inp = wl.mlp_inputs(cfg)
    X = [bf16.to_f64(x) for x in inp["X_shards"]]
    Wc = [bf16.to_f64(w) for w in inp["W_col"]]
    Wr = [bf16.to_f64(w) for w in inp["W_row"]]
    Yd, Hd, Zd = ops.mlp_layer(X, Wc, Wr, gated=False, decomposed=True)
    Yu, Hu, Zu = ops.mlp_layer(X, Wc, Wr, gated=False, decomposed=False)
    for a, b in zip(Zd + Yd, Zu + Yu):
        assert np.array_equal(bf16.from_f64(a), bf16.from_f64(b))
    # every intermediate stays below 2^24: fp32 accumulation is exact in any order
    assert max(np.abs(z).max() for z in Zd) < 2 ** 24


def test_gated_chain_sampled_rows_equal_full_rows():
    cfg = wl.MLPConfig("g", 1, P=3, tokens=12, hidden=16, ffn=24, gated=True, integer=False)
    inp = wl.mlp_inputs(cfg)
    X = [bf16.to_f64(x) for x in inp["X_shards"]]
    Wc = [bf16.to_f64(w) for w in inp["W_col"]]
    Wr = [bf16.to_f64(w) for w in inp["W_row"]]
    _, _, Z = ops.mlp_layer(X, Wc, Wr, gated=True)
    rows = [np.array([0, 3]), np.array([1]), np.array([2, 3])]
    _, _, Zs = ops.mlp_layer([X[s][rows[s]] for s in range(3)], Wc, Wr, gated=True)
    for d in range(3):
        assert np.array_equal(Zs[d], Z[d][rows[d]])


@pytest.mark.parametrize("P", [2, 4, 8])
def test_timeline_flash_hides_communication(P):
    for hop in (0.1, 0.5, 1.0):
        assert schedule.timeline("ag_flash", P, hop=hop)["exposed"] == pytest.approx(0.0)
        assert schedule.timeline("rs_flash", P, hop=hop)["exposed"] == pytest.approx(0.0)
        # serial exposes the whole ring, slicing exposes one chunk's transfer
        assert schedule.timeline("ag_serial", P, hop=hop)["exposed"] == pytest.approx((P - 1) * hop)
        sl = schedule.timeline("ag_slicing", P, hop=hop)["exposed"]
        assert sl == pytest.approx((P - 1) * hop / P)
        sl = schedule.timeline("rs_slicing", P, hop=hop)["exposed"]
        assert sl == pytest.approx((P - 1) * hop / P)
        assert schedule.timeline("rs_naive", P, hop=hop)["exposed"] > 0.0
