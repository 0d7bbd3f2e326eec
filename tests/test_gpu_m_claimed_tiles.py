"""SM-pair launches with at least 128 tiles per pair claim their tiles in order from a
launch-wide counter; the leader CTA's producer hands each index to both CTAs' roles through a
ring in shared memory.  Capping the grid at four SM pairs makes small launches long enough to
take that path.  Checked bit-exact against the oracle's ring on integer inputs: twice in a row
(the launch's last claim resets the counter for the next launch), after a launch that timed out
(fo_ctx_poll resets the counter with the rest of the control block), and for the one-launch
MLP layer, whose reduce-scatter tiles wait for the all-gather tiles that wrote their rows."""
import pytest
import torch

import fo_workloads as wl
from helpers import assert_bits_equal, f64, padded, to_bits, to_dev
from oracle import ops

pytestmark = pytest.mark.gpu

GRID = dict(num_sms=8)  # four SM pairs: 512 tiles or more claim


def _ag_inputs(P, m, K, N, seed):
    inp = wl.ag_inputs(P, m, K, N, seed, True)
    X = [to_dev(x) for x in inp["X_shards"]]
    W = [to_dev(w) for w in inp["W_col"]]
    ref, _ = ops.ag_gemm_ring([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]])
    return X, W, ref


def test_claimed_ag_bit_exact_twice_in_a_row():
    import overlapped_tensor_gemm_gb300 as fo
    P, m, K, N = 4, 256, 256, 8192  # 16 units x 32 tiles = 512 tiles on 4 pairs
    X, W, ref = _ag_inputs(P, m, K, N, 91)
    with fo.Context(0) as ctx:
        for call in range(2):
            Y = [padded(P * m, N, torch.bfloat16) for _ in range(P)]
            ctx.ag_gemm(X, W, Y, **GRID)
            torch.cuda.synchronize()
            ctx.poll()
            for r in range(P):
                assert_bits_equal(to_bits(Y[r]), ref[r], f"claimed AG call {call} rank {r}")


def test_claimed_rs_bit_exact():
    import overlapped_tensor_gemm_gb300 as fo
    P, m, Kr, N = 4, 256, 256, 8192  # 16 units x 32 tiles
    inp = wl.rs_inputs(P, P * m, N, Kr, 92, True)
    X = [to_dev(x) for x in inp["X"]]
    W = [to_dev(w) for w in inp["W_row"]]
    chunks = [[f64(x)[c * m:(c + 1) * m] for c in range(P)] for x in inp["X"]]
    ref, _ = ops.gemm_rs_ring(chunks, [f64(w) for w in inp["W_row"]])
    with fo.Context(0) as ctx:
        for order in ("flash", "naive"):
            Y = [padded(m, N, torch.bfloat16) for _ in range(P)]
            ctx.gemm_rs(X, W, Y, order=order, **GRID)
            torch.cuda.synchronize()
            ctx.poll()
            for r in range(P):
                assert_bits_equal(to_bits(Y[r]), ref[r], f"claimed RS {order} rank {r}")


def test_claimed_ag_timeout_then_recovers():
    import overlapped_tensor_gemm_gb300 as fo
    P, m, K, N = 4, 256, 256, 8192
    X, W, ref = _ag_inputs(P, m, K, N, 93)
    with fo.Context(0) as ctx:
        Y = [padded(P * m, N, torch.bfloat16) for _ in range(P)]
        ctx.ag_gemm(X, W, Y, fault="skip_hop", timeout_us=20000, **GRID)
        torch.cuda.synchronize()
        with pytest.raises(fo.FoError) as e:
            ctx.poll()
        assert e.value.status == fo.FO_ERR_TIMEOUT
        Y = [padded(P * m, N, torch.bfloat16) for _ in range(P)]
        ctx.ag_gemm(X, W, Y, **GRID)
        torch.cuda.synchronize()
        ctx.poll()
        for r in range(P):
            assert_bits_equal(to_bits(Y[r]), ref[r], f"claimed AG after recovery rank {r}")


def test_claimed_one_launch_layer_bit_exact():
    import overlapped_tensor_gemm_gb300 as fo
    # AG: 16 units x 32 tiles, RS: 16 units x 2 tiles = 544 tiles on 4 pairs
    cfg = wl.MLPConfig("claimed-int", 0, P=4, tokens=1024, hidden=512, ffn=32768, gated=False, integer=True)
    inp = wl.mlp_inputs(cfg, seed_offset=94)
    X = [to_dev(x) for x in inp["X_shards"]]
    Wc = [to_dev(w) for w in inp["W_col"]]
    Wr = [to_dev(w) for w in inp["W_row"]]
    _, _, ref = ops.mlp_layer([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]],
                              [f64(w) for w in inp["W_row"]], gated=False)
    with fo.Context(0) as ctx:
        Z = [padded(cfg.m, cfg.hidden, torch.bfloat16) for _ in range(cfg.P)]
        ctx.mlp_layer(X, Wc, Wr, Z, gated=False, **GRID)
        torch.cuda.synchronize()
        ctx.poll()
        for r in range(cfg.P):
            assert_bits_equal(to_bits(Z[r]), ref[r], f"claimed one-launch layer rank {r}")
