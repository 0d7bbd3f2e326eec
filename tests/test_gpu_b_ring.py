"""Parity of Flash-AG / Flash-RS / the MLP layer (and their baselines) against the
oracle's simulated ring, through the C ABI (FlashOverlap technical summary, section 2)."""
import numpy as np
import pytest
import torch

import fo_workloads as wl
from helpers import assert_bits_equal, assert_close, f64, padded, to_bits, to_dev
from oracle import bf16, ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import overlapped_tensor_gemm_gb300 as fo
    c = fo.Context(0)
    yield c
    c.close()


def _ag(ctx, P, m, K, N, integer, seed, **kw):
    inp = wl.ag_inputs(P, m, K, N, seed, integer)
    X = [to_dev(x) for x in inp["X_shards"]]
    W = [to_dev(w) for w in inp["W_col"]]
    Y = [padded(P * m, N, torch.bfloat16) for _ in range(P)]
    ctx.ag_gemm(X, W, Y, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    ref, _ = ops.ag_gemm_ring([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]])
    return Y, ref


def _rs(ctx, P, m, Kr, N, integer, seed, **kw):
    inp = wl.rs_inputs(P, P * m, N, Kr, seed, integer)
    X = [to_dev(x) for x in inp["X"]]
    W = [to_dev(w) for w in inp["W_row"]]
    Y = [padded(m, N, torch.bfloat16) for _ in range(P)]
    ctx.gemm_rs(X, W, Y, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    chunks = [ops.split_chunks(f64(x), P) for x in inp["X"]]
    ref, _ = ops.gemm_rs_ring(chunks, [f64(w) for w in inp["W_row"]])
    return Y, ref


@pytest.mark.parametrize("P,m,K,N", [(1, 128, 256, 256), (2, 128, 256, 512), (4, 256, 512, 768),
                                     (3, 200, 136, 300), (8, 128, 128, 256)])
def test_ag_flash_integer_bit_exact(ctx, P, m, K, N):
    Y, ref = _ag(ctx, P, m, K, N, True, 100 + P)
    for r in range(P):
        assert_bits_equal(to_bits(Y[r]), ref[r], f"AG P={P} rank {r}")


@pytest.mark.parametrize("order", ["serial", "slicing"])
def test_ag_baselines_integer_bit_exact(ctx, order):
    P, m, K, N = 4, 256, 512, 512
    Y, ref = _ag(ctx, P, m, K, N, True, 7, order=order)
    for r in range(P):
        assert_bits_equal(to_bits(Y[r]), ref[r], f"AG {order} rank {r}")


@pytest.mark.parametrize("P,m,Kr,N", [(1, 128, 256, 256), (2, 128, 256, 512), (4, 256, 384, 512),
                                      (3, 72, 200, 264), (8, 64, 128, 1024)])
@pytest.mark.parametrize("order", ["flash", "naive"])
def test_rs_integer_bit_exact(ctx, P, m, Kr, N, order):
    Y, ref = _rs(ctx, P, m, Kr, N, True, 200 + P, order=order)
    for r in range(P):
        assert_bits_equal(to_bits(Y[r]), ref[r], f"RS {order} P={P} rank {r}")


@pytest.mark.parametrize("order", ["serial", "slicing"])
def test_rs_baselines_integer_bit_exact(ctx, order):
    P, m, Kr, N = 4, 256, 256, 512
    Y, ref = _rs(ctx, P, m, Kr, N, True, 9, order=order)
    for r in range(P):
        assert_bits_equal(to_bits(Y[r]), ref[r], f"RS {order} rank {r}")


def test_ag_rs_gaussian_tolerance(ctx):
    Y, ref = _ag(ctx, 4, 256, 1024, 512, False, 11)
    for r in range(4):
        assert_close(f64(to_bits(Y[r])), ref[r], f"AG gaussian rank {r}")
    Y, ref = _rs(ctx, 4, 256, 1024, 512, False, 12)
    for r in range(4):
        assert_close(f64(to_bits(Y[r])), ref[r], f"RS gaussian rank {r}")


def test_tiny_mlp_layer_bit_exact(ctx):
    cfg = wl.TINY
    inp = wl.mlp_inputs(cfg)
    X = [to_dev(x) for x in inp["X_shards"]]
    Wc = [to_dev(w) for w in inp["W_col"]]
    Wr = [to_dev(w) for w in inp["W_row"]]
    Z = [torch.empty((cfg.m, cfg.hidden), dtype=torch.bfloat16, device="cuda") for _ in range(cfg.P)]
    ctx.mlp_layer(X, Wc, Wr, Z, gated=False)
    torch.cuda.synchronize()
    ctx.poll()
    _, _, ref = ops.mlp_layer([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]],
                              [f64(w) for w in inp["W_row"]], gated=False)
    for r in range(cfg.P):
        assert_bits_equal(to_bits(Z[r]), ref[r], f"tiny MLP rank {r}")


def test_gated_mlp_layer_tolerance(ctx):
    cfg = wl.MLPConfig("small-gated", 1, P=4, tokens=512, hidden=256, ffn=1024, gated=True, integer=False)
    inp = wl.mlp_inputs(cfg)
    X = [to_dev(x) for x in inp["X_shards"]]
    Wc = [to_dev(w) for w in inp["W_col"]]
    Wr = [to_dev(w) for w in inp["W_row"]]
    Z = [torch.empty((cfg.m, cfg.hidden), dtype=torch.bfloat16, device="cuda") for _ in range(cfg.P)]
    ctx.mlp_layer(X, Wc, Wr, Z, gated=True)
    torch.cuda.synchronize()
    ctx.poll()
    _, _, ref = ops.mlp_layer([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]],
                              [f64(w) for w in inp["W_row"]], gated=True)
    for r in range(cfg.P):
        assert_close(f64(to_bits(Z[r])), ref[r], f"gated MLP rank {r}")


def test_silu_mul_standalone(ctx):
    # layer glue on its own: H = SiLU(G) * U from the bf16 gate/up block, rounded once
    P, M, F = 2, 256, 384
    g = torch.Generator().manual_seed(31)
    GU = [wl.gaussian_bf16(g, (M, 2 * F), 3.0) for _ in range(P)]
    H = [torch.empty((M, F), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ctx.silu_mul([to_dev(x) for x in GU], H)
    torch.cuda.synchronize()
    for r in range(P):
        ref = ops.silu_mul(f64(GU[r])[:, :F], f64(GU[r])[:, F:])
        assert_close(f64(to_bits(H[r])), ref, f"silu_mul rank {r}")


def test_gated_fused_epilogue_matches_unfused(ctx):
    # the fused Flash-AG epilogue (SiLU(gate)*up) against the unfused AG GEMM + glue kernel
    cfg = wl.MLPConfig("fused", 1, P=2, tokens=256, hidden=512, ffn=768, gated=True, integer=False)
    inp = wl.mlp_inputs(cfg)
    X = [to_dev(x) for x in inp["X_shards"]]
    Wc = [to_dev(w) for w in inp["W_col"]]
    Wr = [to_dev(w) for w in inp["W_row"]]
    Z = [torch.empty((cfg.m, cfg.hidden), dtype=torch.bfloat16, device="cuda") for _ in range(cfg.P)]
    ctx.mlp_layer(X, Wc, Wr, Z, gated=True)
    Y = [torch.empty((cfg.tokens, cfg.n_col), dtype=torch.bfloat16, device="cuda") for _ in range(cfg.P)]
    H = [torch.empty((cfg.tokens, cfg.k_row), dtype=torch.bfloat16, device="cuda") for _ in range(cfg.P)]
    Z2 = [torch.empty_like(z) for z in Z]
    ctx.ag_gemm(X, Wc, Y)
    ctx.silu_mul(Y, H)
    ctx.gemm_rs(H, Wr, Z2)
    torch.cuda.synchronize()
    ctx.poll()
    for r in range(cfg.P):
        assert np.array_equal(to_bits(Z[r]), to_bits(Z2[r])), f"rank {r}: fused and unfused glue differ"


# Slices of 32-128 rows run on transposed tiles (the weight's features on the MMA's M side,
# the token rows of 256/m consecutive ring steps of one rank on its N side), on single SMs by
# default and on SM pairs on request (pairs=True); a grid smaller than P falls back to the
# step-ordered tiles.  Ragged feature counts leave the last feature block partly empty.
@pytest.mark.parametrize("P,m,Kr,N", [(8, 64, 256, 1024), (4, 64, 136, 516), (2, 128, 192, 260),
                                      (8, 32, 128, 512), (8, 128, 64, 768)])
@pytest.mark.parametrize("order", ["flash", "naive"])
@pytest.mark.parametrize("pairs", [False, True])
def test_rs_transposed_tiles_integer_bit_exact(ctx, P, m, Kr, N, order, pairs):
    Y, ref = _rs(ctx, P, m, Kr, N, True, 400 + P + m, order=order, pairs=pairs)
    for r in range(P):
        assert_bits_equal(to_bits(Y[r]), ref[r], f"RS transposed {order} P={P} m={m} rank {r}")


def test_rs_small_grid_falls_back_to_step_tiles(ctx):
    P, m, Kr, N = 8, 64, 128, 512
    Y, ref = _rs(ctx, P, m, Kr, N, True, 77, num_sms=4)
    for r in range(P):
        assert_bits_equal(to_bits(Y[r]), ref[r], f"RS small grid rank {r}")


def test_rs_transposed_tiles_gaussian_tolerance(ctx):
    Y, ref = _rs(ctx, 8, 64, 1024, 2048, False, 78)
    for r in range(8):
        assert_close(f64(to_bits(Y[r])), ref[r], f"RS transposed gaussian rank {r}")
