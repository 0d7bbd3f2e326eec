"""One persistent launch for a whole MLP layer (fo_mlp_layer with split_layer = 0):
Flash-AG -> SiLU(gate)*up -> Flash-RS in one tile sequence, the reduce-scatter's tiles
waiting per 256-row (SM pairs) or 128-row block for the rows of the intermediate they read
(FlashOverlap technical summary, section 2: row/column parallel projection of the MLP).

Checked against the oracle's layer (bit-exact on integers with the identity activation,
within tolerance when gated) and against the two-launch layer, bit for bit: the tiles, and
so every summation order, are the same."""
import numpy as np
import pytest
import torch

import fo_workloads as wl
from helpers import assert_bits_equal, assert_close, f64, guarded, to_bits, to_dev
from oracle import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import overlapped_tensor_gemm_gb300 as fo
    c = fo.Context(0)
    yield c
    c.close()


def _layer(ctx, cfg, inp, **kw):
    X = [to_dev(x) for x in inp["X_shards"]]
    Wc = [to_dev(w) for w in inp["W_col"]]
    Wr = [to_dev(w) for w in inp["W_row"]]
    Z = [guarded((cfg.m, cfg.hidden), torch.bfloat16) for _ in range(cfg.P)]
    ctx.mlp_layer(X, Wc, Wr, Z, gated=cfg.gated, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    return [to_bits(z) for z in Z]


# 256-row slices: SM-pair tiles; 192-row slices: single-SM tiles (and no transposed
# reduce-scatter tiles, which would need a launch of their own)
@pytest.mark.parametrize("P,tokens,hidden,ffn", [(4, 1024, 512, 1024), (2, 384, 256, 768), (8, 2048, 256, 2048)])
def test_one_launch_layer_integer_bit_exact(ctx, P, tokens, hidden, ffn):
    cfg = wl.MLPConfig("fused-int", 0, P=P, tokens=tokens, hidden=hidden, ffn=ffn, gated=False, integer=True)
    inp = wl.mlp_inputs(cfg, seed_offset=70 + P)
    got = _layer(ctx, cfg, inp)
    _, _, ref = ops.mlp_layer([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]],
                              [f64(w) for w in inp["W_row"]], gated=False)
    for r in range(P):
        assert_bits_equal(got[r], ref[r], f"one-launch layer P={P} rank {r}")


@pytest.mark.parametrize("P,tokens,hidden,ffn,order", [(4, 1024, 512, 2048, "flash"), (2, 384, 256, 512, "flash"),
                                                       (4, 1024, 512, 2048, "naive")])
def test_one_launch_layer_gated_matches_two_launches_and_oracle(ctx, P, tokens, hidden, ffn, order):
    cfg = wl.MLPConfig("fused-gated", 1, P=P, tokens=tokens, hidden=hidden, ffn=ffn, gated=True, integer=False)
    inp = wl.mlp_inputs(cfg, seed_offset=80 + P)
    one = _layer(ctx, cfg, inp, order=order)
    two = _layer(ctx, cfg, inp, order=order, split_layer=True)
    for r in range(P):
        assert np.array_equal(one[r], two[r]), f"one launch vs two launches, rank {r}"
    _, _, ref = ops.mlp_layer([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]],
                              [f64(w) for w in inp["W_row"]], gated=True)
    for r in range(P):
        assert_close(f64(one[r]), ref[r], f"one-launch gated layer rank {r}")


def test_one_launch_layer_llama8b_shape_sampled_rows(ctx):
    """The Llama-3-8B layer (P=4, 1024-row slices, SM pairs) in one launch."""
    cfg = wl.LLAMA8B
    inp = wl.mlp_inputs(cfg)
    got = _layer(ctx, cfg, inp)
    rows = [wl.sample_rows(cfg.m, 128, 2, 90 + s) for s in range(cfg.P)]
    _, _, ref = ops.mlp_layer([f64(inp["X_shards"][s])[rows[s]] for s in range(cfg.P)],
                              [f64(w) for w in inp["W_col"]], [f64(w) for w in inp["W_row"]], gated=True)
    for d in range(cfg.P):
        assert_close(f64(got[d][rows[d]]), ref[d], f"llama8b one-launch rank {d}")
