"""Parity at the benchmark configurations' full sizes, in the launch configuration
bench.py times, on sampled output rows that the oracle computes one by one
(an output row of these layers depends only on its own token row / query row).

Configurations (FlashOverlap summary, section 4 workloads: MLP layer, sequence
1K-16K, attention): Llama-3-8B MLP P=4; 70B-like MLP P=8 at 1K (all rows) and
16K (sampled); tail-dominated GEMM-RS P=8 (flash and naive order);
query-split causal attention P=4, seq 16384, 32 heads."""
import numpy as np
import pytest
import torch

import fo_workloads as wl
from helpers import assert_close, f64, to_bits, to_dev, guarded
from oracle import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import overlapped_tensor_gemm_gb300 as fo
    c = fo.Context(0)
    yield c
    c.close()


def _mlp_check(ctx, cfg, X_bits, Wc_bits, Wr_bits, rows_per_slice, seed):
    X = [to_dev(x) for x in X_bits]
    Wc = [to_dev(w) for w in Wc_bits]
    Wr = [to_dev(w) for w in Wr_bits]
    Z = [guarded((cfg.m, cfg.hidden), torch.bfloat16) for _ in range(cfg.P)]
    ctx.mlp_layer(X, Wc, Wr, Z, gated=cfg.gated)
    torch.cuda.synchronize()
    ctx.poll()
    if rows_per_slice is None:
        rows = [np.arange(cfg.m) for _ in range(cfg.P)]
    else:
        rows = [wl.sample_rows(cfg.m, 128, rows_per_slice, seed + s) for s in range(cfg.P)]
    _, _, ref = ops.mlp_layer([f64(X_bits[s])[rows[s]] for s in range(cfg.P)], [f64(w) for w in Wc_bits],
                              [f64(w) for w in Wr_bits], gated=cfg.gated)
    for d in range(cfg.P):
        got = f64(to_bits(Z[d][torch.as_tensor(rows[d], device="cuda")]))
        assert_close(got, ref[d], f"{cfg.name} rank {d}")


def test_llama8b_mlp_sampled_rows(ctx):
    cfg = wl.LLAMA8B
    inp = wl.mlp_inputs(cfg)
    _mlp_check(ctx, cfg, inp["X_shards"], inp["W_col"], inp["W_row"], 6, 11)


@pytest.fixture(scope="module")
def sweep_weights():
    cfg = wl.sweep(1024)
    g = torch.Generator().manual_seed(cfg.seed)
    Wc = [wl.gaussian_bf16(g, (cfg.n_col, cfg.hidden), wl.W_STD) for _ in range(cfg.P)]
    Wr = [wl.gaussian_bf16(g, (cfg.hidden, cfg.k_row), wl.W_STD) for _ in range(cfg.P)]
    return Wc, Wr


@pytest.mark.parametrize("tokens,rows", [(1024, None), (16384, 3)])
def test_sweep_mlp(ctx, sweep_weights, tokens, rows):
    cfg = wl.sweep(tokens)
    g = torch.Generator().manual_seed(cfg.seed + tokens)
    X = [wl.gaussian_bf16(g, (cfg.m, cfg.hidden)) for _ in range(cfg.P)]
    _mlp_check(ctx, cfg, X, sweep_weights[0], sweep_weights[1], rows, 21)


@pytest.mark.parametrize("order", ["flash", "naive"])
def test_tail_rs_full(ctx, order):
    c = wl.TAIL_RS
    inp = wl.rs_inputs(c.P, c.tokens, c.n_out, c.k_row, c.seed, integer=False)
    X = [to_dev(x) for x in inp["X"]]
    W = [to_dev(w) for w in inp["W_row"]]
    Y = [guarded((c.m, c.n_out), torch.bfloat16) for _ in range(c.P)]
    ctx.gemm_rs(X, W, Y, order=order)
    torch.cuda.synchronize()
    ctx.poll()
    chunks = [ops.split_chunks(f64(x), c.P) for x in inp["X"]]
    ref = ops.gemm_rs_definition(chunks, [f64(w) for w in inp["W_row"]])
    for d in range(c.P):
        assert_close(f64(to_bits(Y[d])), ref[d], f"tail RS {order} rank {d}")


def test_attention_full_sampled_rows(ctx):
    c = wl.ATTN
    inp = wl.attn_inputs(c.P, c.seq, c.heads, c.head_dim, c.seed)
    shape = (c.m, c.heads * c.head_dim)
    Q = [to_dev(x).reshape(shape) for x in inp["Q"]]
    K = [to_dev(x).reshape(shape) for x in inp["K"]]
    V = [to_dev(x).reshape(shape) for x in inp["V"]]
    O = [guarded(shape, torch.bfloat16) for _ in range(c.P)]
    ctx.qsplit_attn(Q, K, V, O, heads=c.heads, head_dim=c.head_dim)
    torch.cuda.synchronize()
    ctx.poll()
    Kc = np.concatenate([f64(x) for x in inp["K"]])
    Vc = np.concatenate([f64(x) for x in inp["V"]])
    for r in range(c.P):
        rows = wl.sample_rows(c.m, 1024, 3, 40 + r)
        Qr = f64(inp["Q"][r])
        Qfull = np.zeros((c.seq, c.heads, c.head_dim))
        Qfull[r * c.m + rows] = Qr[rows]
        ref = ops.attention_definition(Qfull, Kc, Vc, q_rows=r * c.m + rows)
        got = f64(to_bits(O[r][torch.as_tensor(rows, device="cuda")])).reshape(len(rows), c.heads, c.head_dim)
        assert_close(got, ref, f"attention rank {r}")
