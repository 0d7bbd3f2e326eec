"""Parity of the attention block (fo_attn_layer: Flash-AG QKV projection, causal
attention of every rank's own heads, Flash-RS output projection) against the oracle
(FlashOverlap technical summary, section 2, architectural instantiations)."""
import numpy as np
import pytest
import torch

import fo_workloads as wl
from helpers import REL_L2_THREE_STAGES, assert_close, f64, to_bits, to_dev, guarded
from oracle import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import overlapped_tensor_gemm_gb300 as fo
    c = fo.Context(0)
    yield c
    c.close()


def _run(ctx, P, tokens, hidden, heads, seed, causal=True, **kw):
    inp = wl.attn_layer_inputs(P, tokens, hidden, heads, 128, seed)
    X = [to_dev(x) for x in inp["X_shards"]]
    Wq = [to_dev(w) for w in inp["W_qkv"]]
    Wo = [to_dev(w) for w in inp["W_o"]]
    m = tokens // P
    Z = [guarded((m, hidden), torch.bfloat16) for _ in range(P)]
    ctx.attn_layer(X, Wq, Wo, Z, heads=heads, causal=causal, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    _, _, ref = ops.attn_layer([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_qkv"]],
                               [f64(w) for w in inp["W_o"]], heads, causal=causal)
    for d in range(P):
        assert_close(f64(to_bits(Z[d])), ref[d], f"attention block rank {d}", rel_l2=REL_L2_THREE_STAGES)


# P=2, 128-row slices: two ring steps per SM-pair tile in the QKV all-gather, transposed tiles
# in the output projection's reduce-scatter, 2 attention query blocks per head;
# P=4, 256-row slices: SM-pair GEMM tiles, 8 query blocks per head, 2 heads per rank.
@pytest.mark.parametrize("P,tokens,hidden,heads", [(2, 256, 256, 1), (4, 1024, 1024, 2)])
def test_attention_block_matches_oracle(ctx, P, tokens, hidden, heads):
    _run(ctx, P, tokens, hidden, heads, 500 + P)


@pytest.mark.parametrize("order", ["naive", "serial", "slicing"])
def test_attention_block_baseline_orders(ctx, order):
    _run(ctx, 2, 512, 256, 1, 510, order=order)


def test_attention_block_non_causal(ctx):
    _run(ctx, 2, 256, 256, 1, 520, causal=False)


def test_attention_block_rejects_bad_shapes(ctx):
    import overlapped_tensor_gemm_gb300 as fo
    inp = wl.attn_layer_inputs(2, 256, 256, 1, 128, 530)
    X = [to_dev(x) for x in inp["X_shards"]]
    Wq = [to_dev(w) for w in inp["W_qkv"]]
    Wo = [to_dev(w) for w in inp["W_o"]]
    Z = [torch.empty((128, 256), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(fo.FoError) as e:
        ctx.attn_layer(X, Wq, Wo, Z, heads=2)  # W_qkv has 3*1*128 rows, not 3*2*128
    assert e.value.status == fo.FO_ERR_SHAPE


def test_attention_block_bench_shape_sampled_rows(ctx):
    """The benchmarked block (P=4, 4096 tokens, hidden 4096, 8 heads of 128 per rank) in
    its launch configuration, checked on sampled output rows.  A sampled row of Z needs
    every rank's attention output at that token, which needs the keys and values of every
    earlier token: the oracle computes the whole QKV projection, attention for the sampled
    query rows only, and the output projection's reduce-scatter of those rows."""
    from oracle import bf16
    c = wl.ATTN_LAYER
    inp = wl.attn_layer_inputs(c.P, c.tokens, c.hidden, c.heads, c.head_dim, c.seed)
    X = [to_dev(x) for x in inp["X_shards"]]
    Wq = [to_dev(w) for w in inp["W_qkv"]]
    Wo = [to_dev(w) for w in inp["W_o"]]
    P, m, hd = c.P, c.m, c.heads * c.head_dim
    Z = [guarded((m, c.hidden), torch.bfloat16) for _ in range(P)]
    ctx.attn_layer(X, Wq, Wo, Z, heads=c.heads)
    torch.cuda.synchronize()
    ctx.poll()
    Xs = [f64(x) for x in inp["X_shards"]]
    rows = [wl.sample_rows(m, 128, 3, 60 + d) for d in range(P)]
    q_rows = np.concatenate([d * m + rows[d] for d in range(P)])
    O = []  # O[r]: rank r's attention output at the sampled tokens, bf16-rounded
    for r in range(P):
        qkv = bf16.round_f64(ops.ag_gemm_definition(Xs, [f64(inp["W_qkv"][r])])[0])
        q = qkv[:, :hd].reshape(-1, c.heads, c.head_dim)
        k = qkv[:, hd:2 * hd].reshape(-1, c.heads, c.head_dim)
        v = qkv[:, 2 * hd:].reshape(-1, c.heads, c.head_dim)
        O.append(bf16.round_f64(ops.attention_definition(q, k, v, True, q_rows=q_rows).reshape(len(q_rows), hd)))
    offs = np.cumsum([0] + [len(x) for x in rows])
    chunks = [[O[r][offs[d]:offs[d + 1]] for d in range(P)] for r in range(P)]
    ref = ops.gemm_rs_definition(chunks, [f64(w) for w in inp["W_o"]])
    for d in range(P):
        got = f64(to_bits(Z[d][torch.as_tensor(rows[d], device="cuda")]))
        assert_close(got, ref[d], f"attention block (bench shape) rank {d}", rel_l2=REL_L2_THREE_STAGES)
