"""Edge cases of the hot path on the GPU: empty inputs (every entry point returns without
work and leaves the outputs untouched), one rank (the decomposed collectives reduce to a
plain GEMM / plain causal attention), and the maximum of eight ranks."""
import numpy as np
import pytest
import torch

import fo_workloads as wl
from helpers import assert_bits_equal, assert_close, f64, to_bits, to_dev, guarded
from oracle import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import overlapped_tensor_gemm_gb300 as fo
    c = fo.Context(0)
    yield c
    c.close()


def _bf(shape, fill=3.0):
    return torch.full(shape, fill, dtype=torch.bfloat16, device="cuda")


def test_empty_token_slices_do_nothing(ctx):
    P, K, N = 2, 128, 256
    X = [_bf((0, K)) for _ in range(P)]
    W = [_bf((N, K)) for _ in range(P)]
    Y = [_bf((0, N)) for _ in range(P)]
    ctx.ag_gemm(X, W, Y)
    ctx.gemm_rs([_bf((0, K)) for _ in range(P)], W, [_bf((0, N)) for _ in range(P)])
    ctx.gemm_a2a(X, [_bf((2 * 128, K)) for _ in range(P)], [_bf((0, 128)) for _ in range(P)])
    ctx.a2a_gemm([_bf((0, 64)) for _ in range(P)], [_bf((N, 128)) for _ in range(P)],
                 [_bf((0, N)) for _ in range(P)])
    ctx.qsplit_attn([_bf((0, 128)) for _ in range(P)], [_bf((0, 128)) for _ in range(P)],
                    [_bf((0, 128)) for _ in range(P)], [_bf((0, 128)) for _ in range(P)], heads=1, head_dim=128)
    ctx.mlp_layer([_bf((0, 256)) for _ in range(P)], [_bf((512, 256)) for _ in range(P)],
                  [_bf((256, 256)) for _ in range(P)], [_bf((0, 256)) for _ in range(P)], gated=True)
    torch.cuda.synchronize()
    ctx.poll()


def test_empty_output_columns_leave_no_trace(ctx):
    # N = 0: nothing to compute; the inputs are untouched
    P, m, K = 2, 128, 128
    X = [_bf((m, K), 1.0) for _ in range(P)]
    ctx.ag_gemm(X, [_bf((0, K)) for _ in range(P)], [_bf((P * m, 0)) for _ in range(P)])
    torch.cuda.synchronize()
    ctx.poll()
    assert all(bool((x == 1.0).all()) for x in X)


def test_one_rank_all_to_all_is_a_plain_gemm(ctx):
    g = torch.Generator().manual_seed(900)
    m, K, N = 256, 192, 320
    X = wl.integer_bf16(g, (m, K))
    W = wl.integer_bf16(g, (N, K))
    Y = [torch.empty((m, N), dtype=torch.bfloat16, device="cuda")]
    ctx.gemm_a2a([to_dev(X)], [to_dev(W)], Y)
    Z = [torch.empty((m, N), dtype=torch.bfloat16, device="cuda")]
    ctx.a2a_gemm([to_dev(X[:, :128])], [to_dev(W[:, :128])], Z)
    torch.cuda.synchronize()
    ctx.poll()
    assert_bits_equal(to_bits(Y[0]), f64(X) @ f64(W).T, "gemm->a2a P=1")
    assert_bits_equal(to_bits(Z[0]), f64(X[:, :128]) @ f64(W[:, :128]).T, "a2a->gemm P=1")


def test_eight_rank_all_to_all(ctx):
    P, m, Kc, N = 8, 128, 64, 256
    g = torch.Generator().manual_seed(901)
    C = [wl.integer_bf16(g, (P * m, Kc)) for _ in range(P)]
    W = [wl.integer_bf16(g, (N, P * Kc)) for _ in range(P)]
    Y = [torch.empty((m, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ctx.a2a_gemm([to_dev(c) for c in C], [to_dev(w) for w in W], Y)
    torch.cuda.synchronize()
    ctx.poll()
    ref = ops.a2a_gemm_definition([f64(c) for c in C], [f64(w) for w in W])
    for d in range(P):
        assert_bits_equal(to_bits(Y[d]), ref[d], f"a2a->gemm P=8 rank {d}")


def test_eight_rank_query_split_attention(ctx):
    P, m, H = 8, 128, 1
    inp = wl.attn_inputs(P, P * m, H, 128, 902)
    Q = [to_dev(x).reshape(m, 128) for x in inp["Q"]]
    K = [to_dev(x).reshape(m, 128) for x in inp["K"]]
    V = [to_dev(x).reshape(m, 128) for x in inp["V"]]
    O = [guarded((m, 128), torch.bfloat16) for _ in range(P)]
    ctx.qsplit_attn(Q, K, V, O, heads=H, head_dim=128)
    torch.cuda.synchronize()
    ctx.poll()
    ref = ops.attention_definition(np.concatenate([f64(x) for x in inp["Q"]]),
                                   np.concatenate([f64(x) for x in inp["K"]]),
                                   np.concatenate([f64(x) for x in inp["V"]]))
    got = np.concatenate([f64(to_bits(o)).reshape(m, H, 128) for o in O])
    assert_close(got, ref, "attention P=8")
