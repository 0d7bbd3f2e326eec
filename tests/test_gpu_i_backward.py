"""Parity of the training backward of the two projections (fo_col_linear_backward:
Flash-RS for dX; fo_row_linear_backward: Flash-AG for dH; local GEMMs for dW) against
the oracle.  Integer inputs are bit-exact; Gaussian inputs use the parity tolerance."""
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


def _gen(g, shape, integer, std=1.0):
    return wl.integer_bf16(g, shape) if integer else wl.gaussian_bf16(g, shape, std)


def _cmp(got, ref, integer, what):
    for i, (x, y) in enumerate(zip(got, ref)):
        if integer:
            assert_bits_equal(to_bits(x), y, f"{what} {i}")
        else:
            assert_close(f64(to_bits(x)), y, f"{what} {i}")


def _col(ctx, P, m, K, Nr, seed, integer, **kw):
    g = torch.Generator().manual_seed(seed)
    X = [_gen(g, (m, K), integer) for _ in range(P)]
    W = [_gen(g, (Nr, K), integer, wl.W_STD) for _ in range(P)]
    dY = [_gen(g, (P * m, Nr), integer) for _ in range(P)]
    dX = [guarded((m, K), torch.bfloat16) for _ in range(P)]
    dW = [guarded((Nr, K), torch.bfloat16) for _ in range(P)]
    ctx.col_linear_backward([to_dev(x) for x in X], [to_dev(w) for w in W], [to_dev(d) for d in dY], dX, dW, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    rdx, rdw = ops.col_linear_backward([f64(x) for x in X], [f64(w) for w in W], [f64(d) for d in dY])
    _cmp(dX, rdx, integer, "dX")
    _cmp(dW, rdw, integer, "dW")


def _row(ctx, P, m, Fr, N, seed, integer, **kw):
    g = torch.Generator().manual_seed(seed)
    H = [_gen(g, (P * m, Fr), integer) for _ in range(P)]
    W = [_gen(g, (N, Fr), integer, wl.W_STD) for _ in range(P)]
    dZ = [_gen(g, (m, N), integer) for _ in range(P)]
    dH = [guarded((P * m, Fr), torch.bfloat16) for _ in range(P)]
    dW = [guarded((N, Fr), torch.bfloat16) for _ in range(P)]
    ctx.row_linear_backward([to_dev(h) for h in H], [to_dev(w) for w in W], [to_dev(z) for z in dZ], dH, dW, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    rdh, rdw = ops.row_linear_backward([f64(h) for h in H], [f64(w) for w in W], [f64(z) for z in dZ])
    _cmp(dH, rdh, integer, "dH")
    _cmp(dW, rdw, integer, "dW")


# 128-row slices (P even): two ring steps per SM-pair tile in the all-gather, transposed tiles
# in the reduce-scatter; 256-row slices: SM pairs; P = 3 and ragged K / N / F: single-SM tiles
@pytest.mark.parametrize("P,m,K,Nr", [(2, 128, 256, 256), (4, 256, 384, 512), (3, 128, 200, 136)])
@pytest.mark.parametrize("order", ["flash", "naive", "serial"])
def test_column_parallel_backward_integer_exact(ctx, P, m, K, Nr, order):
    _col(ctx, P, m, K, Nr, 800 + P, True, order=order)


@pytest.mark.parametrize("P,m,Fr,N", [(2, 128, 256, 256), (4, 256, 384, 512), (3, 128, 136, 200)])
@pytest.mark.parametrize("order", ["flash", "serial"])
def test_row_parallel_backward_integer_exact(ctx, P, m, Fr, N, order):
    _row(ctx, P, m, Fr, N, 820 + P, True, order=order)


def test_backward_gaussian(ctx):
    _col(ctx, 4, 512, 1024, 768, 840, False)
    _row(ctx, 4, 512, 768, 1024, 841, False)


def test_single_sm_tiles_match(ctx):
    # both operands of the weight-gradient GEMM and the weight of the collective GEMM are
    # read MN-major; the single-SM kernel stages 128-wide A and 256-wide B blocks of them
    _col(ctx, 4, 256, 384, 512, 850, True, single_sm=True)
    _row(ctx, 4, 256, 384, 512, 851, True, single_sm=True)


@pytest.mark.parametrize("P,m,K,Nr", [(2, 256, 72, 264), (2, 128, 520, 8)])
def test_ragged_transposed_operands(ctx, P, m, K, Nr):
    # MN extents that end inside a 64-wide box (the box's tail reads zeros) and one block
    # of only 8 columns
    _col(ctx, P, m, K, Nr, 860 + K, True)
    _row(ctx, P, m, Nr, K, 870 + K, True)
