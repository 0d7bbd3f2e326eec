"""Parity of the tcgen05 GEMM core (fo_gemm) against the oracle: bit-exact on
integer-valued bf16 inputs, within tolerance on Gaussian inputs; single tile,
several tiles and k-blocks, ragged M/N/K tails, fp32 output."""
import numpy as np
import pytest
import torch

import fo_workloads as wl
from helpers import assert_bits_equal, assert_close, f64, padded, to_bits, to_dev
from oracle import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import overlapped_tensor_gemm_gb300 as fo
    c = fo.Context(0)
    yield c
    c.close()


def _run_gemm(ctx, M, N, K, integer, out_dtype=torch.bfloat16, seed=0):
    g = torch.Generator().manual_seed(seed)
    if integer:
        A = wl.integer_bf16(g, (M, K))
        B = wl.integer_bf16(g, (N, K))
    else:
        A = wl.gaussian_bf16(g, (M, K))
        B = wl.gaussian_bf16(g, (N, K), 0.02)
    C = padded(M, N, out_dtype)
    ctx.gemm(to_dev(A), to_dev(B), C)
    torch.cuda.synchronize()
    ctx.poll()
    ref = ops.gemm(f64(A), f64(B))
    return C, ref


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (128, 256, 512), (256, 512, 128), (384, 768, 1024)])
def test_gemm_integer_bit_exact(ctx, M, N, K):
    C, ref = _run_gemm(ctx, M, N, K, integer=True)
    assert_bits_equal(to_bits(C), ref, f"gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (512, 768, 1024), (1024, 1000, 264)])
def test_sm_pair_tiles_match_single_sm_tiles(ctx, M, N, K):
    """256x256 tiles on SM pairs (tcgen05 cta_group::2) give the same bits as the
    single-SM 128x256 tiles, and both match the oracle on integer inputs."""
    g = torch.Generator().manual_seed(M + N + K)
    A = wl.integer_bf16(g, (M, K))
    B = wl.integer_bf16(g, (N, K))
    C1 = padded(M, N, torch.bfloat16)
    C2 = padded(M, N, torch.bfloat16)
    ctx.gemm(to_dev(A), to_dev(B), C1)                      # rows % 256 == 0: SM pairs
    ctx.gemm(to_dev(A), to_dev(B), C2, single_sm=True)
    torch.cuda.synchronize()
    ctx.poll()
    ref = ops.gemm(f64(A), f64(B))
    assert_bits_equal(to_bits(C1), ref, "pair tiles")
    assert_bits_equal(to_bits(C2), ref, "single-SM tiles")


@pytest.mark.parametrize("M,N,K", [(200, 300, 136), (1, 8, 8), (129, 257, 72), (64, 1000, 200)])
def test_gemm_ragged_integer(ctx, M, N, K):
    C, ref = _run_gemm(ctx, M, N, K, integer=True, seed=1)
    assert_bits_equal(to_bits(C), ref, f"gemm {M}x{N}x{K}")


def test_gemm_fp32_output_exact(ctx):
    C, ref = _run_gemm(ctx, 256, 512, 320, integer=True, out_dtype=torch.float32, seed=2)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)


def test_gemm_gaussian_tolerance(ctx):
    C, ref = _run_gemm(ctx, 512, 1024, 2048, integer=False, seed=3)
    assert_close(f64(to_bits(C)), ref, "gemm gaussian")


def test_gemm_many_tiles_and_persistence(ctx):
    # more tiles than SMs: every CTA walks several tiles and reuses both accumulators
    C, ref = _run_gemm(ctx, 2048, 4096, 256, integer=True, seed=4)
    assert_bits_equal(to_bits(C), ref, "gemm 2048x4096x256")
