"""Parity of the Flash all-to-all (FlashOverlap technical summary, section 2, "Flash
All-to-All") against the oracle: fo_gemm_a2a (a GEMM whose output blocks belong to
other ranks) and fo_a2a_gemm (the all-to-all in front of a GEMM whose K chunks come
from every rank).  Integer inputs are bit-exact; Gaussian inputs use the tolerance of
the other parity tests."""
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


def _gen(seed, integer, shapes, std):
    g = torch.Generator().manual_seed(seed)
    if integer:
        return [wl.integer_bf16(g, s) for s in shapes]
    return [wl.gaussian_bf16(g, s, sd) for s, sd in zip(shapes, std)]


def _check(got, ref, integer, what):
    for d, (x, y) in enumerate(zip(got, ref)):
        if integer:
            assert_bits_equal(to_bits(x), y, f"{what} rank {d}")
        else:
            assert_close(f64(to_bits(x)), y, f"{what} rank {d}")


def _gemm_a2a(ctx, P, m, K, Nb, seed, integer, **kw):
    X = _gen(seed, integer, [(m, K)] * P, [1.0] * P)
    W = _gen(seed + 1, integer, [(P * Nb, K)] * P, [wl.W_STD] * P)
    Y = [guarded((P * m, Nb), torch.bfloat16) for _ in range(P)]
    ctx.gemm_a2a([to_dev(x) for x in X], [to_dev(w) for w in W], Y, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    ref = ops.gemm_a2a_definition([f64(x) for x in X], [f64(w) for w in W])
    _check(Y, ref, integer, "gemm->a2a")


def _a2a_gemm(ctx, P, m, Kc, N, seed, integer, **kw):
    C = _gen(seed, integer, [(P * m, Kc)] * P, [1.0] * P)
    W = _gen(seed + 1, integer, [(N, P * Kc)] * P, [wl.W_STD] * P)
    Y = [guarded((m, N), torch.bfloat16) for _ in range(P)]
    ctx.a2a_gemm([to_dev(c) for c in C], [to_dev(w) for w in W], Y, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    ref = ops.a2a_gemm_definition([f64(c) for c in C], [f64(w) for w in W])
    _check(Y, ref, integer, "a2a->gemm")


# (P, m, K, Nb): 128-row slices run single-SM tiles, 256-row slices SM pairs; Nb = 384
# leaves a ragged 128-column last tile
SHAPES_PROD = [(2, 128, 256, 256), (4, 256, 512, 384), (3, 128, 192, 128)]
SHAPES_CONS = [(2, 128, 128, 256), (4, 256, 192, 512), (3, 128, 64, 320)]


@pytest.mark.parametrize("P,m,K,Nb", SHAPES_PROD)
@pytest.mark.parametrize("order", ["flash", "naive", "serial"])
def test_gemm_a2a_integer_exact(ctx, P, m, K, Nb, order):
    _gemm_a2a(ctx, P, m, K, Nb, 700 + P, True, order=order)


@pytest.mark.parametrize("P,m,Kc,N", SHAPES_CONS)
@pytest.mark.parametrize("order", ["flash", "naive", "serial"])
def test_a2a_gemm_integer_exact(ctx, P, m, Kc, N, order):
    _a2a_gemm(ctx, P, m, Kc, N, 720 + P, True, order=order)


def test_gemm_a2a_gaussian(ctx):
    _gemm_a2a(ctx, 4, 512, 1024, 768, 740, False)


def test_a2a_gemm_gaussian(ctx):
    _a2a_gemm(ctx, 4, 512, 256, 1024, 750, False)


def test_single_sm_tiles_match(ctx):
    _a2a_gemm(ctx, 4, 256, 192, 512, 760, True, single_sm=True)
    _gemm_a2a(ctx, 4, 256, 512, 384, 770, True, single_sm=True)


def test_a2a_rejects_bad_shapes(ctx):
    import overlapped_tensor_gemm_gb300 as fo
    C = [torch.zeros((256, 100), dtype=torch.bfloat16, device="cuda") for _ in range(2)]  # Kc % 64 != 0
    W = [torch.zeros((128, 200), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Y = [torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(fo.FoError) as e:
        ctx.a2a_gemm(C, W, Y)
    assert e.value.status == fo.FO_ERR_UNSUPPORTED
