"""The MLP layer from host memory (fo_mlp_layer_host: activations in pinned or pageable
host buffers, uploaded slice by slice ahead of their Flash-AG GEMMs, the output copied
back) against the oracle, through the C ABI.  Integer inputs are bit-exact; Gaussian
inputs use the parity tolerance."""
import pytest
import torch

import fo_workloads as wl
from helpers import assert_bits_equal, assert_close, f64, to_bits, to_dev
from oracle import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import overlapped_tensor_gemm_gb300 as fo
    c = fo.Context(0)
    yield c
    c.close()


def _run(ctx, cfg, pinned, **kw):
    inp = wl.mlp_inputs(cfg)
    Xh = [to_dev(x, "cpu") for x in inp["X_shards"]]
    if pinned:
        Xh = [x.pin_memory() for x in Xh]
    Wc = [to_dev(w) for w in inp["W_col"]]
    Wr = [to_dev(w) for w in inp["W_row"]]
    Zh = [torch.full((cfg.m, cfg.hidden), float("nan"), dtype=torch.bfloat16) for _ in range(cfg.P)]
    if pinned:
        Zh = [z.pin_memory() for z in Zh]
    ctx.mlp_layer_host(Xh, Wc, Wr, Zh, gated=cfg.gated, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    _, _, ref = ops.mlp_layer([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]],
                              [f64(w) for w in inp["W_row"]], gated=cfg.gated)
    return Zh, ref


# P = 1 (no ring: only the upload of the own slice), 2, 4 (pair tiles at 256 rows per rank)
@pytest.mark.parametrize("P,tokens", [(1, 128), (2, 256), (4, 1024), (3, 384)])
@pytest.mark.parametrize("order", ["flash", "serial", "slicing"])
def test_host_layer_integer_exact(ctx, P, tokens, order):
    if order == "slicing" and (tokens // P) % P != 0:
        pytest.skip("equal slices need m divisible by P")
    cfg = wl.MLPConfig("host", 40 + P, P=P, tokens=tokens, hidden=256, ffn=768, gated=False, integer=True)
    Zh, ref = _run(ctx, cfg, True, order=order)
    for r in range(P):
        assert_bits_equal(to_bits(Zh[r]), ref[r], f"host layer {order} P={P} rank {r}")


def test_host_layer_pageable_and_gaussian(ctx):
    cfg = wl.MLPConfig("host-g", 50, P=4, tokens=1024, hidden=512, ffn=1024, gated=True, integer=False)
    Zh, ref = _run(ctx, cfg, False)
    for r in range(cfg.P):
        assert_close(f64(to_bits(Zh[r])), ref[r], f"host layer gaussian rank {r}")


def test_host_layer_repeated_calls(ctx):
    # back-to-back calls reuse the device buffers: each call's uploads must follow the
    # previous call's readers, and its flags its own epoch
    cfg = wl.MLPConfig("host-r", 60, P=4, tokens=1024, hidden=256, ffn=512, gated=False, integer=True)
    inp = wl.mlp_inputs(cfg)
    Xh = [to_dev(x, "cpu").pin_memory() for x in inp["X_shards"]]
    Wc = [to_dev(w) for w in inp["W_col"]]
    Wr = [to_dev(w) for w in inp["W_row"]]
    _, _, ref = ops.mlp_layer([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]],
                              [f64(w) for w in inp["W_row"]], gated=False)
    outs = []
    for _ in range(3):
        Zh = [torch.empty((cfg.m, cfg.hidden), dtype=torch.bfloat16).pin_memory() for _ in range(cfg.P)]
        ctx.mlp_layer_host(Xh, Wc, Wr, Zh, gated=False)
        outs.append(Zh)
    torch.cuda.synchronize()
    ctx.poll()
    for Zh in outs:
        for r in range(cfg.P):
            assert_bits_equal(to_bits(Zh[r]), ref[r], f"repeated host layer rank {r}")
