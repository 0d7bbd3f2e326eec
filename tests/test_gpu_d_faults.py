"""Failure detection without a GPU fault: the host skips one ring hop (fault
injection on the host), so a device wait runs past its short limit; the kernel
returns, fo_ctx_poll reports FO_ERR_TIMEOUT, and the context stays usable."""
import pytest
import torch

import fo_workloads as wl
from helpers import assert_bits_equal, f64, to_bits, to_dev
from oracle import ops

pytestmark = pytest.mark.gpu


def _inputs(P, m, K, N):
    inp = wl.ag_inputs(P, m, K, N, 77, True)
    X = [to_dev(x) for x in inp["X_shards"]]
    W = [to_dev(w) for w in inp["W_col"]]
    Y = [torch.zeros((P * m, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    return inp, X, W, Y


def test_skipped_hop_times_out_and_context_recovers():
    import overlapped_tensor_gemm_gb300 as fo
    P, m, K, N = 4, 128, 256, 256
    inp, X, W, Y = _inputs(P, m, K, N)
    with fo.Context(0) as ctx:
        ctx.ag_gemm(X, W, Y, fault="skip_hop", timeout_us=20000)
        torch.cuda.synchronize()
        with pytest.raises(fo.FoError) as e:
            ctx.poll()
        assert e.value.status == fo.FO_ERR_TIMEOUT
        ctx.poll()  # cleared
        # the same context computes the right answer afterwards
        ctx.ag_gemm(X, W, Y)
        torch.cuda.synchronize()
        ctx.poll()
        ref, _ = ops.ag_gemm_ring([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]])
        for r in range(P):
            assert_bits_equal(to_bits(Y[r]), ref[r], f"after recovery rank {r}")


@pytest.mark.parametrize("m", [128, 384])
def test_skipped_kv_hop_times_out_in_attention(m):
    import overlapped_tensor_gemm_gb300 as fo
    P, H = 3, 1
    inp = wl.attn_inputs(P, P * m, H, 128, 78)
    Q = [to_dev(x).reshape(m, 128) for x in inp["Q"]]
    K = [to_dev(x).reshape(m, 128) for x in inp["K"]]
    V = [to_dev(x).reshape(m, 128) for x in inp["V"]]
    O = [torch.zeros((m, 128), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    with fo.Context(0) as ctx:
        ctx.qsplit_attn(Q, K, V, O, heads=H, head_dim=128, fault="skip_hop", timeout_us=20000)
        torch.cuda.synchronize()
        with pytest.raises(fo.FoError) as e:
            ctx.poll()
        assert e.value.status == fo.FO_ERR_TIMEOUT
        ctx.qsplit_attn(Q, K, V, O, heads=H, head_dim=128)
        torch.cuda.synchronize()
        ctx.poll()
    # the recovered context computes what a fresh one does (every item of the launch ran)
    O2 = [torch.zeros((m, 128), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    with fo.Context(0) as ctx2:
        ctx2.qsplit_attn(Q, K, V, O2, heads=H, head_dim=128)
        torch.cuda.synchronize()
        ctx2.poll()
    for r in range(P):
        assert torch.equal(O[r].view(torch.int16), O2[r].view(torch.int16)), f"attention after recovery, rank {r}"


def test_skipped_all_to_all_hop_times_out_and_context_recovers():
    import overlapped_tensor_gemm_gb300 as fo
    P, m, Kc, N = 3, 128, 64, 256
    g = torch.Generator().manual_seed(79)
    C = [to_dev(wl.integer_bf16(g, (P * m, Kc))) for _ in range(P)]
    W = [to_dev(wl.integer_bf16(g, (N, P * Kc))) for _ in range(P)]
    Y = [torch.zeros((m, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    with fo.Context(0) as ctx:
        ctx.a2a_gemm(C, W, Y, fault="skip_hop", timeout_us=20000)
        torch.cuda.synchronize()
        with pytest.raises(fo.FoError) as e:
            ctx.poll()
        assert e.value.status == fo.FO_ERR_TIMEOUT
        ctx.a2a_gemm(C, W, Y)
        torch.cuda.synchronize()
        ctx.poll()


def test_host_layer_with_skipped_hop_releases_its_copies():
    # The host-buffer layer copies each rank's output back on a link stream that waits for
    # the reduce-scatter's completion counter of that rank.  With a skipped all-gather hop
    # the GEMMs give up; the counters' final values, written on the stream after the
    # reduce-scatter launch, still release those copies, so the call completes.
    import time

    import overlapped_tensor_gemm_gb300 as fo
    cfg = wl.MLPConfig("host-f", 70, P=4, tokens=1024, hidden=256, ffn=512, gated=False, integer=True)
    inp = wl.mlp_inputs(cfg)
    Xh = [to_dev(x, "cpu").pin_memory() for x in inp["X_shards"]]
    Wc = [to_dev(w) for w in inp["W_col"]]
    Wr = [to_dev(w) for w in inp["W_row"]]
    Zh = [torch.empty((cfg.m, cfg.hidden), dtype=torch.bfloat16).pin_memory() for _ in range(cfg.P)]
    with fo.Context(0) as ctx:
        ctx.mlp_layer_host(Xh, Wc, Wr, Zh, gated=False, fault="skip_hop", timeout_us=20000)
        done = torch.cuda.Event()
        done.record()
        deadline = time.time() + 30.0
        while not done.query():
            assert time.time() < deadline, "a copy back to the host was not released"
            time.sleep(0.005)
        with pytest.raises(fo.FoError) as e:
            ctx.poll()
        assert e.value.status == fo.FO_ERR_TIMEOUT
        ctx.poll()
        ctx.mlp_layer_host(Xh, Wc, Wr, Zh, gated=False)
        torch.cuda.synchronize()
        ctx.poll()
        _, _, ref = ops.mlp_layer([f64(x) for x in inp["X_shards"]], [f64(w) for w in inp["W_col"]],
                                  [f64(w) for w in inp["W_row"]], gated=False)
        for r in range(cfg.P):
            assert_bits_equal(to_bits(Zh[r]), ref[r], f"host layer after recovery rank {r}")
