"""Parity of query-split attention (fo_qsplit_attn) against the oracle's two-pass fp64
definition and its ring simulation (FlashOverlap technical summary, section 2)."""
import numpy as np
import pytest
import torch

import fo_workloads as wl
from helpers import assert_close, f64, to_bits, to_dev, guarded
from oracle import bf16, ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import overlapped_tensor_gemm_gb300 as fo
    c = fo.Context(0)
    yield c
    c.close()


def _attn(ctx, P, m, H, seed, causal=True, **kw):
    inp = wl.attn_inputs(P, P * m, H, 128, seed)
    Q = [to_dev(x).reshape(m, H * 128) for x in inp["Q"]]
    K = [to_dev(x).reshape(m, H * 128) for x in inp["K"]]
    V = [to_dev(x).reshape(m, H * 128) for x in inp["V"]]
    O = [guarded((m, H * 128), torch.bfloat16) for _ in range(P)]
    ctx.qsplit_attn(Q, K, V, O, heads=H, head_dim=128, causal=causal, **kw)
    torch.cuda.synchronize()
    ctx.poll()
    got = [f64(to_bits(o)).reshape(m, H, 128) for o in O]
    return inp, got


@pytest.mark.parametrize("P,m,H", [(1, 128, 1), (2, 128, 2), (4, 256, 3), (3, 384, 2), (2, 768, 2), (1, 512, 1)])
def test_attention_matches_definition(ctx, P, m, H):
    inp, got = _attn(ctx, P, m, H, 300 + P)
    ref = ops.attention_definition(np.concatenate([f64(x) for x in inp["Q"]]),
                                   np.concatenate([f64(x) for x in inp["K"]]),
                                   np.concatenate([f64(x) for x in inp["V"]]))
    assert_close(np.concatenate(got), ref, f"attention P={P}")


@pytest.mark.parametrize("m", [128, 256])
def test_attention_matches_ring_simulation_pruned(ctx, m):
    P, H = 4, 2
    inp, got = _attn(ctx, P, m, H, 41, causal_prune=True)
    ref, _ = ops.qsplit_attention_ring([f64(x) for x in inp["Q"]], [f64(x) for x in inp["K"]],
                                       [f64(x) for x in inp["V"]], prune=True)
    for r in range(P):
        assert_close(got[r], ref[r], f"pruned ring rank {r}")


@pytest.mark.parametrize("causal", [True, False])
def test_attention_several_items_per_cta(ctx, causal):
    # a grid of 3 CTAs: every CTA walks several (rank, query block, head) items, so the
    # producer's look-ahead crosses item boundaries (next Q while the last blocks run)
    P, m, H = 2, 384, 2
    inp, got = _attn(ctx, P, m, H, 44, causal=causal, num_sms=3)
    ref = ops.attention_definition(np.concatenate([f64(x) for x in inp["Q"]]),
                                   np.concatenate([f64(x) for x in inp["K"]]),
                                   np.concatenate([f64(x) for x in inp["V"]]), causal=causal)
    assert_close(np.concatenate(got), ref, f"attention, 3 CTAs, causal={causal}")


def test_attention_non_causal(ctx):
    P, m, H = 2, 256, 2
    inp, got = _attn(ctx, P, m, H, 42, causal=False)
    ref = ops.attention_definition(np.concatenate([f64(x) for x in inp["Q"]]),
                                   np.concatenate([f64(x) for x in inp["K"]]),
                                   np.concatenate([f64(x) for x in inp["V"]]), causal=False)
    assert_close(np.concatenate(got), ref, "non-causal attention")


@pytest.mark.parametrize("m", [128, 384])
def test_attention_constant_v_is_exact(ctx, m):
    # closed form: a constant V gives that constant at every query
    P, H = 2, 1
    inp = wl.attn_inputs(P, P * m, H, 128, 43)
    c = wl.gaussian_bf16(torch.Generator().manual_seed(5), (1, H, 128))
    V = [np.repeat(c, m, axis=0) for _ in range(P)]
    Q = [to_dev(x).reshape(m, H * 128) for x in inp["Q"]]
    K = [to_dev(x).reshape(m, H * 128) for x in inp["K"]]
    Vd = [to_dev(x).reshape(m, H * 128) for x in V]
    O = [torch.empty((m, H * 128), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ctx.qsplit_attn(Q, K, Vd, O, heads=H, head_dim=128)
    torch.cuda.synchronize()
    want = np.repeat(c.reshape(1, -1), m, axis=0)
    for r in range(P):
        got = to_bits(O[r])
        # one bf16 ulp allowed: the weights' sum and the P.V accumulation round differently
        assert np.abs(f64(got) - f64(want)).max() <= np.abs(f64(want)).max() * 2 ** -7


def test_attention_v_beyond_fp16_range_reports_range_error(ctx):
    """V enters the P.V product as fp16: a finite |v| above 65504 cannot be represented,
    so the call must end with FO_ERR_RANGE from poll (no GPU fault, the context stays
    usable); 65280, the largest bf16 value that fp16 holds, is accepted."""
    import overlapped_tensor_gemm_gb300 as fo
    P, m, H = 2, 128, 1
    inp = wl.attn_inputs(P, P * m, H, 128, 52)
    Q = [to_dev(x).reshape(m, H * 128) for x in inp["Q"]]
    K = [to_dev(x).reshape(m, H * 128) for x in inp["K"]]
    V = [to_dev(x).reshape(m, H * 128) for x in inp["V"]]
    O = [torch.empty((m, H * 128), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    V[1][5, 17] = 65280.0                       # below 65504, exact in bf16 and fp16: accepted
    ctx.qsplit_attn(Q, K, V, O, heads=H, head_dim=128)
    torch.cuda.synchronize()
    ctx.poll()
    V[1][7, 3] = 65536.0                        # the next bf16 value, beyond fp16: reported
    ctx.qsplit_attn(Q, K, V, O, heads=H, head_dim=128)
    torch.cuda.synchronize()
    with pytest.raises(fo.FoError) as e:
        ctx.poll()
    assert e.value.status == fo.FO_ERR_RANGE
    V[1][7, 3] = 0.5                            # the context computes correctly afterwards
    _, got = _attn_with(ctx, Q, K, V, P, m, H)
    ref = ops.attention_definition(np.concatenate([f64(to_bits(q)) for q in Q]).reshape(P * m, H, 128),
                                   np.concatenate([f64(to_bits(k)) for k in K]).reshape(P * m, H, 128),
                                   np.concatenate([f64(to_bits(v)) for v in V]).reshape(P * m, H, 128))
    assert_close(np.concatenate(got), ref, "attention after a range error")


def _attn_with(ctx, Q, K, V, P, m, H):
    O = [guarded((m, H * 128), torch.bfloat16) for _ in range(P)]
    ctx.qsplit_attn(Q, K, V, O, heads=H, head_dim=128)
    torch.cuda.synchronize()
    ctx.poll()
    return None, [f64(to_bits(o)).reshape(m, H, 128) for o in O]
