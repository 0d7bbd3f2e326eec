"""Pins of the oracle's attention block (FlashOverlap technical summary, section 2,
architectural instantiations: the QKV projection is the column-parallel GEMM after the
all-gather, the output projection the row-parallel GEMM before the reduce-scatter).

Each test fixes the composition by something other than the oracle's own formula: the
split of heads over ranks (P=2 against all heads on one rank), closed forms of causal
attention (zero keys give prefix means; the first query sees only the first key), and
the ring decomposition against the undecomposed collectives."""
import numpy as np
import pytest
import torch

from oracle import bf16, ops


def _inputs(P, m, hidden, heads, D, seed):
    rng = np.random.default_rng(seed)
    rb = lambda a: bf16.round_f64(a)  # noqa: E731  values representable in bf16
    X = [rb(rng.standard_normal((m, hidden))) for _ in range(P)]
    Wqkv = [rb(rng.standard_normal((3 * heads * D, hidden)) * 0.2) for _ in range(P)]
    Wo = [rb(rng.standard_normal((hidden, heads * D)) * 0.2) for _ in range(P)]
    return X, Wqkv, Wo


def _merge_heads(Wqkv, Wo, heads, D):
    """The same heads on one rank: Q rows of every rank, then K rows, then V rows; W_o's
    column blocks in the same head order."""
    hd = heads * D
    q = np.concatenate([w[:hd] for w in Wqkv])
    k = np.concatenate([w[hd:2 * hd] for w in Wqkv])
    v = np.concatenate([w[2 * hd:] for w in Wqkv])
    return [np.concatenate([q, k, v])], [np.concatenate(Wo, axis=1)]


def test_heads_split_over_ranks_equals_one_rank_with_all_heads():
    P, m, hidden, heads, D = 2, 8, 16, 2, 4
    X, Wqkv, Wo = _inputs(P, m, hidden, heads, D, 3)
    _, _, Z = ops.attn_layer(X, Wqkv, Wo, heads)
    W1, Wo1 = _merge_heads(Wqkv, Wo, heads, D)
    _, _, Z1 = ops.attn_layer([np.concatenate(X)], W1, Wo1, P * heads)
    # the same fp64 sum in another order before one bf16 rounding: at most one bf16 ulp
    ulp = np.abs(Z1[0]) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(np.concatenate(Z) - Z1[0]) <= ulp)


def test_zero_keys_give_prefix_means_of_v():
    P, m, hidden, heads, D = 2, 6, 8, 2, 4
    X, Wqkv, Wo = _inputs(P, m, hidden, heads, D, 4)
    hd = heads * D
    for w in Wqkv:
        w[hd:2 * hd] = 0.0  # K = 0: every score is 0, causal softmax is uniform over keys <= i
    QKV, O, Z = ops.attn_layer(X, Wqkv, Wo, heads)
    M = P * m
    for r in range(P):
        v = QKV[r][:, 2 * hd:]
        want = np.cumsum(v, axis=0) / np.arange(1, M + 1)[:, None]
        # bf16 rounding of the exact value: within half a bf16 ulp (2^-8 relative)
        assert np.all(np.abs(O[r] - want) <= np.abs(want) * 2.0 ** -8 + 1e-12)


def test_first_token_output_is_its_own_value_projection():
    P, m, hidden, heads, D = 2, 4, 8, 1, 8
    X, Wqkv, Wo = _inputs(P, m, hidden, heads, D, 5)
    QKV, O, Z = ops.attn_layer(X, Wqkv, Wo, heads)
    for r in range(P):
        assert np.array_equal(O[r][0], QKV[r][0, 2 * heads * D:])  # query 0 sees key 0 only
    z0 = sum(O[r][0] @ Wo[r].T for r in range(P))
    assert np.all(np.abs(Z[0][0] - z0) <= np.abs(z0) * 2.0 ** -8 + 1e-12)


def test_attention_of_each_rank_matches_torch_sdpa():
    P, m, hidden, heads, D = 2, 8, 16, 2, 8
    X, Wqkv, Wo = _inputs(P, m, hidden, heads, D, 6)
    QKV, O, _ = ops.attn_layer(X, Wqkv, Wo, heads)
    M, hd = P * m, heads * D
    for r in range(P):
        t = torch.from_numpy(QKV[r])
        q, k, v = (t[:, i * hd:(i + 1) * hd].reshape(M, heads, D).transpose(0, 1) for i in range(3))
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
        ref = ref.transpose(0, 1).reshape(M, hd).numpy()
        assert np.all(np.abs(O[r] - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_ring_decomposition_equals_undecomposed(causal):
    P, m, hidden, heads, D = 3, 4, 8, 1, 4
    X, Wqkv, Wo = _inputs(P, m, hidden, heads, D, 7)
    a = ops.attn_layer(X, Wqkv, Wo, heads, causal=causal)
    b = ops.attn_layer(X, Wqkv, Wo, heads, causal=causal, decomposed=False)
    for x, y in zip(a, b):
        for u, w in zip(x, y):
            assert np.allclose(u, w, rtol=2.0 ** -7, atol=1e-12)
