"""Pins of the oracle's bf16 conversion against a library routine and brute force."""
import numpy as np
import pytest
import torch

from oracle import bf16


def test_decode_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = bf16.to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _torch_bits(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_encode_matches_torch_rne_on_fp32_values():
    rng = np.random.default_rng(0)
    parts = [
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e30).astype(np.float32),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),     # subnormal range
        rng.integers(-70000, 70000, 5000).astype(np.float32),
    ]
    # exact ties: halfway between neighbouring bf16 values (low 16 bits = 0x8000)
    hi = rng.integers(0, 0x7F7F, 5000).astype(np.uint32) << 16
    parts.append((hi | 0x8000).view(np.float32))
    parts.append(((hi | 0x8000) | 0x80000000).view(np.float32))
    parts.append(np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 3.4028235e38, -3.4028235e38,
                           1e-45, -1e-45, 1.1754944e-38], dtype=np.float32))
    x = np.concatenate(parts)
    ours = bf16.from_f64(x.astype(np.float64))
    assert np.array_equal(ours, _torch_bits(x))


def test_encode_nan_is_quiet():
    out = bf16.from_f64(np.array([np.nan, -np.nan]))
    assert out[0] & 0x7FFF == 0x7FC0
    assert np.isnan(bf16.to_f64(out)).all()


def _brute_nearest(x: float, table_vals: np.ndarray, table_bits: np.ndarray) -> int:
    """Nearest finite bf16 by exhaustive search, ties to the even significand."""
    d = np.abs(table_vals - x)
    best = d.min()
    cand = table_bits[d == best]
    if len(cand) == 1:
        return int(cand[0])
    even = [int(b) for b in cand if (int(b) & 1) == 0]
    assert len(even) == 1
    return even[0]


def test_encode_fp64_values_by_brute_force():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bf16.to_f64(bits)
    keep = np.isfinite(vals) & ~((bits == 0x8000))          # one zero is enough
    tv, tb = vals[keep], bits[keep]
    rng = np.random.default_rng(1)
    xs = list(rng.standard_normal(300) * 10.0 ** rng.integers(-30, 30, 300))
    # fp64 values just above / below exact ties (not representable in fp32)
    for b in rng.integers(0x0080, 0x7F00, 100):
        lo = bf16.to_f64(np.array([b], np.uint16))[0]
        hi = bf16.to_f64(np.array([b + 1], np.uint16))[0]
        mid = (lo + hi) / 2
        xs += [mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)]
    for x in xs:
        assert int(bf16.from_f64(np.array([x]))[0]) == _brute_nearest(x, tv, tb), x


@pytest.mark.parametrize("x,expect", [(1.0, 0x3F80), (-2.0, 0xC000), (1.0 + 2 ** -8, 0x3F80),
                                      (1.0 + 3 * 2 ** -8, 0x3F82), (3.5e38, 0x7F80)])
def test_encode_textbook_values(x, expect):
    # 1 + 2^-8 is the tie between 1.0 (even) and 1 + 2^-7; 1 + 3*2^-8 ties up to the even 1 + 2^-6
    assert int(bf16.from_f64(np.array([x]))[0]) == expect
