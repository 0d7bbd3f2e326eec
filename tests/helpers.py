"""Shared helpers of the GPU parity tests (CPU side: bf16 bit transfers, tolerances)."""
import numpy as np
import torch

from oracle import bf16

# Tolerance for Gaussian bf16 inputs with fp32 accumulation (relative L2 and
# max-abs relative to the largest reference magnitude).
REL_L2 = 2e-3
MAX_ABS_FRAC = 1e-2
# A block that chains three operations with bf16-rounded outputs (the attention block: QKV
# projection, attention, output projection) rounds at three points; at each the two sides'
# pre-rounding values may fall on either side of a bf16 boundary.  Independent rounding
# stages add in quadrature: the per-operation bound times sqrt(3).
REL_L2_THREE_STAGES = REL_L2 * 3 ** 0.5


def to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16)
    return t.to(device)


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f64(bits) -> np.ndarray:
    return bf16.to_f64(bits)


def assert_bits_equal(got_bits: np.ndarray, ref_f64: np.ndarray, what: str = ""):
    ref_bits = bf16.from_f64(ref_f64)
    diff = np.nonzero(got_bits != ref_bits)
    if diff[0].size:
        i = tuple(d[0] for d in diff)
        raise AssertionError(f"{what}: {diff[0].size} of {got_bits.size} elements differ; first at {i}: "
                             f"got {bf16.to_f64(got_bits[i])} want {ref_f64[i]}")


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "", round_ref: bool = True, rel_l2: float = REL_L2):
    """Tolerance check of a bf16 result; the reference is rounded to bf16 (the
    operation's output type) unless round_ref is False."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if round_ref:
        ref = bf16.round_f64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    num = np.linalg.norm(got - ref)
    den = np.linalg.norm(ref) or 1.0
    rel = num / den
    mx = np.abs(got - ref).max() if got.size else 0.0
    lim = MAX_ABS_FRAC * (np.abs(ref).max() if ref.size else 0.0)
    assert rel <= rel_l2, f"{what}: rel-L2 {rel:.3e} > {rel_l2}"
    assert mx <= lim, f"{what}: max-abs {mx:.3e} > {lim:.3e}"


# Output buffers whose surroundings are checked after every test (see check_guards).
_GUARDED = []


def guarded(shape, dtype, device="cuda"):
    """A [rows, cols] output view inside a NaN-filled buffer: the row pitch carries at
    least 16 bytes of padding and one guard row sits above and one below the view.
    check_guards(), run after every test, asserts that all of them are still NaN -- a
    cheap canary for out-of-bounds writes of the kernels."""
    rows, cols = shape
    esz = torch.empty((), dtype=dtype).element_size()
    per = 16 // esz
    ld = (cols + per - 1) // per * per + per
    base = torch.full((rows + 2, ld), float("nan"), dtype=dtype, device=device)
    _GUARDED.append((base, rows, cols))
    return base[1:rows + 1, :cols]


def padded(rows: int, cols: int, dtype, fill=float("nan"), device="cuda"):
    """[rows, cols] view of a NaN-filled buffer with a padded row pitch and guard rows
    (guarded()); `fill` is kept for the call sites' readability and must be NaN."""
    assert fill != fill, "the canary needs a NaN fill"
    return guarded((rows, cols), dtype, device)


def check_guards():
    """Asserts that the padding and guard rows of every guarded() buffer of the test that
    just ran are untouched, then forgets the buffers."""
    bad = []
    try:
        for base, rows, cols in _GUARDED:
            pad = base[1:rows + 1, cols:]
            ok = bool(torch.isnan(base[0]).all()) and bool(torch.isnan(base[rows + 1]).all())
            ok = ok and (pad.numel() == 0 or bool(torch.isnan(pad).all()))
            if not ok:
                bad.append((rows, cols))
    finally:
        _GUARDED.clear()
    assert not bad, f"out-of-bounds write next to output buffers of shape {bad}"
