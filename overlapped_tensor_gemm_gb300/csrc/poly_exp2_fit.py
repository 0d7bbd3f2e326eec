"""Derivation of the cubic used by the attention kernel's FMA-pipe exp2.

2^x = 2^floor(x) * 2^f with f = x - floor(x) in [0, 1) (Cody-Waite style range
reduction); 2^f is approximated by the cubic c0 + c1 f + c2 f^2 + c3 f^3 whose
coefficients minimise the relative error in the least-squares sense at 2000
Chebyshev nodes of [0, 1].  Maximum relative error ~7.7e-5, below half an fp16
ulp (2^-12 ~ 2.4e-4) of the softmax weights it produces.

Run:  python overlapped_tensor_gemm_gb300/csrc/poly_exp2_fit.py
"""
import numpy as np


def fit(degree: int = 3, nodes: int = 2000):
    k = np.arange(nodes)
    f = 0.5 - 0.5 * np.cos(np.pi * (k + 0.5) / nodes)
    y = 2.0 ** f
    V = np.vander(f, degree + 1, increasing=True)
    c, *_ = np.linalg.lstsq(V / y[:, None], np.ones_like(y), rcond=None)
    grid = np.linspace(0.0, 1.0, 200001)
    err = np.abs(np.polyval(c[::-1], grid) / 2.0 ** grid - 1.0).max()
    return c, err


if __name__ == "__main__":
    c, err = fit()
    print("coefficients:", ", ".join(f"{x:.8f}f" for x in c))
    print(f"max relative error: {err:.3e}")
