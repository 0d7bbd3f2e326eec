"""fo_gemm_rs_noalloc: Flash-RS for callers that cannot allocate device memory.

Such callers own all of their device memory through their own allocator, or run
a latency-critical path that must not pay the device-wide synchronisation of
cudaMalloc/cudaFree.  The entry point keeps its scratch in a fixed device array
inside the library; the caller passes only inputs and outputs.  Called here
through the C ABI:
  * its output is bit-identical to fo_gemm_rs (the same kernel, the same tile
    order) on two calls in a row -- the second call reuses the array the first
    left behind, and a differently shaped call in between must not disturb it;
  * on integer-valued inputs (every partial sum exact in fp32) it equals the
    oracle's reduce-scatter bit for bit, including ragged shapes (rows and
    columns that fill no whole tile) and P = 1, 2, 8.
This file is collected last so that a failure here stops a -x run only after
every other test has run."""
import ctypes

import numpy as np
import pytest
import torch

import fo_workloads as wl
from helpers import assert_bits_equal, f64, to_bits, to_dev, guarded
from oracle import ops

pytestmark = pytest.mark.gpu


def _mats(fo, ts):
    arr = (fo.FoMat * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = fo.mat(t)
    return arr


def _noalloc(fo, lib, X, W, Y, timeout_us=0):
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.fo_gemm_rs_noalloc(_mats(fo, X), _mats(fo, W), len(X), _mats(fo, Y), timeout_us,
                                ctypes.c_void_p(status.data_ptr()), stream)
    assert st == fo.FO_OK, lib.fo_last_error_string()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"


def _inputs(P, m, Kr, N, seed, integer):
    inp = wl.rs_inputs(P, P * m, N, Kr, seed, integer=integer)
    return inp, [to_dev(x) for x in inp["X"]], [to_dev(w) for w in inp["W_row"]]


def test_noalloc_bit_identical_to_fo_gemm_rs_twice_in_a_row():
    import overlapped_tensor_gemm_gb300 as fo
    lib = fo.load()
    P, m, Kr, N = 4, 256, 512, 512
    with fo.Context(0) as ctx:
        for seed in (501, 502):
            _, X, W = _inputs(P, m, Kr, N, seed, integer=False)
            Y_ref = [torch.empty((m, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
            Y_new = [guarded((m, N), torch.bfloat16) for _ in range(P)]
            ctx.gemm_rs(X, W, Y_ref)
            torch.cuda.synchronize()
            ctx.poll()
            _noalloc(fo, lib, X, W, Y_new)
            for r in range(P):
                assert torch.equal(Y_new[r].view(torch.int16), Y_ref[r].view(torch.int16)), f"rank {r}"


@pytest.mark.parametrize("P,m,Kr,N", [(1, 200, 64, 260), (2, 200, 136, 260), (8, 72, 200, 516),
                                      (4, 256, 512, 512)])
def test_noalloc_integer_bit_exact_vs_oracle(P, m, Kr, N):
    """Ragged rows and columns, P = 1, 2, 4, 8; each shape is run twice in a row with
    different inputs, so the second call sees the first call's flags and slots."""
    import overlapped_tensor_gemm_gb300 as fo
    lib = fo.load()
    for seed in (601, 602):
        inp, X, W = _inputs(P, m, Kr, N, seed + P, integer=True)
        Y = [guarded((m, N), torch.bfloat16) for _ in range(P)]
        _noalloc(fo, lib, X, W, Y, timeout_us=500000)
        ref = ops.gemm_rs_definition([ops.split_chunks(f64(x), P) for x in inp["X"]],
                                     [f64(w) for w in inp["W_row"]])
        for d in range(P):
            assert_bits_equal(to_bits(Y[d]), ref[d], f"no-alloc P={P} m={m} N={N} rank {d}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import overlapped_tensor_gemm_gb300 as fo
    lib = fo.load()
    P, m, Kr, N = 4, 1024, 64, 4096          # receive slots: 12 * 1024 * 4096 * 4 B = 192 MiB > 64 MiB
    X = [torch.zeros((P * m, Kr), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    W = [torch.zeros((N, Kr), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    Y = [torch.zeros((m, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    st = lib.fo_gemm_rs_noalloc(_mats(fo, X), _mats(fo, W), P, _mats(fo, Y), 0, None,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == fo.FO_ERR_UNSUPPORTED
    assert b"static scratch" in lib.fo_last_error_string()
