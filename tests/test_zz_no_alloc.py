"""fo_gemm_rs_noalloc: Flash-RS for callers that cannot allocate device memory
(their memory belongs to their own allocator, or their path must not pay the
synchronisation of cudaMalloc/cudaFree).  Its scratch is a fixed device array in
the library.  Called through the C ABI; its output must match fo_gemm_rs on two
calls in a row (the second reuses the array the first left behind)."""
import ctypes

import numpy as np
import pytest
import torch

import fo_workloads as wl
from helpers import assert_close, f64, to_bits, to_dev

pytestmark = pytest.mark.gpu


def _mats(fo, ts):
    arr = (fo.FoMat * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = fo.mat(t)
    return arr


def _run_pair(fo, lib, ctx, P, m, Kr, N, seed):
    inp = wl.rs_inputs(P, P * m, N, Kr, seed, integer=False)
    X = [to_dev(x) for x in inp["X"]]
    W = [to_dev(w) for w in inp["W_row"]]
    Y_ref = [torch.empty((m, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    Y_new = [torch.full((m, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ctx.gemm_rs(X, W, Y_ref)
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.fo_gemm_rs_noalloc(_mats(fo, X), _mats(fo, W), P, _mats(fo, Y_new), 0,
                                ctypes.c_void_p(status.data_ptr()), stream)
    assert st == fo.FO_OK, lib.fo_last_error_string()
    torch.cuda.synchronize()
    ctx.poll()
    assert int(status.item()) == 0
    for r in range(P):
        assert_close(f64(to_bits(Y_new[r])), f64(to_bits(Y_ref[r])), f"no-alloc rank {r}", round_ref=False)


def test_noalloc_matches_fo_gemm_rs_twice_in_a_row():
    import overlapped_tensor_gemm_gb300 as fo
    lib = fo.load()
    with fo.Context(0) as ctx:
        _run_pair(fo, lib, ctx, 4, 256, 512, 512, 501)
        _run_pair(fo, lib, ctx, 4, 256, 512, 512, 502)


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
