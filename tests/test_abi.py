"""The C-ABI library loads on a host without a GPU, exports every entry point that
include/fo.h declares, and rejects bad arguments synchronously (no compute calls)."""
import ctypes
import os
import re

import pytest

import overlapped_tensor_gemm_gb300 as fo


@pytest.fixture(scope="module")
def lib(repo_root):
    if not os.path.exists(fo.LIB_PATH):
        from overlapped_tensor_gemm_gb300 import _build
        _build.build()
    return fo.load()


def _declared(repo_root):
    with open(os.path.join(repo_root, "include", "fo.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"FO_API\s+[\w\s\*]*?\b(fo_\w+)\s*\(", text)))


def test_header_and_binding_agree(repo_root):
    assert _declared(repo_root) == sorted(fo.ABI_SYMBOLS)


def test_every_declared_symbol_is_exported(lib, repo_root):
    for name in _declared(repo_root):
        assert hasattr(lib, name), name
    assert lib.fo_version() == 100


def test_null_arguments_are_rejected(lib):
    null = ctypes.c_void_p()
    mats = (fo.FoMat * 2)()
    o = fo.opts()
    assert lib.fo_ag_gemm(null, mats, mats, 2, mats, ctypes.byref(o), null) == fo.FO_ERR_INVALID_ARG
    assert b"context" in lib.fo_last_error_string()
    assert lib.fo_gemm_rs(null, mats, mats, 2, mats, ctypes.byref(o), null) == fo.FO_ERR_INVALID_ARG
    assert lib.fo_attn_layer(null, mats, mats, mats, 2, 1, 128, 1, mats, ctypes.byref(o), null) == fo.FO_ERR_INVALID_ARG
    assert lib.fo_ctx_poll(null) == fo.FO_ERR_INVALID_ARG
    assert lib.fo_ctx_create(0, None) == fo.FO_ERR_INVALID_ARG
    assert lib.fo_ctx_destroy(null) == fo.FO_OK


def test_context_creation_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = lib.fo_ctx_create(0, ctypes.byref(h))
    assert st in (fo.FO_ERR_CUDA, fo.FO_ERR_INVALID_ARG)
    assert not h.value
    assert lib.fo_last_error_string()


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_library_step_order_follows_the_oracle_schedule(lib, P):
    """The fused launches' unit order (host logic, no GPU) against the oracle's step
    formulas: AG step 0 is every rank's own slice, RS step P-1 its kept chunk, and
    the naive order computes chunk t on every rank at step t."""
    from oracle import schedule
    ag = fo.step_order("ag", P)
    rs = fo.step_order("rs", P)
    nv = fo.step_order("rs", P, "naive")
    for t in range(P):
        assert sorted(r for r, _ in ag[t]) == list(range(P))
        assert sorted(r for r, _ in rs[t]) == list(range(P))
        for r, s in ag[t]:
            assert s == schedule.ag_slice(r, t, P)
        for r, c in rs[t]:
            assert c == schedule.rs_chunk(r, t, P)
        for h, (r, c) in enumerate(nv[t]):
            assert c == schedule.rs_chunk_naive(r, t, P)
            assert schedule.rs_hop(r, c, P) == h      # chain order inside the step
    # every RS unit consumes a partial sum produced one whole step earlier, same position
    for t in range(1, P):
        for i, (r, c) in enumerate(rs[t]):
            assert rs[t - 1][i] == ((r - 1) % P, c)
    assert lib.fo_step_order(0, P, 1, (ctypes.c_int32 * 64)(), (ctypes.c_int32 * 64)(), 64) == -1


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_library_all_to_all_order_follows_the_oracle_schedule(lib, P):
    """The all-to-all launches' unit order (host logic, no GPU) against the oracle: the
    producer computes its own block last, the consumer folds in its own chunk first."""
    from oracle import schedule
    prod = fo.step_order("gemm_a2a", P)
    cons = fo.step_order("a2a_gemm", P)
    for t in range(P):
        for r, d in prod[t]:
            assert d == schedule.a2a_block(r, t, P)
        for r, s in cons[t]:
            assert s == schedule.a2a_source(r, t, P)
    for r in range(P):
        assert prod[P - 1][r] == (r, r)
        assert cons[0][r] == (r, r)
        assert sorted(d for t in range(P) for rr, d in prod[t] if rr == r) == list(range(P))
        assert sorted(s for t in range(P) for rr, s in cons[t] if rr == r) == list(range(P))


def test_debug_bounds_build_compiles_and_exports(repo_root, tmp_path):
    """The debug build (index checks in the kernels, failures recorded as FO_ERR_INTERNAL)
    compiles for sm_103a and exports the same entry points."""
    from overlapped_tensor_gemm_gb300 import _build
    out = _build.build(debug_bounds=True, out=str(tmp_path / "libfo_debug.so"))
    dbg = ctypes.CDLL(out)
    for name in _declared(repo_root):
        assert hasattr(dbg, name), name


def test_struct_layouts_match_the_header():
    """fo_opts and fo_mat in the binding have the header's size (twelve 4-byte fields,
    and a pointer, two 4-byte and three 8-byte fields)."""
    assert ctypes.sizeof(fo.FoOpts) == 12 * 4
    assert ctypes.sizeof(fo.FoMat) == 8 + 4 + 4 + 3 * 8
