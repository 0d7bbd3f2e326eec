"""GB300-native Flash-Overlap: Python binding of the C ABI in include/fo.h.

This module only marshals arguments (tensor pointers, shapes, the current CUDA
stream) into the C entry points of ``libfo.so``; every step of the hot path
runs in the library's own CUDA kernels.  There is no fallback: if the library
is missing, importing :func:`load` raises.

Method: "FlashOverlap: Minimizing Tail Latency in Communication Overlap for
Distributed LLM Training" (technical summary, section 2): Flash-AG,
Flash-RS with rank-adaptive order, query-split attention -- here with all P
ranks on one GPU.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfo.so")

(FO_OK, FO_ERR_INVALID_ARG, FO_ERR_SHAPE, FO_ERR_UNSUPPORTED, FO_ERR_CUDA, FO_ERR_TIMEOUT, FO_ERR_OOM,
 FO_ERR_RANGE, FO_ERR_INTERNAL) = range(9)
STATUS_NAMES = ["FO_OK", "FO_ERR_INVALID_ARG", "FO_ERR_SHAPE", "FO_ERR_UNSUPPORTED", "FO_ERR_CUDA",
                "FO_ERR_TIMEOUT", "FO_ERR_OOM", "FO_ERR_RANGE", "FO_ERR_INTERNAL"]
FO_BF16, FO_F32 = 0, 1
ORDERS = {"flash": 0, "naive": 1, "slicing": 2, "serial": 3}
LINKS = {"default": 0, "ce": 1, "push": 2}
FAULTS = {"none": 0, "skip_hop": 1}
EPILOGUES = {"plain": 0, "silu": 1}

# Every entry point declared in include/fo.h.
ABI_SYMBOLS = ("fo_version", "fo_last_error_string", "fo_ctx_create", "fo_ctx_destroy", "fo_ctx_poll",
               "fo_ctx_phase_ms", "fo_gemm", "fo_ag_gemm", "fo_gemm_rs", "fo_silu_mul", "fo_mlp_layer",
               "fo_mlp_layer_host", "fo_qsplit_attn", "fo_attn_layer", "fo_gemm_a2a", "fo_a2a_gemm", "fo_col_linear_backward",
               "fo_row_linear_backward", "fo_step_order",
               "fo_gemm_rs_noalloc")


class FoMat(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ld", ctypes.c_int64)]


class FoOpts(ctypes.Structure):
    _fields_ = [("order", ctypes.c_int32), ("link", ctypes.c_int32), ("n_slices", ctypes.c_int32),
                ("timeout_us", ctypes.c_uint32), ("causal_prune", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("fault", ctypes.c_int32), ("epilogue", ctypes.c_int32), ("sm_pairs", ctypes.c_int32),
                ("compute_only", ctypes.c_int32), ("split_layer", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class FoError(RuntimeError):
    def __init__(self, status: int, message: str):
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{name}: {message}")
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Loads libfo.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with overlapped_tensor_gemm_gb300._build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        vp = ctypes.c_void_p
        lib.fo_version.restype = ctypes.c_int
        lib.fo_step_order.restype = ctypes.c_int
        lib.fo_last_error_string.restype = ctypes.c_char_p
        lib.fo_ctx_create.argtypes = [ctypes.c_int, P(vp)]
        lib.fo_ctx_destroy.argtypes = [vp]
        lib.fo_ctx_poll.argtypes = [vp]
        lib.fo_ctx_phase_ms.argtypes = [vp, P(ctypes.c_float), P(ctypes.c_float)]
        lib.fo_gemm.argtypes = [vp, P(FoMat), P(FoMat), P(FoMat), P(FoOpts), vp]
        for name in ("fo_ag_gemm", "fo_gemm_rs", "fo_gemm_a2a", "fo_a2a_gemm"):
            getattr(lib, name).argtypes = [vp, P(FoMat), P(FoMat), ctypes.c_int, P(FoMat), P(FoOpts), vp]
        lib.fo_silu_mul.argtypes = [vp, P(FoMat), ctypes.c_int, P(FoMat), vp]
        for name in ("fo_mlp_layer", "fo_mlp_layer_host"):
            getattr(lib, name).argtypes = [vp, P(FoMat), P(FoMat), P(FoMat), ctypes.c_int, ctypes.c_int,
                                           P(FoMat), P(FoOpts), vp]
        lib.fo_qsplit_attn.argtypes = [vp, P(FoMat), P(FoMat), P(FoMat), ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, P(FoMat), P(FoOpts), vp]
        lib.fo_attn_layer.argtypes = [vp, P(FoMat), P(FoMat), P(FoMat), ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, P(FoMat), P(FoOpts), vp]
        for name in ("fo_col_linear_backward", "fo_row_linear_backward"):
            getattr(lib, name).argtypes = [vp, P(FoMat), P(FoMat), P(FoMat), ctypes.c_int, P(FoMat), P(FoMat),
                                           P(FoOpts), vp]
        lib.fo_step_order.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P(ctypes.c_int32),
                                      P(ctypes.c_int32), ctypes.c_int]
        lib.fo_gemm_rs_noalloc.argtypes = [P(FoMat), P(FoMat), ctypes.c_int, P(FoMat), ctypes.c_uint32,
                                           vp, vp]
        for name in ABI_SYMBOLS:
            if name not in ("fo_version", "fo_last_error_string", "fo_step_order"):
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _check(status: int) -> None:
    if status != FO_OK:
        msg = load().fo_last_error_string().decode(errors="replace")
        raise FoError(status, msg)


def mat(t) -> FoMat:
    """fo_mat view of a 2-D (or [rows, a, b] contiguous-inner) torch tensor."""
    import torch
    if t.dim() > 2:
        t = t.reshape(t.shape[0], -1) if t[0].is_contiguous() else None
        if t is None:
            raise ValueError("inner dimensions must be contiguous")
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError("need a row-major 2-D view (unit column stride)")
    if t.dtype == torch.bfloat16:
        dt = FO_BF16
    elif t.dtype == torch.float32:
        dt = FO_F32
    else:
        raise TypeError(f"unsupported dtype {t.dtype}")
    ld = t.stride(0) if t.shape[0] > 1 else t.shape[1]
    return FoMat(t.data_ptr(), dt, 0, t.shape[0], t.shape[1], max(ld, t.shape[1]))


def _mats(ts: Sequence) -> ctypes.Array:
    arr = (FoMat * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = mat(t)
    return arr


def opts(order: str = "flash", link: str = "default", n_slices: int = 0, timeout_us: int = 0,
         causal_prune: bool = False, num_sms: int = 0, fault: str = "none", epilogue: str = "plain",
         single_sm: bool = False, compute_only: bool = False, split_layer: bool = False,
         pairs: bool = False) -> FoOpts:
    tiles = 2 if pairs else int(single_sm)  # fo_opts.sm_pairs
    return FoOpts(ORDERS[order], LINKS[link], n_slices, timeout_us, int(causal_prune), num_sms, FAULTS[fault],
                  EPILOGUES[epilogue], tiles, int(compute_only), int(split_layer), 0)


def _stream(stream) -> ctypes.c_void_p:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Context:
    """Owns one fo_ctx (link streams, ring workspace, flags) on one device."""

    def __init__(self, device: int = 0):
        self._lib = load()
        self._h = ctypes.c_void_p()
        _check(self._lib.fo_ctx_create(device, ctypes.byref(self._h)))
        self.device = device

    def close(self) -> None:
        if self._h:
            self._lib.fo_ctx_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def poll(self) -> None:
        """Raises FoError if a device wait of an earlier (synchronised) call gave up."""
        _check(self._lib.fo_ctx_poll(self._h))

    def phase_ms(self) -> tuple[float, float]:
        """(collective_ms, gemm_ms) of the last serial-baseline call."""
        a, b = ctypes.c_float(), ctypes.c_float()
        _check(self._lib.fo_ctx_phase_ms(self._h, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def gemm(self, A, B, C, stream=None, **kw) -> None:
        o = opts(**kw)
        _check(self._lib.fo_gemm(self._h, ctypes.byref(mat(A)), ctypes.byref(mat(B)), ctypes.byref(mat(C)),
                                 ctypes.byref(o), _stream(stream)))

    def ag_gemm(self, X_shards, W_col, Y, stream=None, **kw) -> None:
        P = len(X_shards)
        o = opts(**kw)
        _check(self._lib.fo_ag_gemm(self._h, _mats(X_shards), _mats(W_col), P, _mats(Y), ctypes.byref(o),
                                    _stream(stream)))

    def gemm_rs(self, X, W_row, Y, stream=None, **kw) -> None:
        P = len(X)
        o = opts(**kw)
        _check(self._lib.fo_gemm_rs(self._h, _mats(X), _mats(W_row), P, _mats(Y), ctypes.byref(o),
                                    _stream(stream)))

    def gemm_a2a(self, X_shards, W, Y, stream=None, **kw) -> None:
        """Y[d][rows r*m..] = X_shards[r] W[r][rows d*Nb..]^T (the all-to-all's producer GEMM)."""
        P = len(X_shards)
        o = opts(**kw)
        _check(self._lib.fo_gemm_a2a(self._h, _mats(X_shards), _mats(W), P, _mats(Y), ctypes.byref(o),
                                     _stream(stream)))

    def a2a_gemm(self, C, W, Y, stream=None, **kw) -> None:
        """Y[d] = [C[0] rows d*m.. | ... | C[P-1] rows d*m..] W[d]^T (the all-to-all's consumer GEMM)."""
        P = len(C)
        o = opts(**kw)
        _check(self._lib.fo_a2a_gemm(self._h, _mats(C), _mats(W), P, _mats(Y), ctypes.byref(o), _stream(stream)))

    def col_linear_backward(self, X_shards, W_col, dY, dX, dW, stream=None, **kw) -> None:
        """Backward of Y[r] = AG(X) W_col[r]^T: dX (token slices, Flash-RS) and dW (per rank)."""
        P = len(X_shards)
        o = opts(**kw)
        _check(self._lib.fo_col_linear_backward(self._h, _mats(X_shards), _mats(W_col), _mats(dY), P, _mats(dX),
                                                _mats(dW), ctypes.byref(o), _stream(stream)))

    def row_linear_backward(self, H, W_row, dZ_shards, dH, dW, stream=None, **kw) -> None:
        """Backward of Z = RS(H[r] W_row[r]^T): dH (Flash-AG) and dW (per rank)."""
        P = len(H)
        o = opts(**kw)
        _check(self._lib.fo_row_linear_backward(self._h, _mats(H), _mats(W_row), _mats(dZ_shards), P, _mats(dH),
                                                _mats(dW), ctypes.byref(o), _stream(stream)))

    def silu_mul(self, GU, H, stream=None) -> None:
        _check(self._lib.fo_silu_mul(self._h, _mats(GU), len(GU), _mats(H), _stream(stream)))

    def mlp_layer(self, X_shards, W_col, W_row, Z, gated: bool, stream=None, **kw) -> None:
        P = len(X_shards)
        o = opts(**kw)
        _check(self._lib.fo_mlp_layer(self._h, _mats(X_shards), _mats(W_col), _mats(W_row), P, int(gated),
                                      _mats(Z), ctypes.byref(o), _stream(stream)))

    def mlp_layer_host(self, X_shards, W_col, W_row, Z, gated: bool, stream=None, **kw) -> None:
        """X_shards and Z are CPU tensors (pinned for asynchronous copies)."""
        P = len(X_shards)
        o = opts(**kw)
        _check(self._lib.fo_mlp_layer_host(self._h, _mats(X_shards), _mats(W_col), _mats(W_row), P, int(gated),
                                           _mats(Z), ctypes.byref(o), _stream(stream)))

    def qsplit_attn(self, Q, K, V, O, heads: int, head_dim: int, causal: bool = True, stream=None, **kw) -> None:
        P = len(Q)
        o = opts(**kw)
        _check(self._lib.fo_qsplit_attn(self._h, _mats(Q), _mats(K), _mats(V), P, heads, head_dim, int(causal),
                                        _mats(O), ctypes.byref(o), _stream(stream)))

    def attn_layer(self, X_shards, W_qkv, W_o, Z, heads: int, head_dim: int = 128, causal: bool = True,
                   stream=None, **kw) -> None:
        """Flash-AG QKV projection -> per-rank causal attention -> Flash-RS output projection."""
        P = len(X_shards)
        o = opts(**kw)
        _check(self._lib.fo_attn_layer(self._h, _mats(X_shards), _mats(W_qkv), _mats(W_o), P, heads, head_dim,
                                       int(causal), _mats(Z), ctypes.byref(o), _stream(stream)))


def step_order(op: str, P: int, order: str = "flash") -> list[list[tuple[int, int]]]:
    """The library's launch order: per step, (rank, slice or chunk) of each unit."""
    lib = load()
    n = P * P
    rank = (ctypes.c_int32 * n)()
    item = (ctypes.c_int32 * n)()
    got = lib.fo_step_order({"ag": 0, "rs": 1, "gemm_a2a": 2, "a2a_gemm": 3}[op], P, ORDERS[order], rank, item, n)
    if got != n:
        raise FoError(FO_ERR_INVALID_ARG, "bad step-order request")
    return [[(rank[t * P + i], item[t * P + i]) for i in range(P)] for t in range(P)]
