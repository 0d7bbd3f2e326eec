"""Seeded synthetic workloads for the Flash-Overlap hot path.

This module is shared by the CPU oracle (``oracle/``) and the CUDA path
(``overlapped_tensor_gemm_gb300``).  It holds shapes and random-number
generation only -- none of the method's arithmetic.  Every tensor is returned
as raw bf16 bit patterns (``numpy.uint16``) so that both sides see identical
bytes.

Workload shapes (the pages give none; these follow the five benchmark
configurations of the build):

* ``tiny``   -- Flash-AG + Flash-RS MLP, P=2, tokens 256, hidden 256, ffn 512,
  integer values uniform in {-2..2}, up-projection only (identity activation).
* ``llama8b`` -- Llama-3-8B-shaped MLP, P=4, tokens 4096, hidden 4096,
  ffn 14336, X~N(0,1), W~N(0,0.02).
* ``sweep``  -- 70B-like MLP, P=8, tokens S in {1K..16K}, hidden 8192,
  ffn 28672.
* ``tail_rs`` -- GEMM-RS only, P=8, tokens 512, hidden (out) 8192,
  in-features 28672.
* ``attn``   -- query-split causal attention, P=4, seq 16384, 32 heads,
  head_dim 128, Q,K,V~N(0,1); ``attn1k``..``attn16k`` the same at other lengths.
* ``a2a``    -- Flash all-to-all (Ulysses): QKV projection -> all-to-all and
  all-to-all -> output projection, P=4, tokens 16384, hidden 4096.
* ``attn_layer`` -- attention block (Flash-AG QKV projection, per-rank causal
  attention of the rank's heads, Flash-RS output projection), Llama-3-8B-shaped:
  P=4, tokens 4096, hidden 4096, 32 heads of 128 (8 per rank), X~N(0,1),
  W~N(0,0.02).

Seeds are ``1234 + config index``.  Generation uses the torch CPU generator
(a library PRNG); conversion to bf16 uses torch's round-to-nearest-even cast.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

W_STD = 0.02


@dataclasses.dataclass(frozen=True)
class MLPConfig:
    name: str
    index: int
    P: int
    tokens: int
    hidden: int
    ffn: int
    gated: bool          # True: SiLU(gate)*up with gate+up fused per rank
    integer: bool        # True: values uniform in {-2..2}

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def m(self) -> int:
        return self.tokens // self.P

    @property
    def n_col(self) -> int:
        """Output columns of one rank's column-parallel (AG) weight."""
        f = self.ffn // self.P
        return 2 * f if self.gated else f

    @property
    def k_row(self) -> int:
        """In-features of one rank's row-parallel (RS) weight."""
        return self.ffn // self.P

    def flops(self) -> dict:
        ag = 2 * self.tokens * self.hidden * self.n_col * self.P
        rs = 2 * self.tokens * self.k_row * self.hidden * self.P
        return {"ag": ag, "rs": rs, "total": ag + rs}

    def copy_bytes(self) -> dict:
        """Algorithmic one-way ring bytes: AG forwards bf16 slices, RS fp32 partials."""
        ag = (self.P - 1) * self.tokens * self.hidden * 2
        rs = (self.P - 1) * self.tokens * self.hidden * 4
        return {"ag": ag, "rs": rs}


@dataclasses.dataclass(frozen=True)
class RSConfig:
    name: str
    index: int
    P: int
    tokens: int
    n_out: int
    k_total: int
    integer: bool

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def m(self) -> int:
        return self.tokens // self.P

    @property
    def k_row(self) -> int:
        return self.k_total // self.P

    def flops(self) -> int:
        return 2 * self.tokens * self.k_total * self.n_out


@dataclasses.dataclass(frozen=True)
class AttnConfig:
    name: str
    index: int
    P: int
    seq: int
    heads: int
    head_dim: int

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def m(self) -> int:
        return self.seq // self.P

    def flops(self) -> int:
        """Causal-only algorithmic FLOP: QK^T and PV over the i>=j triangle."""
        pairs = self.seq * (self.seq + 1) // 2
        return 4 * pairs * self.heads * self.head_dim


TINY = MLPConfig("tiny", 0, P=2, tokens=256, hidden=256, ffn=512, gated=False, integer=True)
LLAMA8B = MLPConfig("llama8b", 1, P=4, tokens=4096, hidden=4096, ffn=14336, gated=True, integer=False)


def sweep(tokens: int) -> MLPConfig:
    return MLPConfig(f"sweep{tokens // 1024}k", 2, P=8, tokens=tokens, hidden=8192, ffn=28672,
                     gated=True, integer=False)


SWEEP_TOKENS = (1024, 2048, 4096, 8192, 16384)
TAIL_RS = RSConfig("tail_rs", 3, P=8, tokens=512, n_out=8192, k_total=28672, integer=False)
ATTN = AttnConfig("attn", 4, P=4, seq=16384, heads=32, head_dim=128)


@dataclasses.dataclass(frozen=True)
class AttnLayerConfig:
    name: str
    index: int
    P: int
    tokens: int
    hidden: int
    heads: int          # heads per rank
    head_dim: int = 128

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def m(self) -> int:
        return self.tokens // self.P

    def flops(self) -> dict:
        """Algorithmic FLOP: QKV and output projections (2*M*K*N each), causal attention
        (QK^T and PV over the i>=j triangle) of all P*heads heads."""
        hd = self.heads * self.head_dim
        qkv = 2 * self.tokens * self.hidden * 3 * hd * self.P
        attn = 4 * (self.tokens * (self.tokens + 1) // 2) * self.heads * self.P * self.head_dim
        out = 2 * self.tokens * hd * self.P * self.hidden
        return {"qkv": qkv, "attn": attn, "out": out, "total": qkv + attn + out}


ATTN_LAYER = AttnLayerConfig("attn_layer", 5, P=4, tokens=4096, hidden=4096, heads=8)


@dataclasses.dataclass(frozen=True)
class A2AConfig:
    """Ulysses-style projections around attention: the QKV projection feeding the
    all-to-all (producer, N = 3 * hidden split into P head groups) and the output
    projection behind it (consumer, K = hidden split into P head groups)."""
    name: str
    index: int
    P: int
    tokens: int
    hidden: int

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def m(self) -> int:
        return self.tokens // self.P

    def flops(self) -> dict:
        prod = 2 * self.tokens * self.hidden * 3 * self.hidden
        cons = 2 * self.tokens * self.hidden * self.hidden
        return {"gemm_a2a": prod, "a2a_gemm": cons}


A2A = A2AConfig("a2a", 6, P=4, tokens=16384, hidden=4096)


def attn_sweep(seq: int) -> AttnConfig:
    """The query-split attention workload at another sequence length (P=4, 32 heads)."""
    return AttnConfig(f"attn{seq // 1024}k", 4, P=4, seq=seq, heads=32, head_dim=128)


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------

def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _to_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def integer_bf16(gen: torch.Generator, shape, lo: int = -2, hi: int = 2) -> np.ndarray:
    """Integers uniform in [lo, hi], stored as bf16 bits (exactly representable)."""
    t = torch.randint(lo, hi + 1, tuple(shape), generator=gen, dtype=torch.int32)
    return _to_bits(t.to(torch.float32))


def gaussian_bf16(gen: torch.Generator, shape, std: float = 1.0) -> np.ndarray:
    t = torch.randn(tuple(shape), generator=gen, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return _to_bits(t)


def bits_to_torch(bits: np.ndarray) -> torch.Tensor:
    """bf16 bit array -> CPU torch.bfloat16 tensor sharing no memory with the input."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16)


def mlp_inputs(cfg: MLPConfig, integer: bool | None = None, seed_offset: int = 0) -> dict:
    """X shards (sequence-sharded tokens), column-parallel W_col[r] and row-parallel W_row[r].

    Shapes: X_shards[r] [m, hidden]; W_col[r] [n_col, hidden] (nn.Linear [out, in], gate rows
    first when gated); W_row[r] [hidden, k_row] (columns r*k_row..(r+1)*k_row of the full
    down-projection [hidden, ffn]).
    """
    integer = cfg.integer if integer is None else integer
    g = _gen(cfg.seed + seed_offset)
    P, m, H = cfg.P, cfg.m, cfg.hidden
    if integer:
        X = [integer_bf16(g, (m, H)) for _ in range(P)]
        Wc = [integer_bf16(g, (cfg.n_col, H)) for _ in range(P)]
        Wr = [integer_bf16(g, (H, cfg.k_row)) for _ in range(P)]
    else:
        X = [gaussian_bf16(g, (m, H)) for _ in range(P)]
        Wc = [gaussian_bf16(g, (cfg.n_col, H), W_STD) for _ in range(P)]
        Wr = [gaussian_bf16(g, (H, cfg.k_row), W_STD) for _ in range(P)]
    return {"X_shards": X, "W_col": Wc, "W_row": Wr}


def rs_inputs(P: int, tokens: int, n_out: int, k_row: int, seed: int, integer: bool) -> dict:
    """Inputs of one GEMM-RS: X[r] [tokens, k_row] (rank r's in-feature shard), W_row[r] [n_out, k_row]."""
    g = _gen(seed)
    if integer:
        X = [integer_bf16(g, (tokens, k_row)) for _ in range(P)]
        W = [integer_bf16(g, (n_out, k_row)) for _ in range(P)]
    else:
        X = [gaussian_bf16(g, (tokens, k_row)) for _ in range(P)]
        W = [gaussian_bf16(g, (n_out, k_row), W_STD) for _ in range(P)]
    return {"X": X, "W_row": W}


def ag_inputs(P: int, m: int, k: int, n_col: int, seed: int, integer: bool) -> dict:
    """Inputs of one AG-GEMM: X_shards[r] [m, k], W_col[r] [n_col, k]."""
    g = _gen(seed)
    if integer:
        X = [integer_bf16(g, (m, k)) for _ in range(P)]
        W = [integer_bf16(g, (n_col, k)) for _ in range(P)]
    else:
        X = [gaussian_bf16(g, (m, k)) for _ in range(P)]
        W = [gaussian_bf16(g, (n_col, k), W_STD) for _ in range(P)]
    return {"X_shards": X, "W_col": W}


def attn_inputs(P: int, seq: int, heads: int, head_dim: int, seed: int) -> dict:
    """Q/K/V shards [seq/P, heads, head_dim] (head_dim contiguous), N(0,1) bf16."""
    g = _gen(seed)
    m = seq // P
    Q = [gaussian_bf16(g, (m, heads, head_dim)) for _ in range(P)]
    K = [gaussian_bf16(g, (m, heads, head_dim)) for _ in range(P)]
    V = [gaussian_bf16(g, (m, heads, head_dim)) for _ in range(P)]
    return {"Q": Q, "K": K, "V": V}


def attn_layer_inputs(P: int, tokens: int, hidden: int, heads: int, head_dim: int, seed: int) -> dict:
    """X shards [tokens/P, hidden] ~N(0,1); per rank W_qkv [3*heads*head_dim, hidden] and
    W_o [hidden, heads*head_dim] ~N(0, 0.02); bf16 bits."""
    g = _gen(seed)
    m = tokens // P
    hd = heads * head_dim
    X = [gaussian_bf16(g, (m, hidden)) for _ in range(P)]
    W_qkv = [gaussian_bf16(g, (3 * hd, hidden), W_STD) for _ in range(P)]
    W_o = [gaussian_bf16(g, (hidden, hd), W_STD) for _ in range(P)]
    return {"X_shards": X, "W_qkv": W_qkv, "W_o": W_o}


def sample_rows(n_rows: int, block: int, per_block: int, seed: int) -> np.ndarray:
    """Deterministic row sample: first/last row of every block, plus seeded random rows.

    Used to check outputs of large workloads row by row (a GEMM or attention output row
    depends only on its own input/query row).
    """
    rng = np.random.default_rng(seed)
    rows = set()
    for b0 in range(0, n_rows, block):
        b1 = min(b0 + block, n_rows)
        rows.add(b0)
        rows.add(b1 - 1)
        k = max(0, min(per_block - 2, b1 - b0 - 2))
        if k:
            rows.update(int(x) for x in rng.choice(np.arange(b0 + 1, b1 - 1), size=k, replace=False))
    return np.array(sorted(rows), dtype=np.int64)
