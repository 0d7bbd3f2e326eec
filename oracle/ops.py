"""Definitions and ring-decomposed versions of the Flash-Overlap operations.

Test infrastructure only (see the package docstring).  Source: "FlashOverlap:
Minimizing Tail Latency in Communication Overlap for Distributed LLM
Training", technical summary:

* section 2, Flash-All-Gather: all-gather decomposed into ring P2P steps,
  local slice computed first;
* section 2, Flash-Reduce-Scatter: reduce-scatter decomposed into P2P steps,
  the kept slice computed last (rank-adaptive scheduling);
* section 2, Architectural instantiations: row/column-parallel projections of
  the MLP and attention layers, and query-split attention;
* section 3: the decomposition is exact -- the result equals the undecomposed
  collective followed by (or preceded by) the GEMM.

Conventions.  P ranks; rank r holds the token slice r (rows r*m..(r+1)*m of the
sequence).  Weights use the nn.Linear layout [out, in].  Arithmetic is fp64 on
the exact values of the bf16 inputs; ``bf16.round_f64`` is applied once per
operation output.  Each ``*_definition`` is the plain undecomposed result; each
``*_ring`` runs the decomposed schedule through ``ring.Ring`` and logs
(rank, step, slice) for the schedule invariants.
"""
from __future__ import annotations

import math

import numpy as np

from . import bf16
from .ring import Ring
from .schedule import a2a_block, a2a_source, ag_slice, rs_chunk, rs_hop


def gemm(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """C = A @ B^T in fp64; A [rows, K], B [N, K] (nn.Linear weight layout)."""
    return np.asarray(A, np.float64) @ np.asarray(B, np.float64).T


# --------------------------------------------------------------------------
# AG -> GEMM (column-parallel projection)
# --------------------------------------------------------------------------

def ag_gemm_definition(X_slices, W_col):
    """Undecomposed: X = concat of all ranks' slices, Y_r = X @ W_r^T for every rank r.

    X_slices[s]: rows of token slice s (fp64, any row count); W_col[r]: [N_r, K].
    Returns Y[r] with the slices' rows stacked in slice order.
    """
    X = np.concatenate([np.asarray(x, np.float64) for x in X_slices], axis=0)
    return [gemm(X, W) for W in W_col]


def ag_gemm_ring(X_slices, W_col, direction: int = 1, compute_order=None, fault=None):
    """Flash-AG through the simulated ring.

    Rank r starts with only its own slice.  At hop t (1..P-1) every rank
    forwards the slice it used at step t-1 (its own at t=1) to its ring
    successor.  With ``compute_order=None`` rank r computes slice
    ag_slice(r, t) at step t, interleaved with the hops (local slice first).
    Otherwise the ring runs to completion first and rank r computes its slices
    in the order ``compute_order[r]`` (a permutation of 0..P-1).

    Returns (Y, log) with Y[r] stacked in slice order and log entries
    (rank, step, slice).
    """
    P = len(X_slices)
    ring = Ring(P, direction, fault)
    held = [{r: np.array(X_slices[r], np.float64, copy=True)} for r in range(P)]
    blocks = [dict() for _ in range(P)]
    log = []

    def hop(t):
        for r in range(P):
            s = ag_slice(r, t - 1, P, direction)
            ring.send(r, seq=t, item=s, payload=held[r][s])
        for r in range(P):
            s = ag_slice(r, t, P, direction)
            held[r][s] = ring.recv(r, seq=t, item=s)

    if compute_order is None:
        for t in range(P):
            for r in range(P):
                s = ag_slice(r, t, P, direction)
                blocks[r][s] = gemm(held[r][s], W_col[r])
                log.append((r, t, s))
            if t < P - 1:
                hop(t + 1)
    else:
        for t in range(1, P):
            hop(t)
        for r in range(P):
            if sorted(compute_order[r]) != list(range(P)):
                raise ValueError("compute_order[r] must be a permutation of the slices")
            for t, s in enumerate(compute_order[r]):
                blocks[r][s] = gemm(held[r][s], W_col[r])
                log.append((r, t, s))
    ring.check_drained()
    Y = [np.concatenate([blocks[r][s] for s in range(P)], axis=0) for r in range(P)]
    return Y, log


# --------------------------------------------------------------------------
# GEMM -> RS (row-parallel projection)
# --------------------------------------------------------------------------

def split_chunks(X: np.ndarray, P: int):
    """Rows of a [M, K] activation split into P equal token chunks."""
    m = X.shape[0] // P
    return [X[c * m:(c + 1) * m] for c in range(P)]


def gemm_rs_definition(X_chunks, W_row):
    """Undecomposed: Z_r = X_r @ W_r^T (rank r's K-shard), Y = sum_r Z_r, rank d keeps chunk d.

    X_chunks[r][c]: rows of token chunk c of rank r's input; W_row[r]: [N, K/P].
    """
    P = len(W_row)
    Y = []
    for d in range(P):
        total = None
        for r in range(P):
            z = gemm(X_chunks[r][d], W_row[r])
            total = z if total is None else total + z
        Y.append(total)
    return Y


def gemm_rs_ring(X_chunks, W_row, order: str = "flash", direction: int = 1, fault=None):
    """Flash-RS through the simulated ring.

    ``order='flash'`` (rank-adaptive): at step t rank r computes the partial of
    chunk rs_chunk(r, t), adds the accumulator received from its predecessor
    (none at t=0) and sends the sum on (t < P-1) or keeps it (t = P-1, where
    the chunk is r itself).

    ``order='naive'``: every rank computes its partials in ascending chunk
    order; the reduction of chunk c still walks the ring from rank c+1 to its
    owner c (the same association as 'flash'), each add waiting for its
    accumulator.  The log records the compute order.

    Returns (Y, log); Y[d] is the reduced chunk d, log entries (rank, step, chunk).
    """
    P = len(W_row)
    ring = Ring(P, direction, fault)
    Y = [None] * P
    log = []

    def contribute(r, c, step):
        h = rs_hop(r, c, P, direction)
        part = gemm(X_chunks[r][c], W_row[r])
        acc = part if h == 0 else part + ring.recv(r, seq=h, item=c)
        if h < P - 1:
            ring.send(r, seq=h + 1, item=c, payload=acc)
        else:
            if c != r:
                raise AssertionError("the chain of chunk c must end at its owner")
            Y[r] = acc
        log.append((r, step, c))

    if order == "flash":
        for t in range(P):
            for r in range(P):
                contribute(r, rs_chunk(r, t, P, direction), t)
    elif order == "naive":
        for c in range(P):
            # every rank computes chunk c at step c; adds happen in chain order
            for h in range(P):
                r = (c + direction * (1 + h)) % P
                contribute(r, c, c)
    else:
        raise ValueError(order)
    ring.check_drained()
    return Y, log


# --------------------------------------------------------------------------
# MLP layer: AG-GEMM (gate/up) -> SiLU(gate)*up -> GEMM-RS (down)
# --------------------------------------------------------------------------

def silu_mul(G: np.ndarray, U: np.ndarray) -> np.ndarray:
    """SiLU(g) * u = g / (1 + exp(-g)) * u, in fp64."""
    G = np.asarray(G, np.float64)
    with np.errstate(over="ignore"):
        return G / (1.0 + np.exp(-G)) * np.asarray(U, np.float64)


def activation(Y_r: np.ndarray, gated: bool) -> np.ndarray:
    """Layer glue of the MLP: gate rows come first in the fused column-parallel weight."""
    if not gated:
        return Y_r
    f = Y_r.shape[1] // 2
    return silu_mul(Y_r[:, :f], Y_r[:, f:])


def mlp_layer(X_slices, W_col, W_row, gated: bool, decomposed: bool = True):
    """One MLP layer on P ranks; every operation output is rounded to bf16.

    X_slices[s]: rows of token slice s (fp64 values of bf16 inputs).  Returns
    (Y_ag, H, Z): per-rank AG-GEMM outputs, activations and the RS outputs
    (Z[d] = rank d's kept token slice).  All three are bf16-rounded fp64.
    """
    P = len(W_col)
    if decomposed:
        Y, _ = ag_gemm_ring(X_slices, W_col)
    else:
        Y = ag_gemm_definition(X_slices, W_col)
    Y = [bf16.round_f64(y) for y in Y]
    H = [bf16.round_f64(activation(y, gated)) for y in Y]
    rows = [np.asarray(x).shape[0] for x in X_slices]
    offs = np.cumsum([0] + rows)
    H_chunks = [[h[offs[c]:offs[c + 1]] for c in range(P)] for h in H]
    if decomposed:
        Z, _ = gemm_rs_ring(H_chunks, W_row)
    else:
        Z = gemm_rs_definition(H_chunks, W_row)
    Z = [bf16.round_f64(z) for z in Z]
    return Y, H, Z


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def attention_definition(Q, K, V, causal: bool = True, q_rows=None):
    """softmax(Q K^T / sqrt(d) + mask) V per head, two-pass (max, then exp-sum), fp64.

    Q, K, V: [S, H, D]; the causal mask removes key j > query i (diagonal kept).
    ``q_rows`` (optional) restricts the output to those query rows.
    Returns O [len(q_rows) or S, H, D].
    """
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    S, H, D = K.shape
    qi = np.arange(Q.shape[0]) if q_rows is None else np.asarray(q_rows)
    scale = 1.0 / math.sqrt(D)
    O = np.zeros((len(qi), H, D))
    for h in range(H):
        s = (Q[qi, h, :] @ K[:, h, :].T) * scale
        if causal:
            s = np.where(np.arange(S)[None, :] > qi[:, None], -np.inf, s)
        mx = s.max(axis=1, keepdims=True)
        p = np.exp(s - mx)
        O[:, h, :] = (p @ V[:, h, :]) / p.sum(axis=1, keepdims=True)
    return O


def qsplit_attention_ring(Q_shards, K_shards, V_shards, causal: bool = True, prune: bool = False,
                          direction: int = 1, fault=None, q_rows=None):
    """Query-split causal attention through the simulated ring (online softmax, fp64).

    Rank r keeps its query slice Q_r; K/V slices travel the ring like Flash-AG
    slices (local slice first).  At step t rank r folds slice s = ag_slice(r, t)
    into its running (max, sum, weighted-V) state; with ``causal`` a slice that
    lies wholly above the diagonal (s > r) is skipped, and the local slice uses
    the diagonal mask.  ``prune`` forwards a slice only to ranks that use it.
    ``q_rows[r]`` (optional) restricts rank r's queries to those local rows.

    Returns (O, log): O[r] [rows, H, D]; log entries (rank, step, slice, used).
    """
    P = len(Q_shards)
    m, H, D = np.asarray(K_shards[0]).shape
    scale = 1.0 / math.sqrt(D)
    ring = Ring(P, direction, fault)
    held = [{r: (np.array(K_shards[r], np.float64), np.array(V_shards[r], np.float64))}
            for r in range(P)]
    rows = [np.arange(np.asarray(Q_shards[r]).shape[0]) if q_rows is None else np.asarray(q_rows[r])
            for r in range(P)]
    Qs = [np.asarray(Q_shards[r], np.float64)[rows[r]] for r in range(P)]
    mx = [np.full((H, len(rows[r])), -np.inf) for r in range(P)]
    lsum = [np.zeros((H, len(rows[r]))) for r in range(P)]
    acc = [np.zeros((H, len(rows[r]), D)) for r in range(P)]
    log = []

    if prune and direction != 1:
        raise ValueError("pruned forwarding is defined for the +1 ring only")

    def forwarded(dst: int, t1: int) -> bool:
        """Does rank dst receive a slice at hop t1?  Pruned: only slices s < dst."""
        return not (prune and causal) or dst - t1 >= 0

    for t in range(P):
        for r in range(P):
            s = ag_slice(r, t, P, direction)
            if causal and s > r:
                log.append((r, t, s, False))
                continue
            Ks, Vs = held[r][s]
            qg = r * m + rows[r]
            kg = s * m + np.arange(Ks.shape[0])
            for h in range(H):
                sc = (Qs[r][:, h, :] @ Ks[:, h, :].T) * scale
                if causal:
                    sc = np.where(kg[None, :] > qg[:, None], -np.inf, sc)
                m_new = np.maximum(mx[r][h], sc.max(axis=1))
                alpha = np.exp(mx[r][h] - m_new)
                p = np.exp(sc - m_new[:, None])
                lsum[r][h] = lsum[r][h] * alpha + p.sum(axis=1)
                acc[r][h] = acc[r][h] * alpha[:, None] + p @ Vs[:, h, :]
                mx[r][h] = m_new
            log.append((r, t, s, True))
        if t < P - 1:
            for r in range(P):
                if forwarded(ring.dst(r), t + 1):
                    s = ag_slice(r, t, P, direction)
                    ring.send(r, seq=t + 1, item=s, payload=np.stack(held[r][s]))
            for r in range(P):
                if forwarded(r, t + 1):
                    s = ag_slice(r, t + 1, P, direction)
                    kv = ring.recv(r, seq=t + 1, item=s)
                    held[r][s] = (kv[0], kv[1])
    ring.check_drained()
    O = [np.transpose(acc[r] / lsum[r][:, :, None], (1, 0, 2)) for r in range(P)]
    return O, log


# --------------------------------------------------------------------------
# attention block (QKV projection -> attention -> output projection)
# --------------------------------------------------------------------------

def attn_layer(X_slices, W_qkv, W_o, heads: int, causal: bool = True, decomposed: bool = True):
    """One attention block on P ranks; every operation output is rounded to bf16.

    Technical summary, section 2 (architectural instantiations): the QKV
    projection is the column-parallel GEMM after the all-gather, the output
    projection the row-parallel GEMM before the reduce-scatter; attention itself
    needs no communication because rank r owns ``heads`` whole heads for every
    token.  W_qkv[r] = [Q rows; K rows; V rows] of rank r's heads ([3*heads*D, Hd]),
    W_o[r] = the output projection's columns of rank r's heads ([Hd, heads*D]).

    Returns (QKV, O, Z): QKV[r] [M, 3*heads*D], O[r] [M, heads*D] (attention of
    rank r's heads over all M tokens) and Z[d] [m, Hd] (rank d's token slice).
    """
    P = len(W_qkv)
    if decomposed:
        QKV, _ = ag_gemm_ring(X_slices, W_qkv)
    else:
        QKV = ag_gemm_definition(X_slices, W_qkv)
    QKV = [bf16.round_f64(y) for y in QKV]
    O = []
    for r in range(P):
        M, three_hd = QKV[r].shape
        HD = three_hd // 3
        D = HD // heads
        q = QKV[r][:, :HD].reshape(M, heads, D)
        k = QKV[r][:, HD:2 * HD].reshape(M, heads, D)
        v = QKV[r][:, 2 * HD:].reshape(M, heads, D)
        O.append(bf16.round_f64(attention_definition(q, k, v, causal).reshape(M, HD)))
    rows = [np.asarray(x).shape[0] for x in X_slices]
    offs = np.cumsum([0] + rows)
    chunks = [[o[offs[c]:offs[c + 1]] for c in range(P)] for o in O]
    if decomposed:
        Z, _ = gemm_rs_ring(chunks, W_o)
    else:
        Z = gemm_rs_definition(chunks, W_o)
    Z = [bf16.round_f64(z) for z in Z]
    return QKV, O, Z


# --------------------------------------------------------------------------
# Flash all-to-all (Ulysses parallelism): GEMM -> A2A and A2A -> GEMM
# --------------------------------------------------------------------------

def gemm_a2a_definition(X_slices, W):
    """Undecomposed producer side: rank r's output X_r @ W_r^T is split into P column
    blocks of N/P; block d belongs to rank d, which stacks the blocks by source rank.

    X_slices[r] [m, K]; W[r] [N, K].  Returns Y[d] [P*m, N/P] (rows r*m.. from rank r).
    """
    P = len(W)
    Nb = np.asarray(W[0]).shape[0] // P
    return [np.concatenate([gemm(X_slices[r], np.asarray(W[r])[d * Nb:(d + 1) * Nb]) for r in range(P)])
            for d in range(P)]


def gemm_a2a_ring(X_slices, W, order: str = "flash", direction: int = 1, fault=None):
    """Producer side through simulated P2P messages.  At step t rank r computes block
    a2a_block(r, t) ('naive': block t) and sends it straight to that rank (its own block
    stays).  Returns (Y, log); log entries (rank, step, block)."""
    P = len(W)
    Nb = np.asarray(W[0]).shape[0] // P
    ring = Ring(P, direction, fault)
    got = [dict() for _ in range(P)]
    log = []
    for t in range(P):
        sent = []
        for r in range(P):
            d = a2a_block(r, t, P, direction) if order == "flash" else t
            blk = gemm(X_slices[r], np.asarray(W[r])[d * Nb:(d + 1) * Nb])
            log.append((r, t, d))
            if d == r:
                got[r][r] = blk
            else:
                ring.send_to(r, d, seq=t, item=r, payload=blk)
                sent.append((d, r))
        for d, r in sent:
            got[d][r] = ring.recv(d, seq=t, item=r)
    ring.check_drained()
    return [np.concatenate([got[d][r] for r in range(P)]) for d in range(P)], log


def a2a_gemm_definition(C, W):
    """Undecomposed consumer side: rows d*m.. of every rank's C_s are rank d's K chunks;
    rank d multiplies their column concatenation by W_d^T.

    C[s] [P*m, Kc]; W[d] [N, P*Kc].  Returns Y[d] [m, N].
    """
    P = len(W)
    m = np.asarray(C[0]).shape[0] // P
    out = []
    for d in range(P):
        A = np.concatenate([np.asarray(C[s], np.float64)[d * m:(d + 1) * m] for s in range(P)], axis=1)
        out.append(gemm(A, W[d]))
    return out


def a2a_gemm_ring(C, W, order: str = "flash", direction: int = 1, fault=None):
    """Consumer side through simulated P2P messages.  At hop t (1..P-1) rank s sends its
    chunk for rank d = s + t; rank d's GEMM is a sum over K chunks, one per source, folded
    in the order a2a_source(d, t) ('flash': own chunk first, then each as it arrives) or
    ascending source ('naive', after every hop).  Returns (Y, log); log entries
    (rank, step, source)."""
    P = len(W)
    m = np.asarray(C[0]).shape[0] // P
    Kc = np.asarray(C[0]).shape[1]
    ring = Ring(P, direction, fault)
    held = [{d: np.asarray(C[d], np.float64)[d * m:(d + 1) * m].copy()} for d in range(P)]
    acc = [None] * P
    log = []

    def hop(t):
        for s in range(P):
            d = (s + direction * t) % P
            ring.send_to(s, d, seq=t, item=s, payload=np.asarray(C[s], np.float64)[d * m:(d + 1) * m])
        for d in range(P):
            s = (d - direction * t) % P
            held[d][s] = ring.recv(d, seq=t, item=s)

    def fold(d, s, t):
        part = gemm(held[d][s], np.asarray(W[d])[:, s * Kc:(s + 1) * Kc])
        acc[d] = part if acc[d] is None else acc[d] + part
        log.append((d, t, s))

    if order == "flash":
        for t in range(P):
            if t > 0:
                hop(t)
            for d in range(P):
                fold(d, a2a_source(d, t, P, direction), t)
    elif order == "naive":
        for t in range(1, P):
            hop(t)
        for t in range(P):
            for d in range(P):
                fold(d, t, t)
    else:
        raise ValueError(order)
    ring.check_drained()
    return acc, log


# --------------------------------------------------------------------------
# training backward of the two projections
# --------------------------------------------------------------------------

def col_linear_backward(X_slices, W_col, dY, decomposed: bool = True):
    """Backward of the column-parallel projection Y_r = AG(X) @ W_r^T.

    The all-gather's adjoint is a reduce-scatter: dX (rank d's token slice) =
    sum_r dY_r[rows of slice d] @ W_r, computed through the Flash-RS ring with the
    transposed weight; dW_r = dY_r^T @ AG(X) is local.  Outputs rounded to bf16.
    Returns (dX [P] of [m, K], dW [P] of [Nr, K]).
    """
    P = len(W_col)
    Wt = [np.asarray(w, np.float64).T for w in W_col]
    chunks = [split_chunks(np.asarray(d, np.float64), P) for d in dY]
    if decomposed:
        dX, _ = gemm_rs_ring(chunks, Wt)
    else:
        dX = gemm_rs_definition(chunks, Wt)
    X_full = np.concatenate([np.asarray(x, np.float64) for x in X_slices])
    dW = [gemm(np.asarray(d, np.float64).T, X_full.T) for d in dY]
    return [bf16.round_f64(x) for x in dX], [bf16.round_f64(w) for w in dW]


def row_linear_backward(H, W_row, dZ_slices, decomposed: bool = True):
    """Backward of the row-parallel projection Z = RS(H_r @ W_r^T).

    The reduce-scatter's adjoint is an all-gather: dH_r = AG(dZ) @ W_r, computed through
    the Flash-AG ring with the transposed weight; dW_r = AG(dZ)^T @ H_r is local.
    Outputs rounded to bf16.  Returns (dH [P] of [M, Fr], dW [P] of [N, Fr]).
    """
    Wt = [np.asarray(w, np.float64).T for w in W_row]
    if decomposed:
        dH, _ = ag_gemm_ring(dZ_slices, Wt)
    else:
        dH = ag_gemm_definition(dZ_slices, Wt)
    dZ_full = np.concatenate([np.asarray(z, np.float64) for z in dZ_slices])
    dW = [gemm(dZ_full.T, np.asarray(h, np.float64).T) for h in H]
    return [bf16.round_f64(x) for x in dH], [bf16.round_f64(w) for w in dW]
