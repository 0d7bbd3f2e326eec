"""Step orders of the decomposed collectives, and a unit-time timeline model.

Source: "FlashOverlap: Minimizing Tail Latency in Communication Overlap for
Distributed LLM Training", technical summary section 2 (Methodology):

* Flash-All-Gather decomposes the all-gather into ring P2P steps; a rank first
  computes the slice it already holds, then each slice as it arrives.
* Flash-Reduce-Scatter decomposes the reduce-scatter into P2P steps; with
  rank-adaptive scheduling the slice that stays on the rank (needs no further
  transfer) is computed at the last step.
* Flash All-to-All (section 2) extends the decomposition to the all-to-all of
  Ulysses parallelism; the pages give no detail, the step orders below apply the
  two rules above to its producer and consumer GEMMs.
* Section 1 (Problem statement): data slicing interleaves chunks of compute and
  communication, but the communication of the last chunk cannot overlap.

Readings taken where the pages are silent: the ring sends rank r -> r+1
(``direction=+1``; ``-1`` is the mirror ring); one slice per rank (M/P rows);
the naive order computes chunks in ascending index on every rank.
"""
from __future__ import annotations


def ag_slice(r: int, t: int, P: int, direction: int = 1) -> int:
    """Flash-AG: the slice rank r computes at step t.  Step 0 is its own slice."""
    return (r - direction * t) % P


def rs_chunk(r: int, t: int, P: int, direction: int = 1) -> int:
    """Flash-RS rank-adaptive order: the chunk rank r computes at step t.

    Rank r's partial for this chunk is added to the accumulator that arrived
    from its ring predecessor and forwarded; at t = P-1 the chunk is r itself
    (the kept slice) and the sum is final.
    """
    return (r - direction * (t + 1)) % P


def rs_chunk_naive(r: int, t: int, P: int) -> int:
    """Rank-oblivious order: every rank computes chunk t at step t."""
    return t % P


def a2a_block(r: int, t: int, P: int, direction: int = 1) -> int:
    """Flash all-to-all, producer side (a GEMM whose output block d belongs to rank d):
    the block rank r computes at step t.  Remote blocks first, so each can be sent as
    soon as it is done; the own block (no transfer) last, at t = P-1 -- the
    rank-adaptive rule of Flash-RS applied to the all-to-all."""
    return (r + direction * (t + 1)) % P


def a2a_source(r: int, t: int, P: int, direction: int = 1) -> int:
    """Flash all-to-all, consumer side (a GEMM whose K chunks come from every rank): the
    source rank whose chunk rank r folds in at step t.  Own chunk first (no wait), then
    the chunk that arrives at hop t (source r - t sends to r at step t) -- the
    local-first rule of Flash-AG applied to the all-to-all."""
    return (r - direction * t) % P


def rs_hop(r: int, c: int, P: int, direction: int = 1) -> int:
    """Position of rank r on the reduction chain of chunk c (0 = first, P-1 = owner c)."""
    return (direction * (r - c) - 1) % P


# --------------------------------------------------------------------------
# unit-time timeline model
# --------------------------------------------------------------------------

def timeline(kind: str, P: int, comp: float = 1.0, hop: float = 0.5, n_chunks: int | None = None) -> dict:
    """Finish time of one layer under a simple model.

    Each rank owns one compute unit and one outgoing link.  Computing one slice
    (M/P rows of the layer's rows for that rank) takes ``comp``; sending one
    slice-sized message over one hop takes ``hop``; link and compute run
    concurrently.  ``exposed = finish - P*comp`` is the communication time that
    was not hidden behind compute.

    kinds: ag_flash, ag_serial, ag_slicing, rs_flash, rs_serial, rs_slicing, rs_naive.
    """
    n = n_chunks or P
    if kind == "ag_flash":
        arrive = {(r, 0): 0.0 for r in range(P)}          # slice used at step t is there
        link_free = [0.0] * P
        for t in range(1, P):
            for r in range(P):
                src = (r - 1) % P                           # forwards what it used at step t-1
                start = max(link_free[src], arrive[(src, t - 1)])
                link_free[src] = start + hop
                arrive[(r, t)] = start + hop
        finish = 0.0
        for r in range(P):
            end = 0.0
            for t in range(P):
                end = max(end, arrive[(r, t)]) + comp
            finish = max(finish, end)
    elif kind == "ag_serial":
        finish = (P - 1) * hop + P * comp
    elif kind == "ag_slicing":
        # all-gather of chunk i ((P-1) hops of 1/n-sized messages), then compute chunk i
        gather_end, comp_end = 0.0, 0.0
        for i in range(n):
            gather_end = gather_end + (P - 1) * hop / n
            comp_end = max(comp_end, gather_end) + P * comp / n
        finish = comp_end
    elif kind == "rs_flash":
        end = {}
        link_free = [0.0] * P
        arrive = {}
        for t in range(P):
            for r in range(P):
                start = end.get((r, t - 1), 0.0)
                ready = start + comp
                if t > 0:
                    ready = max(ready, arrive[(r, t)])
                end[(r, t)] = ready
                if t < P - 1:
                    dst = (r + 1) % P
                    s = max(link_free[r], ready)
                    link_free[r] = s + hop
                    arrive[(dst, t + 1)] = s + hop
        finish = max(end.values())
    elif kind == "rs_serial":
        finish = P * comp + (P - 1) * hop
    elif kind == "rs_slicing":
        comp_end, red_end = 0.0, 0.0
        for i in range(n):
            comp_end = comp_end + P * comp / n
            red_end = max(red_end, comp_end) + (P - 1) * hop / n
        finish = red_end
    elif kind == "rs_naive":
        # every rank computes chunk c at step c; the partial is added to the incoming
        # accumulator when both are there (fused add: the step ends then)
        end = {}
        link_free = [0.0] * P
        arrive = {}
        for c in range(P):
            for h in range(P):
                r = (c + 1 + h) % P
                start = end.get((r, c - 1), 0.0)
                ready = start + comp
                if h > 0:
                    ready = max(ready, arrive[(r, c)])
                end[(r, c)] = ready
                if h < P - 1:
                    dst = (r + 1) % P
                    s = max(link_free[r], ready)
                    link_free[r] = s + hop
                    arrive[(dst, c)] = s + hop
        finish = max(end.values())
    else:
        raise ValueError(kind)
    return {"finish": finish, "compute": P * comp, "exposed": finish - P * comp}
