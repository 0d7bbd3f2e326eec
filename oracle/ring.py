"""Explicit simulated ring for the oracle (test infrastructure only).

FlashOverlap (technical summary, section 2) replaces each collective by
asynchronous ring P2P transfers.  The simulation keeps one FIFO per directed
link.  Every message carries a sequence tag (the hop index) and the index of
the slice or chunk it carries; every send copies its payload into a fresh
buffer (a per-step receive buffer), so no rank ever aliases another rank's
data.  A receive checks both tags, so a dropped, duplicated or reordered
message raises ``RingError`` instead of silently changing the result.

``fault`` is a test hook: ``fault(src, dst, message) -> list[message]``
decides what actually enters the link (``[]`` drops, ``[m, m]`` duplicates).
"""
from __future__ import annotations

import collections
import dataclasses

import numpy as np


class RingError(RuntimeError):
    pass


@dataclasses.dataclass
class Message:
    seq: int
    item: int
    payload: np.ndarray


class Ring:
    def __init__(self, P: int, direction: int = 1, fault=None):
        if direction not in (1, -1):
            raise ValueError("direction must be +1 or -1")
        self.P = P
        self.direction = direction
        self.fault = fault
        self.inbox = [collections.deque() for _ in range(P)]
        self.log = []            # (src, dst, seq, item) of every send

    def dst(self, src: int) -> int:
        return (src + self.direction) % self.P

    def send(self, src: int, seq: int, item: int, payload: np.ndarray) -> None:
        msg = Message(seq, item, np.array(payload, copy=True))
        dst = self.dst(src)
        msgs = [msg] if self.fault is None else self.fault(src, dst, msg)
        self.inbox[dst].extend(msgs)
        self.log.append((src, dst, seq, item))

    def send_to(self, src: int, dst: int, seq: int, item: int, payload: np.ndarray) -> None:
        """A direct P2P message to any rank (the decomposed all-to-all's step t sends to
        rank src + t); same tagging and fault hook as ``send``."""
        msg = Message(seq, item, np.array(payload, copy=True))
        msgs = [msg] if self.fault is None else self.fault(src, dst, msg)
        self.inbox[dst].extend(msgs)
        self.log.append((src, dst, seq, item))

    def recv(self, dst: int, seq: int, item: int) -> np.ndarray:
        q = self.inbox[dst]
        if not q:
            raise RingError(f"rank {dst}: no message (expected seq={seq}, item={item})")
        msg = q.popleft()
        if msg.seq != seq or msg.item != item:
            raise RingError(f"rank {dst}: got seq={msg.seq} item={msg.item}, "
                            f"expected seq={seq} item={item}")
        return msg.payload

    def check_drained(self) -> None:
        for r, q in enumerate(self.inbox):
            if q:
                m = q[0]
                raise RingError(f"rank {r}: unexpected extra message seq={m.seq} item={m.item}")
