"""Writes the stored schedule tables under tests/golden/ from the oracle only.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import schedule  # noqa: E402


def main():
    out = {"source": "oracle.schedule (FlashOverlap technical summary, section 2: Flash-AG local "
                     "slice first; Flash-RS kept slice last; ring r -> r+1)",
           "tables": {}}
    for P in (2, 4, 8):
        out["tables"][str(P)] = {
            "ag_slice": [[schedule.ag_slice(r, t, P) for t in range(P)] for r in range(P)],
            "rs_chunk": [[schedule.rs_chunk(r, t, P) for t in range(P)] for r in range(P)],
            "rs_chunk_naive": [[schedule.rs_chunk_naive(r, t, P) for t in range(P)] for r in range(P)],
        }
    with open(os.path.join(HERE, "schedules.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
