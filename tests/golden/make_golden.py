"""Writes tests/golden/oracle_small.txt: oracle outputs for a small seeded case.

Calls only the oracle (and the seeded input generator).  The case is the
(B=2, T=2000, H=5) workload shape cut down to T=100 so that it holds one full
and one partial chunk per sequence.  Stored: every entry of the first and last
three rows of each chunk for head 0 and head 4, with their indices.

Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads  # noqa: E402

WL = workloads.CONFIGS["B2_T2000_H5_K128"].with_(name="golden_B2_T100_H5_K128", T=100)


def rows_to_store(wl):
    picks = []
    for n, c, h, r0, L in workloads.tile_list(wl):
        if h not in (0, wl.H - 1):
            continue
        for i in sorted({0, 1, 2, L - 3, L - 2, L - 1}):
            picks.append((r0 + i, h))
    return picks


def main():
    inp = workloads.make_inputs(WL)
    out = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], threads=1).reshape(-1, WL.H, 64)
    path = os.path.join(HERE, "oracle_small.txt")
    with open(path, "w") as f:
        f.write("# oracle (I+A)^-1 rows for the seeded workload B=2 T=100 H=5 K=128, seed 2, chunk 64\n")
        f.write("# definition: chunk-forward kkt_solve (MindSpeed-Ops PR #135 page, section 'What this PR does')\n")
        f.write("# written by tests/golden/make_golden.py, which calls only oracle/\n")
        f.write("# columns: token_row head then 64 values\n")
        for r, h in rows_to_store(WL):
            f.write(f"{r} {h} " + " ".join(repr(float(v)) for v in out[r, h]) + "\n")


if __name__ == "__main__":
    main()
