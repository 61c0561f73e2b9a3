"""Writes tests/golden/config0_oracle.npz: the fp64 oracle's outputs on the
tiny fp32 workload (1 sequence, 1 head, dk = dv = 32, 8-node tree with
parent[i] uniform in [-1, i-1], seed 1000).  Calls only the oracle and the
input generators.  The pages print no worked example for this path, so this
file is a regression record of the pinned oracle, not an independent pin."""

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads as W  # noqa: E402


def main():
    w = W.make_config(0)
    o, U = oracle.verify_workload(w, mode="path")
    S1 = oracle.commit_workload(w)
    np.savez(os.path.join(HERE, "config0_oracle.npz"), o=o, U=U, S1=S1,
             parent=w.parent, path=w.path, path_len=w.path_len)


if __name__ == "__main__":
    main()
