"""Writes the stored expected values under tests/golden/ from the oracle only.

    python tests/golden/make_golden.py

plan_llama7b_world8.txt: owner of each of the 224 matrices of the 32-layer
7B-shaped set (4 x 4096^2, 2 x 4096x11008, 1 x 11008x4096 per layer) on 8
ranks, NS k = 5, equal byte and flop weights -- the owner planner of
"Riassunto Tecnico: MatrixFSDP" §Metodologia 2 read as LPT greedy.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import planner  # noqa: E402
from workloads import llama7b_shapes  # noqa: E402


def main():
    owner, _ = planner.plan_owners(llama7b_shapes(), 8, 5)
    with open(os.path.join(HERE, "plan_llama7b_world8.txt"), "w") as f:
        f.write("# owner rank per matrix, index order; written by make_golden.py from "
                "oracle.planner (MatrixFSDP owner planner, LPT reading)\n")
        f.write(" ".join(str(o) for o in owner) + "\n")


if __name__ == "__main__":
    main()
