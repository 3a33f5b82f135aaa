"""Writes tests/golden/pr1_oracle.txt from the fp64 oracle alone.

The pages print no worked numeric example, so this fixture is a regression pin:
it freezes the oracle's output (and the seeded input recipe) on the smallest
attention workload (B=1, H=1, S=128, D=64, fp16, non-causal, seed 0, scale
1/8), so any later change to the oracle or to the input recipe shows up as a
diff.  It calls only ``oracle`` and the input generator.

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from attention_forward_gb300 import inputs  # noqa: E402

ROWS = (0, 1, 63, 64, 127)


def main():
    w = inputs.PR1
    q, k, v = (t.float().numpy() for t in w.make())
    o, lse = oracle.attention(q, k, v, w.scale, w.causal)
    lines = [f"# fp64 oracle, workload {w.name}, scale {w.scale!r}",
             "# lse: one value per query row 0..127",
             " ".join(f"{x:.17g}" for x in lse.reshape(-1))]
    for r in ROWS:
        lines.append(f"# O row {r}")
        lines.append(" ".join(f"{x:.17g}" for x in o[0, 0, r]))
    with open(os.path.join(HERE, "pr1_oracle.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
