"""Writes the stored expected values under tests/golden/ (calls only the CPU
oracle and the seeded input generators).

  spans_<workload>_g<max_gap>.txt : the ordered active spans of each
      workload's loss mask, one "start end" pair per line (half-open).
  tiny_fp32_forward.txt : logprob, entropy, lse of the tiny fp32 workload
      (float64, repr precision), one row per token.

Run:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from entropy_active_span_gb300 import workloads  # noqa: E402
from oracle import active_spans, lmhead_forward  # noqa: E402


def main():
    for name, w in workloads.WORKLOADS.items():
        mask = workloads.make_mask(w)
        for g in (0, 128):
            sp = active_spans(mask, g)
            with open(os.path.join(HERE, f"spans_{name}_g{g}.txt"), "w") as f:
                f.write(f"# active spans of the {name} loss mask (seed {w.seed}), "
                        f"max_gap={g}; {len(sp)} spans, half-open [start end)\n")
                for s, e in sp:
                    f.write(f"{s} {e}\n")
    inp = workloads.make_inputs("tiny_fp32")
    lp, ent, lse = lmhead_forward(workloads.to_f64(inp["hidden"]), workloads.to_f64(inp["weight"]),
                                  inp["targets"], inp["mask"])
    with open(os.path.join(HERE, "tiny_fp32_forward.txt"), "w") as f:
        f.write("# tiny_fp32 workload (seed 1001): token logprob entropy lse (float64 oracle)\n")
        for i in range(len(lp)):
            f.write(f"{i} {float(lp[i])!r} {float(ent[i])!r} {float(lse[i])!r}\n")


if __name__ == "__main__":
    main()
