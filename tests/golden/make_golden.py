"""Write the stored expected values under tests/golden/ from the fp64 oracle.

Run from the repository root:  python tests/golden/make_golden.py

The pages print no worked example for the cross-entropy path, so the stored
values come from the oracle (and nothing else) on the seeded tiny workload
(B=8, C=10, fp32 logits ~ N(0,1), targets uniform in [0, 10), seed 0).  The
fixture keeps its inputs as exact fp32 hex strings, so it stands on its own;
tests/test_golden.py re-derives every stored value with an independent
50-digit restatement.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads  # noqa: E402


def main() -> None:
    w = workloads.WORKLOADS_BY_NAME["tiny_8x10_f32"]
    inp = workloads.make_inputs(w)
    L, l, g = oracle.loss_and_grad(inp.logits, inp.targets)
    doc = {
        "workload": w.name,
        "source": "fp64 oracle (oracle/ce_oracle.c) via tests/golden/make_golden.py; "
                  "the pages print no worked example for this path",
        "B": w.B,
        "C": w.C,
        "logits_f32_hex": [[float(v).hex() for v in row] for row in inp.logits],
        "targets": [int(t) for t in inp.targets],
        "row_loss": [float(v).hex() for v in l],
        "loss": float(L).hex(),
        "grad": [[float(v).hex() for v in row] for row in g],
    }
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_8x10_f32.json")
    with open(out, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    print("wrote", out)


if __name__ == "__main__":
    main()
