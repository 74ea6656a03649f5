"""Write the frozen oracle output of the tiny workload (33 x 64 -> 176 -> 64, fp16, erf GELU).

Calls only the oracle and the seeded input generator.  The file it writes pins
the oracle against accidental change: a later edit of the oracle's arithmetic
must reproduce it, or regenerate it in a commit that names the passage or
reading that justifies the change.

    python tests/golden/make_tiny_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from transformer_mlp_gemms_gb300 import workloads as wl  # noqa: E402


def main():
    w = wl.WORKLOADS["tiny"]
    t = {k: wl.bits(v) for k, v in wl.generate(w).items()}
    H, _, Y = oracle.mlp(t["X"], t["W_up"], t["W_down"], act=w.act, dtype=w.dtype)
    path = os.path.join(HERE, "tiny_oracle_f16.txt")
    with open(path, "w") as f:
        f.write(f"# {w.describe()}\n# rows of H[{w.M},{w.F}] then Y[{w.M},{w.D}] as fp16 hex bit patterns\n")
        for name, arr in (("H", H), ("Y", Y)):
            for r in range(arr.shape[0]):
                f.write(name + " " + " ".join(f"{int(v):04x}" for v in arr[r]) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
