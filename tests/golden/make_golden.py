"""Write tests/golden/oracle_small_rows.txt from the fp64 oracle alone.

The snapshot pins the oracle plus the seeded input generator across hosts
(x86_64 where it was written, aarch64 where the GPU tests run): the same
seeded bits must give the same fp64 rows to ~1e-12.  Run:
    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from causal_scaled_dot_gb300.inputs import qkv_bf16  # noqa: E402
from causal_scaled_dot_gb300.workloads import SMALL  # noqa: E402

ROWS = [0, 1, 2, 63, 64, 127, 128, 129, 200, 255, 256, 257, 300, 383, 384, 511]
NDIM = 8


def main() -> None:
    w = SMALL
    q, k, v = qkv_bf16(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, sigma=w.sigma)
    out, lse = oracle.attention(q, k, v, w.scale, w.causal, rows=np.array(ROWS, np.int64))
    path = os.path.join(HERE, "oracle_small_rows.txt")
    with open(path, "w") as f:
        f.write(f"# workload {w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} S={w.S} D={w.D} "
                f"seed={w.seed} sigma={w.sigma} causal scale=1/sqrt(D)\n")
        f.write("# written by tests/golden/make_golden.py (fp64 oracle only)\n")
        f.write(f"# columns: flat_row lse out[0:{NDIM}]\n")
        for r, l, o in zip(ROWS, lse, out):
            f.write(f"{r} {l:.17e} " + " ".join(f"{x:.17e}" for x in o[:NDIM]) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
