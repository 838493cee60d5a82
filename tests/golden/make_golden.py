"""Write the stored expected values under tests/golden/ from the float64 oracle.

Only the oracle and the seeded input generator are used.  The pages print no
numeric worked example for the selective scan, so these fixtures hold the
oracle's own result for the tiny fp32 workload (batch 1, 16 channels, 64
steps, 4 states; seed 0).  They guard the oracle against silent changes: any
later edit of its arithmetic has to regenerate them, and says why.

Run:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from selective_state_space_122_b300 import inputs  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
SEED = 0

HEADER = ("selective scan, tiny fp32 workload (batch 1, dim 16, L 64, N 4, seed 0): {what}\n"
          "definition: 'Mamba: Selective State Space Models' README, sections 'State Space Model', "
          "'Selective Mechanism', 'Efficient Scan' (sequential scan); dA = exp(Delta A), dB u = Delta B u, "
          "Delta = softplus(Delta_raw + delta_bias), y = C.h + D u, gated by silu(z)\n"
          "written by tests/golden/make_golden.py from the float64 oracle; shape {shape}")


def main():
    inp = inputs.make_scan_inputs(inputs.TINY_F32, SEED)
    f = inp.as_f64()
    out, last = oracle.scan(f["u"], f["delta"], f["A"], f["B"], f["C"], f["D"], f["z"],
                            f["delta_bias"], f["softplus"])
    np.savetxt(os.path.join(HERE, "tiny_f32_out.txt"), out.reshape(-1), fmt="%.17g",
               header=HEADER.format(what="out[b][t][d], flattened", shape=list(out.shape)))
    np.savetxt(os.path.join(HERE, "tiny_f32_last_state.txt"), last.reshape(-1), fmt="%.17g",
               header=HEADER.format(what="last_state[b][d][n], flattened", shape=list(last.shape)))


if __name__ == "__main__":
    main()
