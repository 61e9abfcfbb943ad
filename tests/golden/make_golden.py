"""Writes the stored expected values under tests/golden/ (calls only oracle/).

    python tests/golden/make_golden.py

worked_16x8x32.txt  D of the "mma.sync" page's worked example ("Example: a
                    16x8 result with two K16 issues"): inputs regenerated from
                    the page's recipe (default_rng(0), integers in [-4, 4] / 4,
                    16 x 32 and 8 x 32, f16), D = a @ b.T computed by the oracle.
tma_copy_16x16.txt  the "cp.async.bulk.tensor" page's copy example ("Example:
                    two explicit 8x16 boxes"): x = arange(256) as 16 x 16
                    uint32, which the copy must reproduce unchanged.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from tensor_core_gemm_02_gb300 import workloads  # noqa: E402


def main():
    p = workloads.worked_16x8x32()
    ref, _, _ = oracle.gemm(p.A, p.B)
    np.savetxt(os.path.join(HERE, "worked_16x8x32.txt"), ref, fmt="%.4f",
               header="D = a @ b.T for the mma.sync page's worked example (16 x 8, exact)")
    np.savetxt(os.path.join(HERE, "tma_copy_16x16.txt"), np.arange(256).reshape(16, 16),
               fmt="%d", header="cp.async.bulk.tensor page copy example: arange(256) as 16 x 16")


if __name__ == "__main__":
    main()
