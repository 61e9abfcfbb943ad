"""The oracle against values the pages and the mathematics fix (CPU only)."""
import os

import numpy as np
import pytest

import oracle
import oracle_pins
from tensor_core_gemm_02_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_golden_worked_example_file():
    """tests/golden/worked_16x8x32.txt was written by make_golden.py from the oracle.

    It fixes the expected D of the "mma.sync" page's worked example so the GPU
    tests do not need the oracle for this case; here it must agree with the
    oracle and with exact arithmetic.
    """
    stored = np.loadtxt(os.path.join(GOLDEN, "worked_16x8x32.txt"), dtype=np.float64)
    p = workloads.worked_16x8x32()
    ref, _, _ = oracle.gemm(p.A, p.B)
    assert stored.shape == (16, 8)
    assert np.array_equal(stored, ref)
    assert np.array_equal(stored.astype(np.float32).astype(np.float64), stored)


def test_golden_tma_example_file():
    """The "cp.async.bulk.tensor" page's copy example: x = arange(256) as 16 x 16 uint32."""
    stored = np.loadtxt(os.path.join(GOLDEN, "tma_copy_16x16.txt"), dtype=np.int64)
    assert np.array_equal(stored, np.arange(256).reshape(16, 16))


def test_workload_recipes_are_deterministic():
    a = workloads.worked_16x8x32()
    b = workloads.worked_16x8x32()
    assert (a.A == b.A).all() and (a.B == b.B).all()
    assert a.A.shape == (16, 32) and a.B.shape == (8, 32)
    vals = set((a.A.float() * 4).flatten().tolist())
    assert vals <= set(range(-4, 5))


def test_prefix_draw_property():
    """Drawing fewer rows yields the leading rows of the larger draw (used for C[:16])."""
    r1 = np.random.default_rng(3).standard_normal((40, 33), dtype=np.float32)
    r2 = np.random.default_rng(3).standard_normal((16, 33), dtype=np.float32)
    assert np.array_equal(r1[:16], r2)
