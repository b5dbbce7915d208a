"""Arithmetic identities the CUDA path relies on, checked exhaustively on CPU.

The drafter reports a chain probability c / c0 and a score sum / c0 as the
float nearest to the double quotient (the oracle's definition).  The kernel
divides in single precision: with integers c <= 64 * c0 (k <= 64 depths) and
c0 <= 128 (max_occurrences), both operands are exact floats and a correctly
rounded single division lands on the same float as rounding the correctly
rounded double quotient.  This test checks every such pair.
"""
import numpy as np


def test_single_division_equals_rounded_double_quotient():
    for c0 in range(1, 129):
        num = np.arange(0, 64 * c0 + 1, dtype=np.int64)
        via_double = (num.astype(np.float64) / np.float64(c0)).astype(np.float32)
        via_single = num.astype(np.float32) / np.float32(c0)
        assert np.array_equal(via_double.view(np.uint32), via_single.view(np.uint32)), c0
