"""bfloat16 bit patterns -> float64 (exact).

Test infrastructure only (see the package docstring).

A bfloat16 value is the upper 16 bits of an IEEE float32, so widening is a
16-bit left shift followed by float32 -> float64, both exact.  NumPy has no
bfloat16 type, so the oracle takes bf16 tensors as ``uint16`` bit arrays.
"""

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen an array of bfloat16 bit patterns (uint16/int16) to float64."""
    b = np.asarray(bits)
    if b.dtype == np.int16:
        b = b.view(np.uint16)
    if b.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {b.dtype}")
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
