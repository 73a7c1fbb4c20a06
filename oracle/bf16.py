"""bf16 storage rounding for the oracle (test infrastructure only).

The CUDA path stores every activation in bf16; the oracle computes in fp64
and rounds to the nearest bf16 value (ties to even) at the same points, so
that the two chains stay comparable.  Written from the definition of the
format (8 significant bits, exponent range of fp32), not from any library.
"""
import numpy as np


def decode(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    A finite x = m * 2**e with 0.5 <= |m| < 1 has bf16 quantum 2**(e - 8)
    for normal results; below 2**-126 the quantum stays at 2**-133
    (subnormal bf16).  Magnitudes past the largest finite bf16 become inf.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    quantum = np.ldexp(1.0, e - 8)
    r = np.rint(x / quantum) * quantum          # np.rint rounds half to even
    max_bf16 = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > max_bf16, np.copysign(np.inf, r), r)
    return np.where(x == 0, x, r)
