"""Exact decoding of the 16-bit storage formats into float64 (oracle side).

IEEE binary16 values are widened by NumPy's own half type.  bfloat16 is the
upper half of an IEEE binary32 word, so widening is a 16-bit left shift
followed by a float32 -> float64 conversion; both steps are exact.
"""
import numpy as np


def decode_bits(bits, dtype: str) -> np.ndarray:
    """Return the float64 values held by an array of fp16 or bf16 bit patterns."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return b.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")
