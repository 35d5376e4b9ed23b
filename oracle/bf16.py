"""bf16 conversions for the oracle (test infrastructure only).

bf16 keeps float32's 8-bit exponent and 8 significant bits.  Values are stored
as uint16 bit patterns.
"""
import numpy as np

_MIN_NORMAL = 2.0 ** -126


def to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def from_f64(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bits, rounding once to nearest (ties to even).

    Rounds directly from float64 (no intermediate float32 rounding).  The
    oracle only meets zeros and normal, finite magnitudes; anything else raises.
    """
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value")
    nz = x != 0
    if np.any(np.abs(x[nz]) < _MIN_NORMAL * 2.0):
        raise ValueError("value outside the normal bf16 range")
    m, e = np.frexp(x)                 # x = m * 2**e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0)             # 8 significant bits, half to even
    y = np.ldexp(r, e - 8)             # exactly representable in bf16
    if np.any(np.abs(y) > 3.3895313892515355e38):
        raise ValueError("bf16 overflow")
    bits32 = y.astype(np.float32).view(np.uint32)
    return (bits32 >> np.uint32(16)).astype(np.uint16)


def ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place between two bit arrays."""
    def ordered(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - b, b)  # monotone integer ordering
    return np.abs(ordered(a_bits) - ordered(b_bits))
