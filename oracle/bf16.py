"""bf16 storage format for the oracle (float64 values that are exactly bf16).

bf16 = 1 sign bit, 8 exponent bits, 7 stored mantissa bits: 8 significant bits.
The weights, the folded block weights and the KV cache are stored in this
format by the method ("Running VLAs at Real-time Speed", reading note, section
9: reproduce under BF16), so the oracle rounds to it exactly where the method
stores a value.
"""
import numpy as np


def decode(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact)."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_rne(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    x = m * 2**e with 0.5 <= |m| < 1 (frexp); keeping 8 significant bits means
    rounding m * 2**8 to an integer.  np.rint rounds half to even.  Values in the
    bf16 subnormal range (|x| < 2**-126) never occur on this path and are not
    treated specially.
    """
    x = np.asarray(x, dtype=np.float64)
    x32 = x.astype(np.float32)
    if np.array_equal(x32.astype(np.float64), x):
        # exactly a float32 (e.g. a product of two bf16 values): round the
        # 32-bit pattern, adding half an ulp of bf16 plus the tie-to-even bit
        u = x32.view(np.uint32)
        u = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) & np.uint32(0xFFFF0000)
        return u.view(np.float32).astype(np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def encode(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns after round_rne (sign, exponent, top 7 bits)."""
    r = round_rne(x).astype(np.float32)  # exact: r has 8 significant bits
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (normal range): 2**(floor(log2|x|) - 7)."""
    _, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(1.0, e - 8)
