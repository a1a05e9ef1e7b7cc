"""CPU oracle for the lossless BF16 bit-field decomposition of expert weights.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference arm may import this module.  The CUDA library never calls it and
shares no code, table or constant with it.

  [ZipMoE]  "ZipMoE: Efficient On-Device MoE Serving via Lossless Compression and
            Cache-Affinity Scheduling" (paper summary page), method details: each BF16
            expert tensor is split into its exponent bits (low entropy, compressed on the
            host into E-chunks) and its sign and mantissa bits (near random, packed
            byte-aligned into SM-chunks); on the device the two parts are merged back
            into the original BF16 tensor, bit for bit.

BF16 layout (IEEE-754 binary32 truncated to its upper 16 bits): bit 15 sign, bits 14..7
exponent (bias 127), bits 6..0 mantissa.  Readings of open points:
  * one exponent byte per element (the decompressed E-chunk is the plain byte array);
  * one SM byte per element: the sign in bit 7 and the 7 mantissa bits in bits 6..0 --
    8 bits per element is exactly byte-aligned, the plainest packing the page allows;
  * the host-side compressors (LZ4 / ZSTD) are out of scope: the device path starts from
    decompressed bytes.
Pins: tests/test_bitfield_pins.py (hand-derived fields, the IEEE value formula, exhaustive
round trips over all 65536 patterns and all byte pairs).
"""
from __future__ import annotations

import numpy as np


def split(bits: np.ndarray):
    """BF16 bit patterns (uint16) -> (exponent bytes, sign|mantissa bytes), both uint8."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
    exp = (b >> 7) & 0xFF
    sm = ((b >> 15) << 7) | (b & 0x7F)
    return exp.astype(np.uint8), sm.astype(np.uint8)


def recombine(exp: np.ndarray, sm: np.ndarray) -> np.ndarray:
    """(exponent bytes, sign|mantissa bytes) -> BF16 bit patterns (uint16)."""
    e = np.asarray(exp, dtype=np.uint8).astype(np.uint32)
    s = np.asarray(sm, dtype=np.uint8).astype(np.uint32)
    return (((s >> 7) << 15) | (e << 7) | (s & 0x7F)).astype(np.uint16)


def value_of_fields(exp: int, sm: int) -> float:
    """The real number a (finite) BF16 with these fields denotes, from the IEEE definition."""
    sign = -1.0 if (sm >> 7) & 1 else 1.0
    mant = sm & 0x7F
    if exp == 0:
        return sign * (mant / 128.0) * 2.0 ** (-126)
    return sign * (1.0 + mant / 128.0) * 2.0 ** (exp - 127)


def exponent_entropy(exp: np.ndarray) -> float:
    """Shannon entropy (bits per element) of the exponent bytes: the redundancy the method
    compresses on the host (reported on the page as about 2.6 bits for real experts)."""
    counts = np.bincount(np.asarray(exp, dtype=np.uint8).ravel(), minlength=256).astype(np.float64)
    p = counts[counts > 0] / counts.sum()
    return float(-(p * np.log2(p)).sum())
