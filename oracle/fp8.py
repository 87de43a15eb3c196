"""Exact decoding of the stored KV element formats (test infrastructure only).

The FP8 KV cache of the pages ("--kv-cache-dtype fp8", scale groups of 128
elements kept contiguous; MooreThreads/vllm-musa PR 178, optimisation table)
stores the latent as OCP FP8 E4M3 ("e4m3fn": no infinities) with one float32
scale per 128-element group. The oracle decodes the stored bytes exactly from
the format definition, in float64:

* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
  subnormal, ``m * 2**-9``; exponent 15 with mantissa 7 is NaN; no infinity.
* bfloat16: the upper 16 bits of an IEEE-754 binary32.
"""

import numpy as np


def e4m3_to_float64(codes):
    """Decode uint8 E4M3 codes to float64, element by element."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    sub = man.astype(np.float64) * 2.0 ** -9
    norm = (1.0 + man.astype(np.float64) / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    val = np.where(exp == 0, sub, norm)
    val = np.where((exp == 15) & (man == 7), np.nan, val)
    return sign * val


def bf16_bits_to_float64(bits):
    """Decode uint16 bfloat16 bit patterns to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)
