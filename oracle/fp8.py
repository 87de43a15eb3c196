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
    with np.errstate(invalid="ignore"):   # signalling-NaN patterns convert to NaN, as they should
        return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- encoding
# The FP8 cache write ("Attention cache write" and "FP8 quantization: keep
# FP32 scale groups contiguous" in the MooreThreads/vllm-musa PR 178
# optimisation table) quantises each new latent row. The pages fix the
# element format and the contiguous fp32 group scales, not the scale rule;
# the plain reading taken here: per group of 128 latent dims,
# scale = amax / 448 (448 is the largest finite E4M3 value; scale 1 for an
# all-zero group), code = E4M3(x / scale) rounded to nearest, ties to even,
# saturating at +-448. The quantities that decide a code (amax, the scale,
# x / scale) are float32 values computed with float32 division, as a GPU
# kernel computes them; the rounding to E4M3 is then exact.

E4M3_MAX = 448.0
FP8_ROW_BYTES = 656   # [0, 512) codes, [512, 528) 4 float32 scales, [528, 656) 64 bf16 rope


def e4m3_encode(x):
    """float32 values -> uint8 E4M3 codes: nearest, ties to even, saturating.

    Normal codes hold (1 + m/8) * 2**(e - 7) for exponent field e in 1..15
    (e = 15 with m = 7 is NaN, so the largest finite value is 448); exponent
    field 0 holds m * 2**-9. NaN maps to the NaN code 0x7F (sign kept).
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x).astype(np.int64)
    a = np.abs(x)
    code = np.zeros(a.shape, dtype=np.int64)
    nan = np.isnan(a)
    sat = ~nan & (a >= E4M3_MAX)
    # Subnormal range: multiples of 2**-9 below 2**-6 (a multiple of 8 in
    # units of 2**-9 is the smallest normal, code 0x08, and comes out right).
    small = ~nan & ~sat & (a < 2.0 ** -6)
    m_sub = np.rint(np.where(small, a, 0.0) * 2.0 ** 9)   # exact scaling; rint ties to even
    code = np.where(small, m_sub.astype(np.int64), code)
    # Normal range: a = f * 2**E with f in [0.5, 1) (frexp is exact).
    norm = ~nan & ~sat & ~small
    f, E = np.frexp(np.where(norm, a, 1.0))
    e = E - 1                                      # a = (2 f) * 2**e, 2 f in [1, 2)
    m = np.rint((2.0 * f - 1.0) * 8.0)             # 3 mantissa bits, ties to even
    carry = m >= 8.0
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 0.0, m)
    ncode = (e + 7) * 8 + m.astype(np.int64)
    ncode = np.where(ncode > 0x7E, 0x7E, ncode)    # rounding up past 448 saturates
    code = np.where(norm, ncode, code)
    code = np.where(sat, 0x7E, code)
    code = np.where(nan, 0x7F, code)
    return (code | (sign << 7)).astype(np.uint8)


def quantize_latent_rows(latent_bits):
    """bfloat16 latent rows (uint16 bits [n, 576]) -> FP8 cache rows (uint8 [n, 656])."""
    bits = np.asarray(latent_bits, dtype=np.uint16)
    n = bits.shape[0]
    x = (bits[:, :512].astype(np.uint32) << np.uint32(16)).view(np.float32).reshape(n, 4, 128)
    amax = np.abs(x).max(axis=2)                                       # float32 [n, 4]
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = (x / scale[:, :, None]).astype(np.float32)                     # float32 division
    out = np.zeros((n, FP8_ROW_BYTES), dtype=np.uint8)
    out[:, :512] = e4m3_encode(q.reshape(n, 512))
    out[:, 512:528] = scale.astype("<f4").view(np.uint8).reshape(n, 16)
    out[:, 528:] = bits[:, 512:].astype("<u2").view(np.uint8).reshape(n, 128)
    return out


def kv_cache_write(pool, latent_bits, slots, kv_dtype):
    """Write new latent rows into a copy of the paged pool; returns (pool, flagged).

    Row i goes to slot ``slots[i]`` = page * 64 + offset ("[Bugfix] Make DSV4
    sparse MLA work end-to-end ...", section "What is fixed": slot =
    block_id * block_size + offset). A negative slot is a padding row and is
    skipped (the null-block guard the same section calls for); a slot beyond
    the pool is skipped and reported in ``flagged``.
    """
    pool = np.array(pool, copy=True)
    slots = np.asarray(slots, dtype=np.int64)
    num_slots = pool.shape[0] * pool.shape[1]
    flat = pool.reshape(num_slots, -1)
    rows = quantize_latent_rows(latent_bits) if kv_dtype == "fp8" else \
        np.asarray(latent_bits, dtype=np.uint16)
    flagged = False
    for i, s in enumerate(slots):
        if s < 0:
            continue
        if s >= num_slots:
            flagged = True
            continue
        flat[s] = rows[i]
    return pool, flagged
