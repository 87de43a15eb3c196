"""Pins of the oracle's FP8 cache-write quantiser (oracle/fp8.py).

The encoder is checked against things other than itself: the exact decoder
over every code, torch's float8_e4m3fn conversion (a library routine) on
random values, exact ties and subnormals, the saturation rule of the format
definition, closed forms of the row quantiser, and the E4M3 rounding bound.
"""

import numpy as np
import torch

import oracle


def test_every_finite_code_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_to_float64(codes)
    fin = np.isfinite(v)
    assert np.array_equal(oracle.e4m3_encode(v[fin].astype(np.float32)), codes[fin])
    assert fin.sum() == 254   # 0x7F and 0xFF are NaN


def test_matches_torch_conversion_including_ties_and_subnormals():
    rng = np.random.default_rng(0)
    finite = oracle.e4m3_to_float64(np.arange(256, dtype=np.uint8))
    finite = np.unique(finite[np.isfinite(finite)])
    mids = ((finite[1:] + finite[:-1]) / 2).astype(np.float32)      # exact ties
    near = np.concatenate([np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(-np.inf))]).astype(np.float32)
    rand = np.concatenate([rng.standard_normal(50000) * 40, rng.standard_normal(20000) * 2e-3,
                           rng.uniform(-448, 448, 20000)]).astype(np.float32)
    x = np.clip(np.concatenate([mids, near, rand]), -448, 448).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), want)


def test_saturation_and_specials():
    enc = oracle.e4m3_encode(np.array([448, 449, 464, 1e9, -500, 0.0, -0.0, np.nan, 2 ** -10,
                                       3 * 2 ** -10], np.float32))
    assert enc.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x00, 0x80, 0x7F, 0x00, 0x02]


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_row_quantiser_closed_forms():
    x = np.zeros((3, 576), np.float32)
    x[0, :128] = np.linspace(-448, 448, 128)     # group max 448: scale 1
    x[0, 128:256] = 0.0                          # all-zero group: scale 1, codes 0
    x[0, 256:384] = 2.0 ** -20                   # one value: scale = v / 448
    x[0, 384:512] = -3.5
    x[0, 512:] = np.arange(64)                   # rope
    x[1] = np.random.default_rng(1).standard_normal(576) * 7
    x[2, :512] = 1e-3 * np.random.default_rng(2).standard_normal(512)
    bits = _bf16_bits(x)
    rows = oracle.quantize_latent_rows(bits)
    assert rows.shape == (3, 656) and rows.dtype == np.uint8
    scales = rows[:, 512:528].copy().view("<f4").reshape(3, 4)
    xv = oracle.bf16_bits_to_float64(bits).astype(np.float32)
    assert scales[0, 0] == 1.0 and scales[0, 1] == 1.0
    assert scales[0, 2] == np.float32(xv[0, 256]) / np.float32(448)
    assert (rows[0, 128:256] == 0).all()
    assert np.array_equal(rows[0, :128], oracle.e4m3_encode(xv[0, :128]))
    assert np.array_equal(rows[:, 528:].copy().view("<u2"), bits[:, 512:])   # rope bit-exact
    # Every element decodes to within half an E4M3 step of x / scale.
    codes = oracle.e4m3_to_float64(rows[:, :512]).reshape(3, 4, 128)
    q = xv[:, :512].reshape(3, 4, 128) / scales[:, :, None].astype(np.float64)
    step = np.where(np.abs(q) < 2 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.abs(q) + 1e-300)) - 3))
    assert np.all(np.abs(codes - q) <= step / 2 * (1 + 1e-6))


def test_cache_write_slots():
    pool = np.full((3, 64, 656), 0xAB, np.uint8)
    bits = _bf16_bits(np.random.default_rng(3).standard_normal((4, 576)))
    new, flagged = oracle.kv_cache_write(pool, bits, [5, -1, 64 * 3, 130], "fp8")
    rows = oracle.quantize_latent_rows(bits)
    flat = new.reshape(192, 656)
    assert flagged                                      # slot 192 is past the pool
    assert np.array_equal(flat[5], rows[0]) and np.array_equal(flat[130], rows[3])
    untouched = np.ones(192, bool)
    untouched[[5, 130]] = False
    assert (flat[untouched] == 0xAB).all()              # padding (-1) and the flagged row skipped
    pool16 = np.zeros((2, 64, 576), np.uint16)
    new16, f16 = oracle.kv_cache_write(pool16, bits, [0, 127, -5, 64], "bf16")
    assert not f16 and np.array_equal(new16.reshape(128, 576)[[0, 127, 64]], bits[[0, 1, 3]])
