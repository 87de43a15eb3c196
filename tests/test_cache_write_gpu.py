"""GPU parity of ds_kv_cache_write against the oracle: byte-exact pools.

New latent rows go to slots page * 64 + offset of a paged pool; FP8 pools get
the quantised layout (E4M3 codes, four contiguous fp32 group scales, bf16
rope). Covers random rows, all-zero and single-value groups, values that
saturate or fall to subnormal codes, signed zeros, quotients on and next to
E4M3 rounding midpoints under scales with inexact reciprocals, padding slots
(-1, never written), slots past the pool (flagged, not written), untouched slots, and a
read-back through the FP8 attention path.
"""

import numpy as np
import pytest
import torch

import oracle
from harness import assert_close, ensure_built, kv_np, q_bits
from synthetic import decode_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def ds():
    return ensure_built()


def _rows(n, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, 576), generator=g) * torch.exp(torch.randn((n, 1), generator=g) * 3)
    x[0] = 0.0                                  # all groups zero
    x[1, :128] = 0.0
    x[1, 5] = -3.25                             # a group with one value
    x[2, 128:256] = torch.linspace(-1e30, 1e30, 128)   # huge range: tiny values go subnormal
    x[3, 256:384] = -0.0
    x[3, 300] = 1e-30
    return x.to(torch.bfloat16)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("kv_dtype", ["fp8", "bf16"])
def test_cache_write_exact(ds, kv_dtype):
    pages, n = 40, 700
    rng = np.random.default_rng(7)
    slots = rng.choice(pages * 64, n, replace=False).astype(np.int64)
    slots[::37] = -1                            # padding rows
    slots[5] = pages * 64 + 3                   # past the pool: flagged
    latent = _rows(n, 8).to(DEV)
    if kv_dtype == "fp8":
        pool = torch.randint(0, 256, (pages, 64, 656), dtype=torch.uint8, device=DEV)
    else:
        pool = torch.randint(-3000, 3000, (pages, 64, 576), dtype=torch.int16,
                             device=DEV).view(torch.bfloat16)
    before = kv_np(pool, kv_dtype)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ds.kv_cache_write(latent, torch.as_tensor(slots).to(DEV), pool, kv_dtype, err_flag=err)
    torch.cuda.synchronize()
    want, flagged = oracle.kv_cache_write(before, _bits(latent), slots, kv_dtype)
    got = kv_np(pool, kv_dtype)
    bad = np.nonzero((got != want).reshape(pages * 64, -1).any(1))[0]
    assert bad.size == 0, f"slots differ: {bad[:10].tolist()}"
    assert flagged and int(err.item()) == ds.DEVERR_PAGE


def _boundary_rows(n, seed):
    """bf16 latent rows whose groups have scales odd * 2**k (amax = 448 * scale,
    exactly representable) and whose other values are bf16(scale * v) and its
    bf16 neighbours, v an E4M3 value or a midpoint between two: quotients on or
    within a few float32 units of E4M3 rounding boundaries, where a quotient
    taken as x * (1 / scale) can round to another code than x / scale."""
    rng = np.random.default_rng(seed)
    vals = oracle.e4m3_to_float64(np.arange(0x7F, dtype=np.uint8))
    targets = np.concatenate([vals, (vals[:-1] + vals[1:]) / 2])
    odds = [3, 5, 7, 9, 11, 13, 15, 17, 19, 21, 23, 25, 27, 29, 31, 33, 35]
    bits = np.zeros((n, 576), np.uint16)
    for r in range(n):
        for g in range(4):
            scale = float(rng.choice(odds)) * 2.0 ** int(rng.integers(-24, 25))
            amax = np.float32(448.0 * scale)
            v = rng.choice(targets, 127) * scale * rng.choice([-1.0, 1.0], 127)
            b = (np.asarray(v, np.float32).view(np.uint32) + 0x8000) >> 16   # to bf16 (half up)
            b = (b.astype(np.int64) + rng.integers(-1, 2, 127)) & 0xFFFF       # a bf16 step either way
            x = (b.astype(np.uint32) << 16).view(np.float32)
            b = np.where(np.abs(x) <= amax, b, 0)                              # keep |x| <= amax
            row = np.concatenate([[amax.view(np.uint32) >> 16], b]).astype(np.uint16)
            bits[r, 128 * g:128 * (g + 1)] = rng.permutation(row)
        bits[r, 512:] = rng.integers(0, 0x7F00, 64)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


def test_cache_write_fp8_rounding_boundaries(ds):
    # Quotients at and next to E4M3 rounding midpoints, under scales whose
    # reciprocals are inexact: every code still matches the float32 division.
    n = 512
    latent = _boundary_rows(n, 21).to(DEV)
    pool = torch.zeros((n // 64, 64, 656), dtype=torch.uint8, device=DEV)
    ds.kv_cache_write(latent, torch.arange(n, device=DEV), pool, "fp8")
    torch.cuda.synchronize()
    want = oracle.quantize_latent_rows(_bits(latent.cpu()))
    got = kv_np(pool, "fp8").reshape(n, 656)
    bad = np.nonzero((got != want).any(1))[0]
    assert bad.size == 0, f"rows differ: {bad[:10].tolist()}"


def test_written_fp8_rows_read_back_through_attention(ds):
    # Quantise a bf16 pool's rows into an FP8 pool with the write kernel, then
    # run FP8 decode on it: the result matches the oracle on the same bytes.
    c = decode_case("wr", [3000, 1500], 64, 512, "bf16", seed=12, device="cuda")
    P = c.kv_pages.shape[0]
    fp8 = torch.zeros((P, 64, 656), dtype=torch.uint8, device=DEV)
    ds.kv_cache_write(c.kv_pages.reshape(P * 64, 576), torch.arange(P * 64, device=DEV), fp8,
                      "fp8")
    torch.cuda.synchronize()
    assert np.array_equal(kv_np(fp8, "fp8").reshape(P * 64, 656),
                          oracle.quantize_latent_rows(_bits(c.kv_pages.reshape(P * 64, 576))))
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    out, lse = ds.sparse_mla_decode(c.q, fp8, "fp8", c.block_table, idx, c.lens, c.scale)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.sparse_mla_decode(q_bits(c.q), kv_np(fp8, "fp8"), "fp8",
                                            c.block_table.cpu().numpy(), idx.cpu().numpy(),
                                            c.lens.cpu().numpy(), c.scale)
    assert_close(out, lse, ref, ref_lse, "fp8", "write_then_read")


def test_empty_write_is_a_noop(ds):
    pool = torch.zeros((1, 64, 656), dtype=torch.uint8, device=DEV)
    ds.kv_cache_write(torch.zeros((0, 576), dtype=torch.bfloat16, device=DEV),
                      torch.zeros(0, dtype=torch.int64, device=DEV), pool, "fp8")
    torch.cuda.synchronize()
    assert int(pool.sum()) == 0
