"""GPU parity of ds_kv_cache_write against the oracle: byte-exact pools.

New latent rows go to slots page * 64 + offset of a paged pool; FP8 pools get
the quantised layout (E4M3 codes, four contiguous fp32 group scales, bf16
rope). Covers random rows, all-zero and single-value groups, values that
saturate or fall to subnormal codes, signed zeros, padding slots (-1, never
written), slots past the pool (flagged, not written), untouched slots, and a
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
