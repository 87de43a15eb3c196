"""GPU parity of ds_sparse_mla_decode / ds_sparse_mla_prefill against the oracle.

Tolerance (per element): |gpu - ref| <= atol + 1e-2 |ref|, atol 2e-2 for
bf16 KV and 4e-2 for FP8 KV; lse within 1e-2; the reading of "max abs err
2e-2 and rel err 1e-2 for bf16 and 4e-2 for FP8 KV".

Covers every head count and several k (one tile, several tiles, several
splits, a ragged last split), both KV formats, rows shorter than k (-1
tails), empty rows, invalid entries (skipped and flagged), the closed forms
(one entry returns its V row exactly; q = 0 gives the mean of V), the named
workloads at full size (sampled rows where the oracle would be slow), and
bitwise batch invariance ("Sparse MLA and FlashMLA", PR 54955: the result
must not depend on the other requests in the batch).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from harness import assert_close, compact_rows, ensure_built, kv_np, q_bits
from synthetic import decode_case, invariance_batch, workload_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def ds():
    return ensure_built()


def oracle_idx(c):
    return oracle.topk_per_row(c.np_scores(), c.np_int("row_starts"), c.np_int("row_ends"), c.k)


def run_decode(ds, c, idx, err=None):
    out, lse = ds.sparse_mla_decode(c.q, c.kv_pages, c.kv_dtype, c.block_table,
                                    torch.as_tensor(idx).to(DEV), c.lens, c.scale, err_flag=err)
    torch.cuda.synchronize()
    return out, lse


def oracle_decode(c, idx, rows=None):
    return oracle.sparse_mla_decode(q_bits(c.q), kv_np(c.kv_pages, c.kv_dtype), c.kv_dtype,
                                    c.block_table.cpu().numpy(), idx, c.lens.cpu().numpy(),
                                    c.scale, rows=rows)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("H", [16, 32, 64, 128])
@pytest.mark.parametrize("k", [64, 192, 640, 2048])
def test_decode_small_parity(ds, H, k, kv):
    # Contexts around k: longer, equal, shorter (-1 tail), one page, empty.
    ctx = [3 * k + 17, k, max(1, k // 2 + 5), 64, 0]
    c = decode_case(f"small_{H}_{k}_{kv}", ctx, H, k, kv, seed=H * 7 + k, score_mode="eighths",
                    stride=max(ctx) + 3, device="cuda")
    idx = oracle_idx(c)
    out, lse = run_decode(ds, c, idx)
    ref, ref_lse = oracle_decode(c, idx)
    assert_close(out, lse, ref, ref_lse, kv, f"H={H} k={k} {kv}")
    assert (out[4] == 0).all() and torch.isneginf(lse[4]).all()


def test_tiny_decode_named(ds):
    c = workload_case("tiny_decode", device="cuda")
    idx = oracle_idx(c)
    out, lse = run_decode(ds, c, idx)
    ref, ref_lse = oracle_decode(c, idx)
    assert_close(out, lse, ref, ref_lse, "bf16", "tiny_decode")


def test_tp2_decode_full(ds):
    c = workload_case("tp2_decode", device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    out, lse = run_decode(ds, c, idx)
    ref, ref_lse = oracle_decode(c, idx.cpu().numpy())
    assert_close(out, lse, ref, ref_lse, "bf16", "tp2_decode")


def test_tp1_fp8_decode_sampled(ds):
    c = workload_case("tp1_fp8_decode", device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    out, lse = run_decode(ds, c, idx)
    rows = [0, 1, 63, 64, 127] + np.random.default_rng(1).choice(128, 5, replace=False).tolist()
    qb, kv, bt, idx_s, lens = compact_rows(c, rows, idx.cpu().numpy())
    ref, ref_lse = oracle.sparse_mla_decode(qb, kv, "fp8", bt, idx_s, lens, c.scale)
    assert_close(out[rows], lse[rows], ref, ref_lse, "fp8", "tp1_fp8_decode")


def test_chunked_prefill_sampled(ds):
    c = workload_case("chunked_prefill", device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    del c.scores
    out, lse = ds.sparse_mla_prefill(c.q, c.kv_pages, c.kv_dtype, c.block_table, c.row_req, idx,
                                     c.lens, c.scale)
    torch.cuda.synchronize()
    rows = [0, 1, 2047, 4095] + np.random.default_rng(2).choice(4096, 4, replace=False).tolist()
    qb, kv, bt, idx_s, lens = compact_rows(c, rows, idx.cpu().numpy())
    ref, ref_lse = oracle.sparse_mla_decode(qb, kv, "bf16", bt, idx_s, lens, c.scale)
    assert_close(out[rows], lse[rows], ref, ref_lse, "bf16", "chunked_prefill")


def test_prefill_small_parity(ds):
    # Two requests; tokens point at either one; causal lengths.
    c0 = decode_case("pf", [700, 1500], 64, 256, "bf16", seed=9, device="cuda")
    T = 6
    row_req = torch.tensor([1, 0, 1, 1, 0, 1], dtype=torch.int32, device=DEV)
    lens = torch.tensor([1500, 700, 3, 1200, 64, 0], dtype=torch.int32, device=DEV)
    g = torch.Generator().manual_seed(10)
    q = torch.randn((T, 64, 576), generator=g).to(torch.bfloat16).to(DEV)
    sc = torch.randn((T, 1500), generator=g)
    idx = oracle.topk_per_row(sc.numpy(), np.zeros(T), lens.cpu().numpy(), 256)
    out, lse = ds.sparse_mla_prefill(q, c0.kv_pages, "bf16", c0.block_table, row_req,
                                     torch.as_tensor(idx).to(DEV), lens, c0.scale)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.sparse_mla_prefill(q_bits(q), kv_np(c0.kv_pages, "bf16"), "bf16",
                                             c0.block_table.cpu().numpy(), row_req.cpu().numpy(),
                                             idx, lens.cpu().numpy(), c0.scale)
    assert_close(out, lse, ref, ref_lse, "bf16", "prefill_small")


def test_single_entry_returns_v_row_exactly(ds):
    c = decode_case("one", [500, 500], 64, 128, "bf16", seed=11, device="cuda")
    idx = np.full((2, 128), -1, np.int32)
    idx[0, 0] = 321
    idx[1, 0] = 5
    out, lse = run_decode(ds, c, idx)
    bt = c.block_table.cpu().numpy()
    for r, pos in [(0, 321), (1, 5)]:
        v = c.kv_pages[int(bt[r, pos // 64]), pos % 64, :512]
        assert torch.equal(out[r], v.expand(64, 512))
    ref, ref_lse = oracle_decode(c, idx)
    assert np.abs(lse.cpu().numpy() - ref_lse).max() < 1e-2


def test_zero_query_gives_mean_of_v(ds):
    c = decode_case("mean", [3000], 32, 1024, "bf16", seed=12, device="cuda")
    c.q.zero_()
    idx = oracle_idx(c)
    out, lse = run_decode(ds, c, idx)
    bt = c.block_table.cpu().numpy()[0]
    pos = idx[0][idx[0] >= 0]
    V = oracle.gather_latent_rows(kv_np(c.kv_pages, "bf16"), "bf16", bt, pos)[:, :512]
    mean = V.mean(axis=0)
    assert np.abs(out[0].float().cpu().numpy() - mean[None]).max() <= 2e-2
    assert np.abs(lse[0].cpu().numpy() - math.log(len(pos))).max() <= 1e-3


def test_invalid_entries_skipped_and_flagged(ds):
    c = decode_case("bad", [1000, 1000, 1000], 64, 256, "bf16", seed=13, device="cuda")
    idx = oracle_idx(c)
    bad = idx.copy()
    bad[0, 3] = 5000          # beyond lens: skipped, DS_DEVERR_IDX
    bad[1, 7] = -5            # negative but not -1: skipped, DS_DEVERR_IDX
    c.block_table[2, 1] = 10 ** 6   # page out of range for positions 64..127
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = run_decode(ds, c, bad, err=err)
    flags = int(err.item())
    assert flags & ds.DEVERR_IDX and flags & ds.DEVERR_PAGE
    assert not flags & ds.DEVERR_TIMEOUT
    ref, ref_lse = oracle_decode(c, bad)
    assert_close(out, lse, ref, ref_lse, "bf16", "invalid entries")


def test_batch_invariance_bitwise(ds):
    ref = None
    for B in [1, 7, 64, 256]:
        for slot in sorted({0, B // 2, B - 1}):
            c = invariance_batch(B, slot, device="cuda")
            idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
            out, lse = ds.sparse_mla_decode(c.q, c.kv_pages, "bf16", c.block_table, idx, c.lens,
                                            c.scale)
            got = (idx[slot].cpu(), out[slot].cpu(), lse[slot].cpu())
            if ref is None:
                ref = got
                qb, kv, bt, idx_s, lens = compact_rows(c, [slot], idx.cpu().numpy())
                r_out, r_lse = oracle.sparse_mla_decode(qb, kv, "bf16", bt, idx_s, lens, c.scale)
                assert_close(out[[slot]], lse[[slot]], r_out, r_lse, "bf16", "invariance target")
            assert torch.equal(got[0], ref[0]), (B, slot)
            assert torch.equal(got[1].view(torch.int16), ref[1].view(torch.int16)), (B, slot)
            assert torch.equal(got[2].view(torch.int32), ref[2].view(torch.int32)), (B, slot)


def test_run_to_run_bitwise(ds):
    c = workload_case("tp2_decode", device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    a = run_decode(ds, c, idx)
    b = run_decode(ds, c, idx)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))


def test_batch_invariance_bitwise_fp8_h128(ds):
    # The TP1 shape: FP8 KV, 128 heads (two head-group CTAs per split, each
    # gathering its own copy of every tile), top-k 2048, contexts up to 128K.
    # One request alone and at random slots of batches of 7 and 64.
    rng = np.random.default_rng(21)
    ref = None
    for B in [1, 7, 64]:
        for slot in sorted({int(x) for x in rng.integers(0, B, 2)}):
            c = invariance_batch(B, slot, target_seed=5, batch_seed=6, device="cuda", H=128,
                                 target_ctx=65536, max_ctx=131072, kv_dtype="fp8")
            idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
            out, lse = ds.sparse_mla_decode(c.q, c.kv_pages, "fp8", c.block_table, idx, c.lens,
                                            c.scale)
            got = (idx[slot].cpu(), out[slot].cpu(), lse[slot].cpu())
            if ref is None:
                ref = got
                qb, kv, bt, idx_s, lens = compact_rows(c, [slot], idx.cpu().numpy())
                r_out, r_lse = oracle.sparse_mla_decode(qb, kv, "fp8", bt, idx_s, lens, c.scale)
                assert_close(out[[slot]], lse[[slot]], r_out, r_lse, "fp8", "fp8 H128 target")
            assert torch.equal(got[0], ref[0]), (B, slot)
            assert torch.equal(got[1].view(torch.int16), ref[1].view(torch.int16)), (B, slot)
            assert torch.equal(got[2].view(torch.int32), ref[2].view(torch.int32)), (B, slot)
            del c, idx, out, lse


def test_prefill_token_alone_equals_token_in_chunk_bitwise(ds):
    # "Batch-invariant prefill chunks each request independently": a query
    # token of the 4096-token chunk, run alone (a one-token prefill with the
    # same block-table row, length and top-k row), gives the same bits.
    c = workload_case("chunked_prefill", device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    del c.scores
    out, lse = ds.sparse_mla_prefill(c.q, c.kv_pages, c.kv_dtype, c.block_table, c.row_req, idx,
                                     c.lens, c.scale)
    torch.cuda.synchronize()
    tokens = [0, 1, 2047, 4095] + np.random.default_rng(3).choice(4096, 4, replace=False).tolist()
    for t in tokens:
        sl = slice(t, t + 1)
        o1, l1 = ds.sparse_mla_prefill(c.q[sl], c.kv_pages, c.kv_dtype, c.block_table,
                                       c.row_req[sl], idx[sl], c.lens[sl], c.scale)
        torch.cuda.synchronize()
        assert torch.equal(o1[0].view(torch.int16), out[t].view(torch.int16)), t
        assert torch.equal(l1[0].view(torch.int32), lse[t].view(torch.int32)), t
