"""GPU parity of ds_indexer_logits (the indexer's MQA logits) against the oracle.

Scores: I[r, s] = sum_j w_j max(0, q_j . k_s) (the DeepSeek-V3.2-Exp lightning
indexer; the pages name the logits without a formula). The GPU forms each dot
product from exact bf16 products with fp32 accumulation over 128 dims, then
sums the 64 heads with fp32 fused multiply-adds, so its error is bounded by
about 128 + 64 + 2 float32 roundings (2^-24 each) of the magnitude
M = sum_j |w_j| sum_i |q_ji| |k_si|, i.e. about 2^-16 M; the test allows
2^-16 M (M comes from the oracle itself, evaluated on |q|, |k|, |w|, where
the clamp does nothing). Measured: about 2e-8 M.

The top-k that follows is checked bit for bit on the same logits (GPU top-k of
the GPU logits against the oracle top-k of those logits), since floating point
decides which scores win a near tie.
"""

import numpy as np
import pytest
import torch

import oracle
from harness import ensure_built
from synthetic import indexer_case, indexer_workload

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
REL_BOUND = 2.0 ** -16


@pytest.fixture(scope="module")
def ds():
    return ensure_built()


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _oracle(c, rows=None, row_req=None, width=None, absolute=False):
    rows = list(range(c.q.shape[0])) if rows is None else list(rows)
    q = c.q[rows].float()
    k = c.k_pages.float()
    w = c.w[rows]
    if absolute:
        q, k, w = q.abs(), k.abs(), w.abs()
    qb = _bits(q.to(torch.bfloat16))
    kb = _bits(k.to(torch.bfloat16))
    # A sampled row keeps its own block-table row.
    rr = np.asarray(rows) if row_req is None else row_req.cpu().numpy()[rows]
    lens = c.lens.cpu().numpy()[rows]
    return oracle.indexer_logits(qb, w.cpu().numpy(), kb, c.block_table.cpu().numpy(), lens,
                                 row_req=rr, width=width)


def _check(got, ref, mag, what):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got) & ~fin, np.isneginf(ref) & ~fin), f"{what}: -inf differ"
    err = np.abs(got[fin] - ref[fin])
    bound = REL_BOUND * mag[fin] + 1e-30
    assert np.all(err <= bound), (f"{what}: max err {err.max():.3g}, worst ratio "
                                  f"{(err / bound).max():.3g}")
    print(f"[parity] {what}: max abs err {err.max() if err.size else 0:.3g}, max err / magnitude "
          f"{(err / np.maximum(mag[fin], 1e-30)).max() if err.size else 0:.3g} "
          f"(bound {REL_BOUND:.3g})")


@pytest.mark.parametrize("heads", [16, 32, 64])
def test_small_parity(ds, heads):
    ctx = [4100, 2048 + 5, 200, 65, 64, 63, 1, 0]
    c = indexer_case(f"ix{heads}", ctx, heads=heads, seed=heads, device="cuda")
    got = ds.indexer_logits(c.q, c.w, c.k_pages, c.block_table, c.lens)
    torch.cuda.synchronize()
    width = got.shape[1]
    ref = _oracle(c, width=width)
    mag = _oracle(c, width=width, absolute=True)
    g = got.cpu().numpy().astype(np.float64)
    for r, L in enumerate(ctx):
        _check(g[r, :L], ref[r, :L], mag[r, :L], f"H={heads} row {r} (L={L})")


def test_topk_of_indexer_logits_is_exact(ds):
    ctx = [4100, 3000, 2048, 700]
    c = indexer_case("ixk", ctx, heads=64, seed=3, device="cuda")
    logits = ds.indexer_logits(c.q, c.w, c.k_pages, c.block_table, c.lens)
    starts = torch.zeros_like(c.lens)
    idx = ds.topk_per_row(logits, starts, c.lens, 2048)
    torch.cuda.synchronize()
    want = oracle.topk_per_row(logits.cpu().numpy(), starts.cpu().numpy(), c.lens.cpu().numpy(),
                               2048)
    assert np.array_equal(idx.cpu().numpy(), want)


def test_bad_pages_row_req_and_lengths(ds):
    ctx = [300, 300, 300, 300]
    c = indexer_case("ixbad", ctx, heads=32, seed=4, device="cuda")
    c.block_table[1, 2] = 10 ** 6          # positions 128..191 of row 1: outside the pool
    row_req = torch.tensor([0, 1, 7, 1], dtype=torch.int32, device=DEV)   # 7: no such request
    c.lens = torch.tensor([300, 300, 300, -4], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    logits = torch.full((4, 64 * c.block_table.shape[1]), 7.0, device=DEV)
    ds.indexer_logits(c.q, c.w, c.k_pages, c.block_table, c.lens, row_req=row_req, logits=logits,
                      err_flag=err)
    torch.cuda.synchronize()
    flags = int(err.item())
    assert flags & ds.DEVERR_PAGE and flags & ds.DEVERR_ROWREQ and not flags & ds.DEVERR_TIMEOUT
    g = logits.cpu().numpy()
    assert np.all(np.isneginf(g[1, 128:192]))
    assert np.all(g[2] == 7.0) and np.all(g[3] == 7.0)   # nothing written
    assert np.all(g[0, 300:] == 7.0) and np.all(g[1, 300:] == 7.0)
    ref = _oracle(c, rows=[0, 1], row_req=row_req, width=g.shape[1])
    mag = _oracle(c, rows=[0, 1], row_req=row_req, width=g.shape[1], absolute=True)
    for i in (0, 1):
        _check(g[i, :300].astype(np.float64), ref[i, :300], mag[i, :300], f"row {i}")


def test_batch_invariance_bitwise(ds):
    c = indexer_case("ixinv", [5000, 1200, 9000, 64, 3333], heads=64, seed=5, device="cuda")
    full = ds.indexer_logits(c.q, c.w, c.k_pages, c.block_table, c.lens)
    torch.cuda.synchronize()
    for r in range(5):
        one = ds.indexer_logits(c.q[r:r + 1].contiguous(), c.w[r:r + 1].contiguous(), c.k_pages,
                                c.block_table[r:r + 1].contiguous(), c.lens[r:r + 1].contiguous())
        torch.cuda.synchronize()
        L = int(c.lens[r])
        assert torch.equal(one[0, :L].view(torch.int32), full[r, :L].view(torch.int32)), r


def test_tp2_indexer_workload_sampled(ds):
    c = indexer_workload("tp2_indexer", device="cuda")
    logits = ds.indexer_logits(c.q, c.w, c.k_pages, c.block_table, c.lens)
    idx = ds.topk_per_row(logits, torch.zeros_like(c.lens), c.lens, 2048)
    torch.cuda.synchronize()
    rows = [0, int(torch.argmax(c.lens)), 31]
    ref = _oracle(c, rows=rows, width=logits.shape[1])
    mag = _oracle(c, rows=rows, width=logits.shape[1], absolute=True)
    g = logits.cpu().numpy().astype(np.float64)
    for i, r in enumerate(rows):
        L = int(c.lens[r])
        _check(g[r, :L], ref[i, :L], mag[i, :L], f"tp2_indexer row {r}")
    want = oracle.topk_per_row(logits.cpu().numpy()[rows], np.zeros(3, np.int32),
                               c.lens.cpu().numpy()[rows], 2048)
    assert np.array_equal(idx.cpu().numpy()[rows], want)
