"""GPU parity of ds_sparse_mla_decode_swa: decode over [top-k entries of the
compressed KV || sliding-window entries of the window KV] with per-head
attention sinks, against the oracle; plus the degenerate cases (no window,
sinks only, -inf sinks, rows with no valid entry) and batch invariance.
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


def _window(win_lens, W, kv_dtype, seed):
    """A window pool: row b holds its last min(W, len) positions, -1 padded."""
    w = decode_case("win", [max(1, n) for n in win_lens], 16, 64, kv_dtype, seed=seed,
                    device="cuda")
    idx = torch.full((len(win_lens), W), -1, dtype=torch.int32)
    for b, n in enumerate(win_lens):
        m = min(W, n)
        idx[b, :m] = torch.arange(n - m, n, dtype=torch.int32)
    lens = torch.tensor(win_lens, dtype=torch.int32)
    return w.kv_pages, w.block_table, idx.to(DEV), lens.to(DEV)


def _oracle(c, idx, win, sink):
    swa_pages, swa_bt, swa_idx, swa_lens = win if win is not None else (None,) * 4
    return oracle.sparse_mla_decode_swa(
        q_bits(c.q), kv_np(c.kv_pages, c.kv_dtype), c.kv_dtype, c.block_table.cpu().numpy(),
        idx.cpu().numpy(), c.lens.cpu().numpy(),
        None if win is None else kv_np(swa_pages, c.kv_dtype),
        None if win is None else swa_bt.cpu().numpy(),
        None if win is None else swa_idx.cpu().numpy(),
        None if win is None else swa_lens.cpu().numpy(),
        None if sink is None else sink.cpu().numpy(), c.scale)


def _run(ds, c, idx, win, sink):
    kw = {}
    if win is not None:
        kw = dict(swa_pages=win[0], swa_block_table=win[1], swa_idx=win[2], swa_lens=win[3])
    out, lse = ds.sparse_mla_decode_swa(c.q, c.kv_pages, c.kv_dtype, c.block_table, idx, c.lens,
                                        c.scale, attn_sink=sink, **kw)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("kv_dtype,H,k,W", [("bf16", 64, 2048, 128), ("fp8", 128, 512, 192),
                                            ("bf16", 16, 64, 512), ("bf16", 32, 640, 64)])
def test_window_and_sinks_match_oracle(ds, kv_dtype, H, k, W):
    ctx = [5000, 300, 0, 9000, 64]
    c = decode_case("swa", ctx, H, k, kv_dtype, seed=30 + H, device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    win = _window([700, 0, 40, 128, 1000], W, kv_dtype, seed=31 + H)
    g = torch.Generator().manual_seed(H)
    sink = (torch.randn(H, generator=g) * 4).to(DEV)
    sink[::5] = -float("inf")
    out, lse = _run(ds, c, idx, win, sink)
    ref, ref_lse = _oracle(c, idx, win, sink)
    assert_close(out, lse, ref, ref_lse, kv_dtype, "swa+sink")


def test_sinks_without_window_and_empty_rows(ds):
    c = decode_case("sink", [3000, 0, 700], 64, 512, "bf16", seed=40, device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    sink = torch.linspace(-3, 3, 64).to(DEV)
    out, lse = _run(ds, c, idx, None, sink)
    ref, ref_lse = _oracle(c, idx, None, sink)
    assert_close(out, lse, ref, ref_lse, "bf16", "sink only")
    # Row 1 has no entry: out = 0 and lse = the sink itself.
    assert (out[1] == 0).all()
    assert torch.allclose(lse[1], sink, atol=1e-5, rtol=0)


def test_no_window_and_no_sinks_is_plain_decode_bitwise(ds):
    c = decode_case("plain", [4000, 2500], 64, 2048, "bf16", seed=41, device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    o1, l1 = ds.sparse_mla_decode(c.q, c.kv_pages, "bf16", c.block_table, idx, c.lens, c.scale)
    o2, l2 = _run(ds, c, idx, None, None)
    o3, l3 = _run(ds, c, idx, None, torch.full((64,), -float("inf"), device=DEV))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_row_result_is_batch_invariant(ds):
    ctx = [6000, 200, 12000, 5]
    c = decode_case("inv", ctx, 64, 1024, "bf16", seed=42, device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    win = _window([900, 30, 1500, 3], 128, "bf16", seed=43)
    sink = torch.randn(64, generator=torch.Generator().manual_seed(44)).to(DEV)
    out, lse = _run(ds, c, idx, win, sink)
    for r in range(len(ctx)):
        sub = decode_case("inv", ctx, 64, 1024, "bf16", seed=42, device="cuda")
        sub.q, sub.lens = c.q[r:r + 1], c.lens[r:r + 1]
        sub.block_table = c.block_table[r:r + 1].contiguous()
        w1 = (win[0], win[1][r:r + 1].contiguous(), win[2][r:r + 1].contiguous(), win[3][r:r + 1])
        o1, l1 = _run(ds, sub, idx[r:r + 1], w1, sink)
        assert torch.equal(o1[0], out[r]) and torch.equal(l1[0], lse[r]), r
