"""Multi-token decode rows (MTP): several query tokens per request.

Each request carries next_n query tokens (one target token and next_n - 1
draft tokens) that read the request's block-table row, each with its own
top-k row. Token j of a request scores seq_len - next_n + 1 + j positions: a
signed length, negative for the first tokens of a padded request (seq_len 0),
which must clamp to an empty row rather than wrap ("[Bugfix] Make DSV4 sparse
MLA work end-to-end for plain decode, MTP, and DSpark", section "What is
fixed", negative indexer context lengths under MTP). The rows go through
ds_topk_per_row and ds_sparse_mla_prefill (token -> request map).
"""

import numpy as np
import pytest
import torch

import oracle
from harness import assert_close, ensure_built, kv_np, q_bits
from synthetic import mtp_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def ds():
    return ensure_built()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_mtp_batch_matches_oracle_and_single_row_decode(ds, kv_dtype):
    # Padded requests (0), a request shorter than next_n (2), short and long ones.
    seq_lens = [0, 5000, 2, 20000, 0, 64, 9000, 700]
    next_n = 3
    c = mtp_case("mtp", seq_lens, next_n, 32, 512, kv_dtype, seed=21, device="cuda")
    idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    want_idx = oracle.topk_per_row(c.np_scores(), c.np_int("row_starts"), c.np_int("row_ends"),
                                   c.k)
    got_idx = idx.cpu().numpy()
    assert np.array_equal(got_idx, want_idx)
    padded = [r for r in range(c.R) if int(c.row_ends[r]) <= 0]
    assert padded and (got_idx[padded] == -1).all()

    out, lse = ds.sparse_mla_prefill(c.q, c.kv_pages, kv_dtype, c.block_table, c.row_req, idx,
                                     c.lens, c.scale)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.sparse_mla_prefill(q_bits(c.q), kv_np(c.kv_pages, kv_dtype), kv_dtype,
                                             c.block_table.cpu().numpy(), c.np_int("row_req"),
                                             want_idx, c.np_int("lens"), c.scale)
    assert_close(out, lse, ref, ref_lse, kv_dtype, "mtp")
    assert (out[padded] == 0).all() and torch.isneginf(lse[padded]).all()

    # Every token equals the same token run alone as a one-row plain decode
    # on its request's block-table row: bitwise.
    for r in [1, 4, 8, 11, 17, 23]:
        req = int(c.row_req[r])
        o1, l1 = ds.sparse_mla_decode(c.q[r:r + 1], c.kv_pages, kv_dtype,
                                      c.block_table[req:req + 1].contiguous(), idx[r:r + 1],
                                      c.lens[r:r + 1], c.scale)
        assert torch.equal(o1[0], out[r]), r
        assert torch.equal(l1[0], lse[r]), r
