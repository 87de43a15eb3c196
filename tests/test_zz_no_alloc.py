"""The allocation-free decode entry point, ds_sparse_mla_decode_noalloc.

Some callers cannot give the library device scratch memory: a memory manager
may own all of the device's memory, a CUDA graph may be mid-capture (where a
plain cudaMalloc is not allowed), or a hot loop may not afford cudaMalloc's
implicit synchronisation. For them the library keeps a built-in 32 MiB
device array and this entry point uses it instead of a caller workspace.

These tests call it through the C ABI and compare it with
ds_sparse_mla_decode (same tolerance as every other attention test), over two
calls in a row with different inputs, since the array is shared between
calls and keeps the previous call's contents. This file is named so that
pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from harness import ATOL, RTOL, ensure_built
from synthetic import decode_case, workload_case

DS_ERR_WORKSPACE = 6


@pytest.fixture(scope="module")
def ds():
    return ensure_built()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(ds, c, idx, out, lse, err):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ds.lib().ds_sparse_mla_decode_noalloc(
        _p(c.q), _p(c.kv_pages), 0 if c.kv_dtype == "bf16" else 1, c.kv_pages.shape[0],
        _p(c.block_table), c.block_table.shape[1], _p(idx), _p(c.lens), c.q.shape[0], c.H, c.k,
        c.scale, _p(out), _p(lse), _p(err), stream)


def _close(a_out, a_lse, b_out, b_lse, kv_dtype):
    a, b = a_out.float().cpu().numpy(), b_out.float().cpu().numpy()
    assert np.all(np.abs(a - b) <= ATOL[kv_dtype] + RTOL * np.abs(b))
    la, lb = a_lse.cpu().numpy(), b_lse.cpu().numpy()
    fin = np.isfinite(lb)
    assert np.array_equal(np.isfinite(la), fin)
    assert np.abs(la[fin] - lb[fin]).max(initial=0.0) <= 1e-2


@pytest.mark.gpu
def test_noalloc_matches_decode_on_two_calls_in_a_row(ds):
    cases = [workload_case("tp2_decode", device="cuda"),
             decode_case("second", [3000, 700, 5000, 0, 64], 128, 512, "fp8", seed=31,
                         device="cuda")]
    for c in cases:
        idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
        want_out, want_lse = ds.sparse_mla_decode(c.q, c.kv_pages, c.kv_dtype, c.block_table,
                                                  idx, c.lens, c.scale)
        out = torch.full_like(want_out, float("nan"))
        lse = torch.full_like(want_lse, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(ds, c, idx, out, lse, err) == 0, ds.last_error()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        _close(out, lse, want_out, want_lse, c.kv_dtype)


@pytest.mark.skipif(torch.cuda.is_available(),
                    reason="passes fake device addresses; host-validation check only")
def test_noalloc_rejects_calls_beyond_its_scratch(ds):
    # 128 rows x 128 heads at top-k 2048 need about 134 MB of scratch: refused on
    # the host, before any CUDA call, with a message that says what to use.
    L = ds.lib()
    need = L.ds_sparse_mla_workspace_size(128, 128, 2048)
    assert need > 32 << 20
    A = 0x7F0000000000
    r = L.ds_sparse_mla_decode_noalloc(A, A, 0, 16, A, 8, A, A, 128, 128, 2048, 0.04, A, A,
                                       None, None)
    assert r == DS_ERR_WORKSPACE
    msg = ds.last_error()
    assert str(need) in msg and "ds_sparse_mla_decode" in msg
