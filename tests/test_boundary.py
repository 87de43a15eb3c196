"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before launching anything.

Host validation follows the pages' contract: unsupported shapes are a hard
error ("Batch-invariant kernels for 0-diff RL", PR 54955), checked before the
kernel launch ("Preallocate DeepSeek V4 padded-query output", PR 671,
"Operation contract"), with a message naming the parameter that missed and
what is available ("Make DSV4 sparse MLA work end-to-end", PR 51538,
"SM120 gate"). None of these calls reaches the CUDA runtime.
"""

import ctypes
import os
import re

import pytest

from harness import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds_sparse_mla.h")

DS_OK, DS_ERR_NULL, DS_ERR_SHAPE, DS_ERR_UNSUPPORTED, DS_ERR_DTYPE, DS_ERR_ALIGN, \
    DS_ERR_WORKSPACE, DS_ERR_CUDA = range(8)

# Fake, never-dereferenced device addresses: validation must fail before use.
A = 0x7F0000000000


def _cuda_visible():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


# The tests that pass fake device addresses run only where no CUDA device is
# visible: if a host check ever regressed there, the call would fail in the
# runtime instead of launching a kernel on addresses that are not mapped.
host_only = pytest.mark.skipif(_cuda_visible(),
                               reason="passes fake device addresses; host-validation check only")


@pytest.fixture(scope="module")
def ds():
    return ensure_built()


@pytest.fixture(scope="module")
def L(ds):
    return ds.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("ds_topk_per_row", "ds_sparse_mla_decode", "ds_sparse_mla_prefill",
                 "ds_last_error", "ds_supported_config"):
        assert want in names


def test_library_exports_every_declared_symbol(ds, L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(ds.EXPORTED) <= set(declared_functions())


def _err(L):
    return L.ds_last_error().decode()


def test_supported_config_matrix(L):
    for h in (16, 32, 64, 128):
        for k in (64, 128, 512, 2048):
            for kvd in (0, 1):
                assert L.ds_supported_config(h, k, 64, 576, 512, kvd) == 1
    cases = [((48, 2048, 64, 576, 512, 0), "num_heads"),
             ((64, 100, 64, 576, 512, 0), "topk"),
             ((64, 4096, 64, 576, 512, 0), "topk"),
             ((64, 0, 64, 576, 512, 0), "topk"),
             ((64, 2048, 128, 576, 512, 0), "page_block_size"),
             ((64, 2048, 64, 512, 512, 0), "d_qk"),
             ((64, 2048, 64, 576, 576, 0), "d_v"),
             ((64, 2048, 64, 576, 512, 7), "kv_dtype")]
    for args, name in cases:
        assert L.ds_supported_config(*args) == 0
        msg = _err(L)
        assert name in msg and "available" in msg, msg


def test_workspace_sizes(L):
    # splits = ceil(k / 512); per split: R*H*512 bf16 partial O plus R*H floats
    # each of m and l, 256-aligned.
    def want(R, H, k):
        n = -(-k // 512) * R * H
        ml = (n * 4 + 255) // 256 * 256
        return n * 512 * 2 + 2 * ml   # bf16 partial O, fp32 m and l
    for R, H, k in [(1, 16, 64), (32, 64, 2048), (128, 128, 2048), (4096, 128, 2048), (3, 32, 576)]:
        if k % 64:
            assert L.ds_sparse_mla_workspace_size(R, H, k) == 0
        else:
            assert L.ds_sparse_mla_workspace_size(R, H, k) == want(R, H, k)
    assert L.ds_sparse_mla_workspace_size(4, 48, 2048) == 0
    assert L.ds_topk_workspace_size(100, 1000, 10) == 0


def test_topk_workspace_sizes(L):
    # The grid top-k's workspace: a 256-byte header (zeroed before each
    # launch), an entry count and a key bound per 8192-score segment, then
    # one 8192-entry (key, position) slot per segment; a row has at most
    # ceil((stride + 255) / 8192) segments. Shapes taken by the other kernels
    # need none.
    def al(b):
        return (b + 255) // 256 * 256

    def want(R, stride):
        ns = (stride + 255 + 8191) // 8192
        return 256 + 2 * al(R * ns * 4) + R * ns * 8192 * 8
    for R, stride in [(128, 131072), (8, 100000), (1, 16384), (15, 32768), (255, 65536),
                      (16, 70000), (1, 8192)]:
        assert L.ds_topk_workspace_size(R, stride, 2048) == want(R, stride), (R, stride)
    # whole rows in shared memory, the streaming grid, rows wider than 128K,
    # more than 2^24 or fewer than 8192 scores, and invalid shapes: none
    for R, stride in [(16, 32768), (1024, 16384), (256, 40000), (8, 131073), (200, 90000),
                      (3, 7), (1, 8191), (0, 1000), (-1, 1000), (4, 0)]:
        assert L.ds_topk_workspace_size(R, stride, 2048) == 0, (R, stride)


def _topk(L, scores=A, stride=1024, rows=4, starts=A, ends=A, k=16, out=A):
    return L.ds_topk_per_row(scores, stride, rows, starts, ends, k, out, None, 0, None)


@host_only
def test_topk_rejects_misaligned_workspace(L):
    rc = L.ds_topk_per_row(A, 1024, 4, A, A, 16, A, ctypes.c_void_p(0x10010), 1 << 20, None)
    assert rc == DS_ERR_ALIGN and "workspace" in _err(L)


@host_only
def test_topk_rejects_bad_arguments(L):
    assert _topk(L, k=0) == DS_ERR_UNSUPPORTED and "k=0" in _err(L)
    assert _topk(L, k=20000) == DS_ERR_UNSUPPORTED
    assert _topk(L, stride=0) == DS_ERR_UNSUPPORTED and "row_stride" in _err(L)
    assert _topk(L, rows=-1) == DS_ERR_SHAPE
    assert _topk(L, scores=None) == DS_ERR_NULL and "scores" in _err(L)
    assert _topk(L, starts=None) == DS_ERR_NULL and "row_starts" in _err(L)
    assert _topk(L, out=None) == DS_ERR_NULL and "idx_out" in _err(L)
    assert _topk(L, scores=A + 2) == DS_ERR_ALIGN
    # Zero rows is a valid empty call: nothing is launched.
    assert _topk(L, rows=0, scores=None, starts=None, ends=None, out=None) == DS_OK


def _decode(L, **kw):
    a = dict(q=A, kv=A, kvd=0, pages=16, bt=A, bts=8, idx=A, lens=A, R=4, H=64, k=2048,
             scale=0.04, out=A, lse=A, ws=A, wsb=1 << 40, err=None)
    a.update(kw)
    return L.ds_sparse_mla_decode(a["q"], a["kv"], a["kvd"], a["pages"], a["bt"], a["bts"],
                                  a["idx"], a["lens"], a["R"], a["H"], a["k"], a["scale"], a["out"],
                                  a["lse"], a["ws"], a["wsb"], a["err"], None)


@host_only
def test_decode_rejects_bad_arguments(L):
    assert _decode(L, H=48) == DS_ERR_UNSUPPORTED and "num_heads=48" in _err(L)
    assert _decode(L, k=100) == DS_ERR_UNSUPPORTED and "topk=100" in _err(L)
    assert _decode(L, kvd=5) == DS_ERR_DTYPE and "kv_dtype" in _err(L)
    assert _decode(L, R=-2) == DS_ERR_SHAPE
    assert _decode(L, pages=0) == DS_ERR_SHAPE and "num_pages" in _err(L)
    assert _decode(L, bts=0) == DS_ERR_SHAPE and "bt_stride" in _err(L)
    assert _decode(L, scale=float("nan")) == DS_ERR_SHAPE and "scale" in _err(L)
    for name in ("q", "kv", "bt", "idx", "lens", "out", "lse", "ws"):
        assert _decode(L, **{name: None}) == DS_ERR_NULL, name
    assert _decode(L, q=A + 8) == DS_ERR_ALIGN and "q must be 16-byte" in _err(L)
    assert _decode(L, kv=A + 4) == DS_ERR_ALIGN and "kv_pages" in _err(L)
    assert _decode(L, ws=A + 16) == DS_ERR_ALIGN and "workspace" in _err(L)
    assert _decode(L, err=A + 2) == DS_ERR_ALIGN and "err_flag" in _err(L)
    need = L.ds_sparse_mla_workspace_size(4, 64, 2048)
    assert _decode(L, wsb=need - 1) == DS_ERR_WORKSPACE and str(need) in _err(L)
    assert _decode(L, R=0, q=None, kv=None, out=None) in (DS_OK, DS_ERR_NULL)


@host_only
def test_prefill_requires_row_req(L):
    r = L.ds_sparse_mla_prefill(A, A, 0, 16, A, 8, 1, None, A, A, 4, 64, 2048, 0.04, A, A, A,
                                1 << 40, None, None)
    assert r == DS_ERR_NULL and "row_req" in _err(L)
    r = L.ds_sparse_mla_prefill(A, A, 0, 16, A, 8, 0, A, A, A, 4, 64, 2048, 0.04, A, A, A,
                                1 << 40, None, None)
    assert r == DS_ERR_SHAPE and "num_requests" in _err(L)


def test_last_error_clears_on_success(L):
    assert L.ds_supported_config(7, 64, 64, 576, 512, 0) == 0
    assert _err(L) != ""
    assert L.ds_supported_config(64, 64, 64, 576, 512, 0) == 1
    assert _err(L) == ""


def test_python_binding_fails_loudly_without_cuda_tensors(ds):
    import torch
    with pytest.raises(ValueError):
        ds.topk_per_row(torch.zeros(2, 8), torch.zeros(2, dtype=torch.int32),
                        torch.zeros(2, dtype=torch.int32), 4)
    with pytest.raises(TypeError):
        ds.topk_per_row(torch.zeros(2, 8, dtype=torch.float64), torch.zeros(2, dtype=torch.int32),
                        torch.zeros(2, dtype=torch.int32), 4)


def _write(L, latent=A, n=4, slots=A, kvd=1, pool=A, pages=16, err=None):
    return L.ds_kv_cache_write(latent, n, slots, kvd, pool, pages, err, None)


@host_only
def test_kv_cache_write_rejects_bad_arguments(L):
    assert _write(L, kvd=3) == DS_ERR_DTYPE and "kv_dtype" in _err(L)
    assert _write(L, n=-1) == DS_ERR_SHAPE and "num_rows" in _err(L)
    assert _write(L, pages=0) == DS_ERR_SHAPE and "num_pages" in _err(L)
    assert _write(L, latent=None) == DS_ERR_NULL and "latent" in _err(L)
    assert _write(L, slots=None) == DS_ERR_NULL and "slots" in _err(L)
    assert _write(L, pool=None) == DS_ERR_NULL and "kv_pages" in _err(L)
    assert _write(L, latent=A + 8) == DS_ERR_ALIGN and "latent" in _err(L)
    assert _write(L, slots=A + 4) == DS_ERR_ALIGN and "slots" in _err(L)
    # Zero rows is a valid empty call: nothing is launched.
    assert _write(L, n=0, latent=None, slots=None) == DS_OK


def _swa(L, width=128, swa_pages=A, swa_np=8, swa_bt=A, swa_bts=2, swa_idx=A, swa_lens=A,
         sink=None, wsb=1 << 40, R=4):
    return L.ds_sparse_mla_decode_swa(A, A, 0, 16, A, 8, A, A, 2048, swa_pages, swa_np, swa_bt,
                                      swa_bts, swa_idx, swa_lens, width, sink, R, 64, 0.04, A, A,
                                      A, wsb, None, None)


@host_only
def test_decode_swa_rejects_bad_window_arguments(L):
    # "Make DSV4 sparse MLA work end-to-end", "What is fixed": the window
    # index list is padded to a multiple of 64 entries.
    for width in (32, 100, 576, -64):
        assert _swa(L, width=width) == DS_ERR_UNSUPPORTED and "swa_width" in _err(L), width
    assert _swa(L, swa_np=0) == DS_ERR_SHAPE and "swa_num_pages" in _err(L)
    assert _swa(L, swa_bts=0) == DS_ERR_SHAPE and "swa_bt_stride" in _err(L)
    for name in ("swa_pages", "swa_bt", "swa_idx", "swa_lens"):
        assert _swa(L, **{name: None}) == DS_ERR_NULL, name
    assert _swa(L, swa_pages=A + 8) == DS_ERR_ALIGN and "swa_pages" in _err(L)
    assert _swa(L, sink=A + 2) == DS_ERR_ALIGN and "attn_sink" in _err(L)
    need = L.ds_sparse_mla_swa_workspace_size(4, 64, 2048, 128)
    # Splits: max(ceil(k / 512), ceil((k + W) / 768)); a window adds one only
    # when the second term wins (k 512 + W 512: 2 splits instead of 1).
    assert need == L.ds_sparse_mla_workspace_size(4, 64, 2048)
    assert (L.ds_sparse_mla_swa_workspace_size(4, 64, 512, 512) ==
            2 * L.ds_sparse_mla_workspace_size(4, 64, 512))
    assert _swa(L, wsb=need - 1) == DS_ERR_WORKSPACE and str(need) in _err(L)
    assert L.ds_sparse_mla_swa_workspace_size(4, 64, 2048, 100) == 0
    # No window: the window arguments may be NULL.
    assert _swa(L, width=0, swa_pages=None, swa_bt=None, swa_idx=None, swa_lens=None,
                wsb=1) == DS_ERR_WORKSPACE


def test_split_geometry_fits_the_kernels(L):
    # The split count is a function of k and the window width alone:
    # S = max(ceil(k / 512), ceil((k + W) / 768)). The split kernel holds at
    # most 12 tiles of 64 entries per split and the combine merges at most 4
    # splits, so every supported (k, W) must satisfy both. S is read back from
    # the workspace size (S x R x H x 512 bf16 partial values, then the fp32
    # m and l arrays, each padded to 256 bytes).
    R, H = 1, 64
    for k in range(64, 2049, 64):
        for W in [0] + list(range(64, 513, 64)):
            ws = L.ds_sparse_mla_swa_workspace_size(R, H, k, W)
            S = -(-k // 512)
            S = max(S, -(-(k + W) // 768))
            ml = -(-(S * R * H * 4) // 256) * 256
            assert ws == S * R * H * 512 * 2 + 2 * ml, (k, W)
            T = (k + W) // 64
            assert S <= 4 and -(-T // S) <= 12, (k, W, S, T)


def _ix(L, q=A, w=A, k=A, pages=16, bt=A, bts=8, nreq=4, row_req=None, lens=A, R=4, H=64, D=128,
        logits=A, ls=512, err=None):
    return L.ds_indexer_logits(q, w, k, pages, bt, bts, nreq, row_req, lens, R, H, D, logits, ls,
                               err, None)


@host_only
def test_indexer_rejects_bad_arguments(L):
    assert _ix(L, H=48) == DS_ERR_UNSUPPORTED and "num_heads=48" in _err(L)
    assert _ix(L, D=64) == DS_ERR_UNSUPPORTED and "head_dim=64" in _err(L)
    assert _ix(L, R=-1) == DS_ERR_SHAPE
    assert _ix(L, pages=0) == DS_ERR_SHAPE and "num_pages" in _err(L)
    assert _ix(L, bts=0) == DS_ERR_SHAPE and "bt_stride" in _err(L)
    assert _ix(L, nreq=0) == DS_ERR_SHAPE and "num_requests" in _err(L)
    # A row can score up to 64 * bt_stride positions: the output row must hold them.
    assert _ix(L, ls=511) == DS_ERR_SHAPE and "logits_stride" in _err(L)
    for name in ("q", "w", "k", "bt", "lens", "logits"):
        assert _ix(L, **{name: None}) == DS_ERR_NULL, name
    assert _ix(L, q=A + 8) == DS_ERR_ALIGN and "q must be 16-byte" in _err(L)
    assert _ix(L, k=A + 4) == DS_ERR_ALIGN and "k_pages" in _err(L)
    assert _ix(L, row_req=A + 2) == DS_ERR_ALIGN and "row_req" in _err(L)
    # Zero rows is a valid empty call: nothing is launched.
    assert _ix(L, R=0, q=None, w=None, k=None) in (DS_OK, DS_ERR_NULL)
