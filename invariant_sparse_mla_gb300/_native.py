"""ctypes binding of libds_sparse_mla.so (argument marshalling only).

Every function here checks torch dtypes, devices and contiguity, then calls
the C ABI of include/ds_sparse_mla.h with raw device pointers and the current
CUDA stream. No computation happens in Python, and there is no fallback: if
the library is missing or a call fails, an exception is raised.
"""

import ctypes
import os
import threading

import torch

from . import build as _build

DS_OK = 0
KV_DTYPES = {"bf16": 0, "fp8": 1, 0: 0, 1: 1}
DEVERR_IDX, DEVERR_PAGE, DEVERR_ROWREQ, DEVERR_TIMEOUT = 1, 2, 4, 8

_lib = None
_lock = threading.Lock()

c_i32p = ctypes.c_void_p


class DSError(RuntimeError):
    """A ds_* call returned an error status (the message names the parameter)."""

    def __init__(self, status, message):
        super().__init__(f"status {status}: {message}")
        self.status = status


def lib():
    """The loaded library (built beforehand by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -m invariant_sparse_mla_gb300.build); there is no fallback")
        L = ctypes.CDLL(path)
        i64, i32, vp, f32, sz = (ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                 ctypes.c_float, ctypes.c_size_t)
        L.ds_last_error.restype = ctypes.c_char_p
        L.ds_last_error.argtypes = []
        L.ds_supported_config.restype = i32
        L.ds_supported_config.argtypes = [i32] * 6
        L.ds_topk_workspace_size.restype = sz
        L.ds_topk_workspace_size.argtypes = [i64, i64, i32]
        L.ds_sparse_mla_workspace_size.restype = sz
        L.ds_sparse_mla_workspace_size.argtypes = [i64, i32, i32]
        L.ds_topk_per_row.restype = i32
        L.ds_topk_per_row.argtypes = [vp, i64, i64, vp, vp, i32, vp, vp, sz, vp]
        L.ds_sparse_mla_decode.restype = i32
        L.ds_sparse_mla_decode.argtypes = [vp, vp, i32, i64, vp, i64, vp, vp, i64, i32, i32, f32,
                                           vp, vp, vp, sz, vp, vp]
        L.ds_sparse_mla_prefill.restype = i32
        L.ds_sparse_mla_prefill.argtypes = [vp, vp, i32, i64, vp, i64, i64, vp, vp, vp, i64, i32,
                                            i32, f32, vp, vp, vp, sz, vp, vp]
        L.ds_sparse_mla_decode_noalloc.restype = i32
        L.ds_sparse_mla_decode_noalloc.argtypes = [vp, vp, i32, i64, vp, i64, vp, vp, i64, i32,
                                                   i32, f32, vp, vp, vp, vp]
        L.ds_sparse_mla_decode_swa.restype = i32
        L.ds_sparse_mla_decode_swa.argtypes = [vp, vp, i32, i64, vp, i64, vp, vp, i32, vp, i64,
                                               vp, i64, vp, vp, i32, vp, i64, i32, f32, vp, vp,
                                               vp, sz, vp, vp]
        L.ds_sparse_mla_swa_workspace_size.restype = sz
        L.ds_sparse_mla_swa_workspace_size.argtypes = [i64, i32, i32, i32]
        L.ds_kv_cache_write.restype = i32
        L.ds_kv_cache_write.argtypes = [vp, i64, vp, i32, vp, i64, vp, vp]
        L.ds_indexer_logits.restype = i32
        L.ds_indexer_logits.argtypes = [vp, vp, vp, i64, vp, i64, i64, vp, vp, i64, i32, i32, vp,
                                        i64, vp, vp]
        _lib = L
        return _lib


EXPORTED = ("ds_last_error", "ds_supported_config", "ds_topk_workspace_size",
            "ds_sparse_mla_workspace_size", "ds_topk_per_row", "ds_sparse_mla_decode",
            "ds_sparse_mla_prefill", "ds_sparse_mla_decode_noalloc", "ds_kv_cache_write",
            "ds_sparse_mla_decode_swa", "ds_sparse_mla_swa_workspace_size", "ds_indexer_logits")


def last_error():
    return lib().ds_last_error().decode()


def _check(status):
    if status != DS_OK:
        raise DSError(status, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, device=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def supported_config(num_heads, topk, page_block_size=64, d_qk=576, d_v=512, kv_dtype="bf16"):
    """(True, "") or (False, message naming the first parameter that missed)."""
    r = lib().ds_supported_config(num_heads, topk, page_block_size, d_qk, d_v,
                                  KV_DTYPES.get(kv_dtype, -1))
    return bool(r), ("" if r else last_error())


def attention_workspace_size(num_rows, num_heads, k):
    return int(lib().ds_sparse_mla_workspace_size(num_rows, num_heads, k))


def topk_workspace_size(num_rows, row_stride, k):
    return int(lib().ds_topk_workspace_size(num_rows, row_stride, k))


def topk_per_row(scores, row_starts, row_ends, k, idx_out=None, stream=None, workspace=None):
    """Deterministic top-k of every row; returns int32 [num_rows, k].

    ``workspace``: None allocates the bytes ``topk_workspace_size`` asks for
    (none for most shapes); a uint8 CUDA tensor is used as given; False runs
    without one. The output is the same either way: the workspace only lets
    the grid kernel run for the shapes that have it.
    """
    _need(scores, "scores", torch.float32, ndim=2)
    dev = scores.device
    _need(row_starts, "row_starts", torch.int32, dev, 1)
    _need(row_ends, "row_ends", torch.int32, dev, 1)
    R, stride = scores.shape
    if row_starts.numel() != R or row_ends.numel() != R:
        raise ValueError("row_starts / row_ends must have num_rows entries")
    if idx_out is None:
        idx_out = torch.empty((R, k), dtype=torch.int32, device=dev)
    _need(idx_out, "idx_out", torch.int32, dev, 2)
    if tuple(idx_out.shape) != (R, k):
        raise ValueError(f"idx_out must be [{R}, {k}]")
    if workspace is None:
        need = topk_workspace_size(R, stride, k) if R > 0 else 0
        workspace = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else False
    if workspace is False:
        ws_ptr, ws_bytes = None, 0
    else:
        _need(workspace, "workspace", torch.uint8, dev)
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel()
    _check(lib().ds_topk_per_row(_ptr(scores), stride, R, _ptr(row_starts), _ptr(row_ends), k,
                                 _ptr(idx_out), ws_ptr, ws_bytes, _stream(stream, dev)))
    return idx_out


def _attention_args(q, kv_pages, kv_dtype, block_table, idx, lens, out, lse, workspace, err_flag):
    _need(q, "q", torch.bfloat16, ndim=3)
    dev = q.device
    R, H, D = q.shape
    if D != 576:
        raise ValueError("q must be [rows, heads, 576]")
    kvd = KV_DTYPES.get(kv_dtype)
    if kvd is None:
        raise ValueError(f"kv_dtype must be 'bf16' or 'fp8', got {kv_dtype!r}")
    if kvd == 0:
        _need(kv_pages, "kv_pages", torch.bfloat16, dev, 3)
        if tuple(kv_pages.shape[1:]) != (64, 576):
            raise ValueError("bf16 kv_pages must be [num_pages, 64, 576]")
    else:
        _need(kv_pages, "kv_pages", torch.uint8, dev, 3)
        if tuple(kv_pages.shape[1:]) != (64, 656):
            raise ValueError("fp8 kv_pages must be [num_pages, 64, 656] bytes")
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(idx, "idx", torch.int32, dev, 2)
    _need(lens, "lens", torch.int32, dev, 1)
    k = idx.shape[1]
    if idx.shape[0] != R or lens.numel() != R:
        raise ValueError("idx and lens must have one row per query row")
    if out is None:
        out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev, 3)
    _need(lse, "lse", torch.float32, dev, 2)
    if tuple(out.shape) != (R, H, 512) or tuple(lse.shape) != (R, H):
        raise ValueError("out must be [rows, heads, 512] and lse [rows, heads]")
    need = attention_workspace_size(R, H, k) if R > 0 else 0
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, dev)
    return dev, R, H, k, kvd, out, lse, workspace


def sparse_mla_decode(q, kv_pages, kv_dtype, block_table, idx, lens, scale, out=None, lse=None,
                      workspace=None, err_flag=None, stream=None):
    """Sparse MLA decode; returns (out bf16 [R, H, 512], lse fp32 [R, H])."""
    dev, R, H, k, kvd, out, lse, workspace = _attention_args(
        q, kv_pages, kv_dtype, block_table, idx, lens, out, lse, workspace, err_flag)
    _check(lib().ds_sparse_mla_decode(
        _ptr(q), _ptr(kv_pages), kvd, kv_pages.shape[0], _ptr(block_table), block_table.shape[1],
        _ptr(idx), _ptr(lens), R, H, k, float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel(), _ptr(err_flag), _stream(stream, dev)))
    return out, lse


def sparse_mla_prefill(q, kv_pages, kv_dtype, block_table, row_req, idx, lens, scale, out=None,
                       lse=None, workspace=None, err_flag=None, stream=None):
    """Sparse MLA prefill (one query row per token); returns (out, lse)."""
    dev, R, H, k, kvd, out, lse, workspace = _attention_args(
        q, kv_pages, kv_dtype, block_table, idx, lens, out, lse, workspace, err_flag)
    _need(row_req, "row_req", torch.int32, dev, 1)
    if row_req.numel() != R:
        raise ValueError("row_req must have one entry per token")
    _check(lib().ds_sparse_mla_prefill(
        _ptr(q), _ptr(kv_pages), kvd, kv_pages.shape[0], _ptr(block_table), block_table.shape[1],
        block_table.shape[0], _ptr(row_req), _ptr(idx), _ptr(lens), R, H, k, float(scale),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(err_flag),
        _stream(stream, dev)))
    return out, lse


def kv_cache_write(latent, slots, kv_pages, kv_dtype, err_flag=None, stream=None):
    """Write new latent rows (bf16 [N, 576]) into the paged pool at ``slots``
    (int64 [N], page * 64 + offset; negative = padding); FP8 pools get the
    quantised layout. Returns ``kv_pages``."""
    _need(latent, "latent", torch.bfloat16, ndim=2)
    dev = latent.device
    if latent.shape[1] != 576:
        raise ValueError("latent must be [rows, 576]")
    _need(slots, "slots", torch.int64, dev, 1)
    if slots.numel() != latent.shape[0]:
        raise ValueError("slots must have one entry per latent row")
    kvd = KV_DTYPES.get(kv_dtype)
    if kvd is None:
        raise ValueError(f"kv_dtype must be 'bf16' or 'fp8', got {kv_dtype!r}")
    if kvd == 0:
        _need(kv_pages, "kv_pages", torch.bfloat16, dev, 3)
        if tuple(kv_pages.shape[1:]) != (64, 576):
            raise ValueError("bf16 kv_pages must be [num_pages, 64, 576]")
    else:
        _need(kv_pages, "kv_pages", torch.uint8, dev, 3)
        if tuple(kv_pages.shape[1:]) != (64, 656):
            raise ValueError("fp8 kv_pages must be [num_pages, 64, 656] bytes")
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, dev)
    _check(lib().ds_kv_cache_write(_ptr(latent), latent.shape[0], _ptr(slots), kvd,
                                   _ptr(kv_pages), kv_pages.shape[0], _ptr(err_flag),
                                   _stream(stream, dev)))
    return kv_pages


def swa_workspace_size(num_rows, num_heads, k, swa_width):
    return int(lib().ds_sparse_mla_swa_workspace_size(num_rows, num_heads, k, swa_width))


def sparse_mla_decode_swa(q, kv_pages, kv_dtype, block_table, idx, lens, scale, swa_pages=None,
                          swa_block_table=None, swa_idx=None, swa_lens=None, attn_sink=None,
                          out=None, lse=None, workspace=None, err_flag=None, stream=None):
    """Decode over [top-k entries || sliding-window entries] with optional
    per-head sinks (float32 [H], natural log); returns (out, lse)."""
    dev, R, H, k, kvd, out, lse, _ = _attention_args(
        q, kv_pages, kv_dtype, block_table, idx, lens, out, lse, torch.empty(0, dtype=torch.uint8,
                                                                             device=q.device),
        err_flag)
    W = 0
    if swa_idx is not None:
        W = swa_idx.shape[1]
        _need(swa_idx, "swa_idx", torch.int32, dev, 2)
        _need(swa_lens, "swa_lens", torch.int32, dev, 1)
        _need(swa_block_table, "swa_block_table", torch.int32, dev, 2)
        _need(swa_pages, "swa_pages", kv_pages.dtype, dev, 3)
        if tuple(swa_pages.shape[1:]) != tuple(kv_pages.shape[1:]):
            raise ValueError("swa_pages must have the row format of kv_pages")
        if swa_idx.shape[0] != R or swa_lens.numel() != R or swa_block_table.shape[0] != R:
            raise ValueError("the window arguments must have one row per query row")
    if attn_sink is not None:
        _need(attn_sink, "attn_sink", torch.float32, dev, 1)
        if attn_sink.numel() != H:
            raise ValueError("attn_sink must have num_heads entries")
    need = swa_workspace_size(R, H, k, W) if R > 0 else 0
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    _check(lib().ds_sparse_mla_decode_swa(
        _ptr(q), _ptr(kv_pages), kvd, kv_pages.shape[0], _ptr(block_table), block_table.shape[1],
        _ptr(idx), _ptr(lens), k, _ptr(swa_pages), swa_pages.shape[0] if W else 0,
        _ptr(swa_block_table), swa_block_table.shape[1] if W else 0, _ptr(swa_idx),
        _ptr(swa_lens), W, _ptr(attn_sink), R, H, float(scale), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel(), _ptr(err_flag), _stream(stream, dev)))
    return out, lse


def indexer_logits(q, weights, k_pages, block_table, lens, row_req=None, logits=None,
                   err_flag=None, stream=None):
    """Indexer scores of every row: float32 [num_rows, 64 * bt_stride] (or
    the given ``logits``); positions at or beyond a row's length are not
    written. See ds_indexer_logits."""
    _need(q, "q", torch.bfloat16, ndim=3)
    dev = q.device
    R, H, D = q.shape
    _need(weights, "weights", torch.float32, dev, 2)
    _need(k_pages, "k_pages", torch.bfloat16, dev, 3)
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(lens, "lens", torch.int32, dev, 1)
    if tuple(weights.shape) != (R, H):
        raise ValueError(f"weights must be [{R}, {H}], got {tuple(weights.shape)}")
    if lens.numel() != R:
        raise ValueError("lens must have one entry per row")
    if k_pages.shape[1] != 64 or k_pages.shape[2] != D:
        raise ValueError(f"k_pages must be [num_pages, 64, {D}], got {tuple(k_pages.shape)}")
    if row_req is not None:
        _need(row_req, "row_req", torch.int32, dev, 1)
        if row_req.numel() != R:
            raise ValueError("row_req must have one entry per row")
    bt_stride = block_table.shape[1]
    if logits is None:
        logits = torch.empty((R, 64 * bt_stride), dtype=torch.float32, device=dev)
    _need(logits, "logits", torch.float32, dev, 2)
    if logits.shape[0] != R:
        raise ValueError("logits must have one row per query row")
    if err_flag is not None:
        _need(err_flag, "err_flag", torch.int32, dev, 1)
    _check(lib().ds_indexer_logits(_ptr(q), _ptr(weights), _ptr(k_pages), k_pages.shape[0],
                                   _ptr(block_table), bt_stride, block_table.shape[0],
                                   _ptr(row_req), _ptr(lens), R, H, D, _ptr(logits),
                                   logits.shape[1], _ptr(err_flag), _stream(stream, dev)))
    return logits
