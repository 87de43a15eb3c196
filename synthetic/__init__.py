"""Seeded synthetic inputs for the sparse top-k + sparse MLA path.

This module only draws random inputs and lays them out in the byte formats
the library reads. It holds none of the method's arithmetic (no top-k, no
gather, no attention): the oracle and the CUDA path both consume exactly the
tensors it returns.

Recipe (every workload):

* indexer scores: float32 N(0,1) on ``[row_start, row_end)``; columns outside
  a row's range are NaN so that any out-of-range read shows up as a mismatch.
  Tie-heavy workloads round N(0,1) to multiples of 1/8, or draw integers 0..7.
* q and the latent KV: N(0,1) rounded to bfloat16.
* FP8 KV (656-byte rows): per 128-element group ``scale = amax / 448`` (1.0 for
  an all-zero group), codes ``= round-to-nearest-even(x / scale)`` as
  ``float8_e4m3fn``, then the 4 float32 scales, then the 64-dim bf16 rope.
* block tables: one random permutation of the pool's pages, handed to the
  requests in turn; unused block-table slots hold -1.
* sizes follow the named workloads (``WORKLOADS``).
"""

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 64
D_QK = 576
D_V = 512
FP8_ROW_BYTES = 656


@dataclass
class Case:
    """One workload instance. Tensors live on ``device``."""
    name: str
    H: int
    k: int
    kv_dtype: str                  # "bf16" or "fp8"
    scale: float
    scores: torch.Tensor           # float32 [R, stride]
    row_starts: torch.Tensor       # int32 [R]
    row_ends: torch.Tensor         # int32 [R]
    q: torch.Tensor                # bfloat16 [R, H, 576]
    kv_pages: torch.Tensor         # bfloat16 [P, 64, 576] or uint8 [P, 64, 656]
    block_table: torch.Tensor      # int32 [num_requests, bt_stride]
    row_req: torch.Tensor          # int32 [R]  (block-table row of each query row)
    lens: torch.Tensor             # int32 [R]  (context length seen by each row)
    meta: dict = field(default_factory=dict)

    @property
    def R(self):
        return self.q.shape[0]

    # NumPy views for the oracle (bit patterns, not converted values).
    def np_scores(self):
        return self.scores.cpu().numpy()

    def np_q_bits(self):
        return self.q.cpu().view(torch.int16).numpy().view(np.uint16)

    def np_kv(self):
        kv = self.kv_pages.cpu()
        if self.kv_dtype == "bf16":
            return kv.view(torch.int16).numpy().view(np.uint16)
        return kv.numpy()

    def np_int(self, name):
        return getattr(self, name).cpu().numpy()


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def quantize_fp8_rows(latent_f32, rope_bf16):
    """Pack float32 latent [n, 512] + bf16 rope [n, 64] into uint8 [n, 656]."""
    n = latent_f32.shape[0]
    groups = latent_f32.reshape(n, 4, 128)
    amax = groups.abs().amax(dim=2)                                  # [n, 4]
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (groups / scale[:, :, None]).to(torch.float8_e4m3fn).reshape(n, 512)
    out = torch.empty((n, FP8_ROW_BYTES), dtype=torch.uint8, device=latent_f32.device)
    out[:, :512] = codes.view(torch.uint8)
    out[:, 512:528] = scale.to(torch.float32).contiguous().view(torch.uint8).reshape(n, 16)
    out[:, 528:] = rope_bf16.contiguous().view(torch.uint8).reshape(n, 128)
    return out


def _kv_pool(num_pages, kv_dtype, g, device, chunk_pages=2048):
    """Latent KV pool, generated in chunks to bound host/device peak memory."""
    if kv_dtype == "bf16":
        pool = torch.empty((num_pages, PAGE, D_QK), dtype=torch.bfloat16, device=device)
    elif kv_dtype == "fp8":
        pool = torch.empty((num_pages, PAGE, FP8_ROW_BYTES), dtype=torch.uint8, device=device)
    else:
        raise ValueError(kv_dtype)
    for p0 in range(0, num_pages, chunk_pages):
        p1 = min(num_pages, p0 + chunk_pages)
        x = _normal(((p1 - p0) * PAGE, D_QK), g, device)
        if kv_dtype == "bf16":
            pool[p0:p1] = x.to(torch.bfloat16).reshape(p1 - p0, PAGE, D_QK)
        else:
            rows = quantize_fp8_rows(x[:, :512], x[:, 512:].to(torch.bfloat16))
            pool[p0:p1] = rows.reshape(p1 - p0, PAGE, FP8_ROW_BYTES)
    return pool


def _scores(rows, stride, starts, ends, mode, g, device):
    s = torch.full((rows, stride), float("nan"), dtype=torch.float32, device=device)
    for r in range(rows):
        a, b = int(starts[r]), int(ends[r])
        a = max(0, a)
        b = min(stride, b)
        if b <= a:
            continue
        if mode == "normal":
            v = _normal((b - a,), g, device)
        elif mode == "eighths":
            v = torch.round(_normal((b - a,), g, device) * 8.0) / 8.0
        elif mode == "int8":
            v = torch.randint(0, 8, (b - a,), generator=g, device=device).to(torch.float32)
        else:
            raise ValueError(mode)
        s[r, a:b] = v
    return s


def _block_table(ctx_lens, g, device):
    """Random permutation of all pages, handed out to the requests in turn."""
    npages = [max(1, math.ceil(int(c) / PAGE)) for c in ctx_lens]
    total = sum(npages)
    perm = torch.randperm(total, generator=g, device=device).to(torch.int32)
    bt_stride = max(npages)
    bt = torch.full((len(ctx_lens), bt_stride), -1, dtype=torch.int32, device=device)
    off = 0
    for r, n in enumerate(npages):
        bt[r, :n] = perm[off:off + n]
        off += n
    return bt, total


def decode_case(name, ctx_lens, H, k, kv_dtype="bf16", seed=0, score_mode="normal",
                stride=None, device="cpu", scale=None):
    """A decode batch: row b is request b, scoring context [0, ctx_lens[b])."""
    ctx_lens = [int(c) for c in ctx_lens]
    B = len(ctx_lens)
    stride = int(stride if stride is not None else max(ctx_lens))
    g = _gen(seed, device)
    bt, num_pages = _block_table(ctx_lens, g, device)
    starts = torch.zeros(B, dtype=torch.int32, device=device)
    ends = torch.tensor(ctx_lens, dtype=torch.int32, device=device)
    scores = _scores(B, stride, [0] * B, ctx_lens, score_mode, g, device)
    q = _normal((B, H, D_QK), g, device).to(torch.bfloat16)
    kv = _kv_pool(num_pages, kv_dtype, g, device)
    return Case(name=name, H=H, k=k, kv_dtype=kv_dtype,
                scale=float(scale if scale is not None else 1.0 / math.sqrt(D_QK)),
                scores=scores, row_starts=starts, row_ends=ends, q=q, kv_pages=kv,
                block_table=bt, row_req=torch.arange(B, dtype=torch.int32, device=device),
                lens=ends.clone(), meta={"ctx_lens": ctx_lens, "seed": seed, "stride": stride})


def prefill_case(name, ctx, first_pos, T, H, k, kv_dtype="bf16", seed=3, device="cpu",
                 score_mode="normal", scale=None):
    """One request of ``ctx`` tokens; query tokens at positions first_pos..first_pos+T-1.

    Token t scores context [0, pos_t + 1) (causal), with row stride ``ctx``.
    """
    g = _gen(seed, device)
    bt, num_pages = _block_table([ctx], g, device)
    pos = torch.arange(first_pos, first_pos + T, dtype=torch.int32, device=device)
    starts = torch.zeros(T, dtype=torch.int32, device=device)
    ends = pos + 1
    if score_mode == "normal" and T * ctx > (1 << 24):
        # Large prefill score matrices: draw the whole matrix at once, then
        # NaN the causal tail (same recipe as ``_scores``, vectorised).
        scores = _normal((T, ctx), g, device)
        col = torch.arange(ctx, device=device)[None, :]
        scores = torch.where(col < ends[:, None], scores, torch.full_like(scores, float("nan")))
    else:
        scores = _scores(T, ctx, [0] * T, ends.tolist(), score_mode, g, device)
    q = _normal((T, H, D_QK), g, device).to(torch.bfloat16)
    kv = _kv_pool(num_pages, kv_dtype, g, device)
    return Case(name=name, H=H, k=k, kv_dtype=kv_dtype,
                scale=float(scale if scale is not None else 1.0 / math.sqrt(D_QK)),
                scores=scores, row_starts=starts, row_ends=ends, q=q, kv_pages=kv,
                block_table=bt, row_req=torch.zeros(T, dtype=torch.int32, device=device),
                lens=ends.clone(), meta={"ctx": ctx, "first_pos": first_pos, "seed": seed,
                                         "stride": ctx})


def mtp_case(name, seq_lens, next_n, H, k, kv_dtype="bf16", seed=5, score_mode="normal",
             stride=None, device="cpu", scale=None):
    """Multi-token decode: ``next_n`` query tokens per request (one target
    token and next_n - 1 draft tokens), every token reading its request's
    block-table row.

    Token j of request r scores the context [0, seq_lens[r] - next_n + 1 + j).
    That length is signed: it is negative for the first tokens of a padded
    request (seq_lens[r] == 0), and the top-k clamps it to an empty row.
    """
    seq_lens = [int(x) for x in seq_lens]
    B = len(seq_lens)
    R = B * next_n
    ends = [sl - next_n + 1 + j for sl in seq_lens for j in range(next_n)]
    stride = int(stride if stride is not None else max(1, max(seq_lens)))
    g = _gen(seed, device)
    bt, num_pages = _block_table([max(1, sl) for sl in seq_lens], g, device)
    starts = torch.zeros(R, dtype=torch.int32, device=device)
    ends_t = torch.tensor(ends, dtype=torch.int32, device=device)
    scores = _scores(R, stride, [0] * R, ends, score_mode, g, device)
    q = _normal((R, H, D_QK), g, device).to(torch.bfloat16)
    kv = _kv_pool(num_pages, kv_dtype, g, device)
    row_req = torch.arange(B, dtype=torch.int32, device=device).repeat_interleave(next_n)
    return Case(name=name, H=H, k=k, kv_dtype=kv_dtype,
                scale=float(scale if scale is not None else 1.0 / math.sqrt(D_QK)),
                scores=scores, row_starts=starts, row_ends=ends_t, q=q, kv_pages=kv,
                block_table=bt, row_req=row_req, lens=ends_t.clamp(min=0),
                meta={"seq_lens": seq_lens, "next_n": next_n, "seed": seed, "stride": stride})


def window_case(win_lens, W, kv_dtype="bf16", seed=7, device="cpu"):
    """A sliding-window pool: row b's window context has win_lens[b]
    positions and its index list holds the last min(W, win_lens[b]) of them,
    padded with -1 to W. Returns (pages, block_table, idx [B, W], lens [B])."""
    win_lens = [int(n) for n in win_lens]
    g = _gen(seed, device)
    bt, num_pages = _block_table([max(1, n) for n in win_lens], g, device)
    pages = _kv_pool(num_pages, kv_dtype, g, device)
    idx = torch.full((len(win_lens), W), -1, dtype=torch.int32)
    for b, n in enumerate(win_lens):
        m = min(W, n)
        idx[b, :m] = torch.arange(n - m, n, dtype=torch.int32)
    lens = torch.tensor(win_lens, dtype=torch.int32)
    return pages, bt, idx.to(device), lens.to(device)


@dataclass
class IndexerCase:
    """Indexer inputs: per-row queries and head weights, a paged key cache."""
    name: str
    q: torch.Tensor            # bfloat16 [R, H_I, 128]
    w: torch.Tensor            # float32 [R, H_I]
    k_pages: torch.Tensor      # bfloat16 [P, 64, 128]
    block_table: torch.Tensor  # int32 [R, bt_stride]
    lens: torch.Tensor         # int32 [R]
    meta: dict = field(default_factory=dict)


def indexer_case(name, ctx_lens, heads=64, dim=128, seed=8, device="cpu"):
    """Indexer inputs for rows of the given context lengths: q and the keys
    N(0,1) rounded to bf16, head weights N(0,1) / sqrt(heads) in float32, one
    random permutation of the key pages handed to the rows in turn."""
    ctx_lens = [int(c) for c in ctx_lens]
    g = _gen(seed, device)
    bt, num_pages = _block_table([max(1, c) for c in ctx_lens], g, device)
    q = _normal((len(ctx_lens), heads, dim), g, device).to(torch.bfloat16)
    w = _normal((len(ctx_lens), heads), g, device) / math.sqrt(heads)
    k = torch.empty((num_pages, PAGE, dim), dtype=torch.bfloat16, device=device)
    for p0 in range(0, num_pages, 4096):
        p1 = min(num_pages, p0 + 4096)
        k[p0:p1] = _normal(((p1 - p0), PAGE, dim), g, device).to(torch.bfloat16)
    lens = torch.tensor(ctx_lens, dtype=torch.int32, device=device)
    return IndexerCase(name=name, q=q, w=w, k_pages=k, block_table=bt, lens=lens,
                       meta={"ctx_lens": ctx_lens, "seed": seed})


def _uniform_ints(lo, hi, n, seed):
    g = torch.Generator().manual_seed(int(seed) + 1000003)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


# The named workloads. Sizes are exact; seeds are fixed.
WORKLOADS = {
    "tiny_decode": dict(kind="decode", B=2, H=16, ctx=(1024, 1024), k=128, kv="bf16",
                        scores="eighths", seed=0),
    "tp2_decode": dict(kind="decode", B=32, H=64, ctx=(4096, 32768), k=2048, kv="bf16",
                       scores="normal", seed=1, stride=32768),
    "tp1_fp8_decode": dict(kind="decode", B=128, H=128, ctx=(8192, 131072), k=2048, kv="fp8",
                           scores="normal", seed=2, stride=131072),
    "chunked_prefill": dict(kind="prefill", T=4096, H=128, ctx=65536, first_pos=61440, k=2048,
                            kv="bf16", scores="normal", seed=3),
    # TP2 decode plus a 128-entry sliding window (second pool) and per-head sinks.
    "tp2_decode_swa": dict(kind="decode_swa", B=32, H=64, ctx=(4096, 32768), k=2048, kv="bf16",
                           scores="normal", seed=6, stride=32768, swa_width=128),
    # MTP4 decode: one target and four draft tokens per request.
    "tp2_mtp4_decode": dict(kind="mtp", B=32, next_n=5, H=64, ctx=(4096, 32768), k=2048,
                            kv="bf16", scores="normal", seed=5, stride=32768),
}


# The indexer in front of the TP2-shaped decode batch: its rows' contexts,
# 64 indexer heads of dimension 128 (the DeepSeek-V3.2 indexer's shape).
INDEXER_WORKLOADS = {
    "tp2_indexer": dict(B=32, ctx=(4096, 32768), ctx_seed=1, heads=64, dim=128, seed=8, k=2048),
}


def indexer_workload(name, device="cpu"):
    w = INDEXER_WORKLOADS[name]
    ctx = _uniform_ints(w["ctx"][0], w["ctx"][1], w["B"], w["ctx_seed"])
    return indexer_case(name, ctx, w["heads"], w["dim"], w["seed"], device)


def workload_case(name, device="cpu", rows=None):
    """Build a named workload. ``rows`` (decode only) truncates the batch."""
    w = WORKLOADS[name]
    if w["kind"] == "decode":
        lo, hi = w["ctx"]
        B = w["B"] if rows is None else int(rows)
        ctx = [lo] * B if lo == hi else _uniform_ints(lo, hi, w["B"], w["seed"])[:B]
        return decode_case(name, ctx, w["H"], w["k"], w["kv"], w["seed"], w["scores"],
                           stride=w.get("stride"), device=device)
    if w["kind"] == "mtp":
        lo, hi = w["ctx"]
        B = w["B"] if rows is None else int(rows)
        return mtp_case(name, _uniform_ints(lo, hi, w["B"], w["seed"])[:B], w["next_n"], w["H"],
                        w["k"], w["kv"], w["seed"], w["scores"], stride=w.get("stride"),
                        device=device)
    T = w["T"] if rows is None else int(rows)
    return prefill_case(name, w["ctx"], w["ctx"] - T if rows is not None else w["first_pos"],
                        T, w["H"], w["k"], w["kv"], w["seed"], device)


def invariance_batch(batch_size, slot, target_seed=0, batch_seed=4, device="cpu",
                     H=64, k=2048, target_ctx=16384, max_ctx=32768, kv_dtype="bf16"):
    """Batch-invariance stress: one fixed request at ``slot`` among random neighbours.

    The target request (ctx ``target_ctx``, integer scores 0..7, its q rows and
    its latent rows) is drawn from ``target_seed`` alone, so it is identical
    in every batch. Neighbours draw lengths uniform in [1, max_ctx] from
    ``batch_seed``. Every batch has its own pool and page permutation, so the
    target's rows sit at different physical pages in each batch. With
    ``kv_dtype="fp8"`` the pool holds 656-byte FP8 rows (the target's rows
    quantised by the same rule as every other row).
    """
    gt = _gen(target_seed, device)
    t_scores = torch.randint(0, 8, (target_ctx,), generator=gt, device=device).to(torch.float32)
    t_q = _normal((H, D_QK), gt, device).to(torch.bfloat16)
    t_rows = _normal((target_ctx, D_QK), gt, device)
    if kv_dtype == "bf16":
        t_rows = t_rows.to(torch.bfloat16)
    else:
        t_rows = quantize_fp8_rows(t_rows[:, :512], t_rows[:, 512:].to(torch.bfloat16))

    gb = _gen(batch_seed * 1000 + batch_size, device)
    nb_ctx = torch.randint(1, max_ctx + 1, (batch_size,), generator=gb, device=device).tolist()
    ctx = [target_ctx if i == slot else int(nb_ctx[i]) for i in range(batch_size)]
    bt, num_pages = _block_table(ctx, gb, device)
    pool = _kv_pool(num_pages, kv_dtype, gb, device)
    # Place the target's rows into its pages of this batch's pool.
    tp = math.ceil(target_ctx / PAGE)
    pages = bt[slot, :tp].long()
    pool[pages] = t_rows.reshape(tp, PAGE, t_rows.shape[-1])

    scores = torch.full((batch_size, max_ctx), float("nan"), dtype=torch.float32, device=device)
    for i in range(batch_size):
        if i == slot:
            scores[i, :target_ctx] = t_scores
        else:
            scores[i, :ctx[i]] = torch.randint(0, 8, (ctx[i],), generator=gb,
                                               device=device).to(torch.float32)
    q = _normal((batch_size, H, D_QK), gb, device).to(torch.bfloat16)
    q[slot] = t_q
    ends = torch.tensor(ctx, dtype=torch.int32, device=device)
    return Case(name=f"invariance_b{batch_size}_s{slot}", H=H, k=k, kv_dtype=kv_dtype,
                scale=1.0 / math.sqrt(D_QK), scores=scores,
                row_starts=torch.zeros(batch_size, dtype=torch.int32, device=device),
                row_ends=ends, q=q, kv_pages=pool, block_table=bt,
                row_req=torch.arange(batch_size, dtype=torch.int32, device=device),
                lens=ends.clone(), meta={"slot": slot, "ctx": ctx})
