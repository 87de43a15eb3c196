"""Oracle for the paged gather + sparse MLA attention (test infrastructure only).

Follows "[DeepSeek-V4][Preview][DO NOT MERGE] Batch-invariant kernels for
0-diff RL", section "Sparse MLA and FlashMLA": decode gathers the selected KV
entries and computes attention over them; prefill processes every query token
independently. The computed quantity is the plain definition

    S[h, j]   = scale * sum_d q[h, d] * K[j, d]          (d over 576 = 512 + 64)
    out[h, :] = sum_j softmax_j(S[h, :]) * V[j, :]        (V = K[:, :512])
    lse[h]    = log(sum_j exp(S[h, j]))                   (natural log)

with one latent KV row per entry shared by every head. The slot of a context
position follows the paged layout of "[Bugfix] Make DSV4 sparse MLA work
end-to-end ...", section "What is fixed" (slot = block_id * block_size +
offset): ``page = block_table[row, pos // 64]``, ``slot = pos % 64``.

Readings where the pages are silent:

* an entry is valid iff ``0 <= idx < lens[row]`` and its page id lies in
  ``[0, num_pages)``; every other entry (the -1 padding included) is skipped;
* a row with no valid entry gives ``out = 0`` and ``lse = -inf``;
* V is the first 512 dims of the same latent row (the rope part only enters
  the scores);
* the FP8 row is 656 bytes: 512 E4M3 codes, then 4 little-endian float32
  scales (dims 0-127, 128-255, 256-383, 384-511), then 64 little-endian
  bfloat16 rope values.

Everything is float64; no blocking, splitting or reordering beyond the
definition above.
"""

import numpy as np

from .fp8 import e4m3_to_float64, bf16_bits_to_float64

PAGE = 64
D_QK = 576
D_V = 512
D_LATENT = 512
FP8_ROW_BYTES = 656


def _decode_fp8_rows(raw):
    """float64 [n, 576] from raw FP8 rows uint8 [n, 656]."""
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    n = raw.shape[0]
    latent = e4m3_to_float64(raw[:, :D_LATENT])
    scales = raw[:, 512:528].copy().view("<f4").astype(np.float64)   # [n, 4]
    latent = latent * np.repeat(scales, 128, axis=1)
    rope = bf16_bits_to_float64(raw[:, 528:656].copy().view("<u2"))  # [n, 64]
    out = np.empty((n, D_QK), dtype=np.float64)
    out[:, :D_LATENT] = latent
    out[:, D_LATENT:] = rope
    return out


def gather_latent_rows(kv_pages, kv_dtype, bt_row, positions):
    """Latent rows of the given context positions as float64 [n, 576].

    ``kv_pages``: uint16 bf16 bits [P, 64, 576] (``kv_dtype == "bf16"``) or
    uint8 [P, 64, 656] (``kv_dtype == "fp8"``). ``bt_row``: the request's
    block-table row. Positions must be valid (see ``_valid_entries``).
    """
    positions = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(bt_row, dtype=np.int64)[positions // PAGE]
    slots = positions % PAGE
    rows = kv_pages[pages, slots]
    if kv_dtype == "bf16":
        return bf16_bits_to_float64(rows)
    if kv_dtype == "fp8":
        return _decode_fp8_rows(rows)
    raise ValueError(f"kv_dtype must be 'bf16' or 'fp8', got {kv_dtype!r}")


def _valid_entries(idx_row, length, bt_row, num_pages):
    """The valid entries of one idx row, in their given order."""
    out = []
    for pos in np.asarray(idx_row, dtype=np.int64).tolist():
        if pos < 0 or pos >= int(length):
            continue
        if pos // PAGE >= len(bt_row):
            continue
        page = int(bt_row[pos // PAGE])
        if page < 0 or page >= num_pages:
            continue
        out.append(pos)
    return out


def sparse_mla_rows(q_rows, K, scale):
    """Attention of H query rows over n gathered latent rows (float64).

    ``q_rows``: float64 [H, 576]; ``K``: float64 [n, 576].
    Returns ``out`` float64 [H, 512] and ``lse`` float64 [H].
    """
    H = q_rows.shape[0]
    if K.shape[0] == 0:
        return np.zeros((H, D_V)), np.full(H, -np.inf)
    S = scale * (q_rows @ K.T)                      # [H, n]
    m = S.max(axis=1, keepdims=True)
    p = np.exp(S - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ K[:, :D_V]) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def _rows(q_bits, kv_pages, kv_dtype, block_table, row_req, idx, lens, scale, rows):
    H = q_bits.shape[1]
    num_pages = kv_pages.shape[0]
    out = np.zeros((len(rows), H, D_V))
    lse = np.full((len(rows), H), -np.inf)
    for i, r in enumerate(rows):
        bt_row = block_table[int(row_req[r])]
        ent = _valid_entries(idx[r], lens[r], bt_row, num_pages)
        K = gather_latent_rows(kv_pages, kv_dtype, bt_row, ent) if ent else np.zeros((0, D_QK))
        q = bf16_bits_to_float64(q_bits[r])
        out[i], lse[i] = sparse_mla_rows(q, K, scale)
    return out, lse


def sparse_mla_decode(q_bits, kv_pages, kv_dtype, block_table, idx, lens, scale, rows=None):
    """Decode: query row b uses block-table row b.

    ``q_bits``: uint16 bf16 bits [B, H, 576]; ``idx``: int32 [B, k];
    ``lens``: int32 [B]. ``rows`` optionally restricts the computation to a
    sample of row ids (results come back in that order).
    Returns ``out`` float64 [len(rows), H, 512] and ``lse`` [len(rows), H].
    """
    B = q_bits.shape[0]
    rows = list(range(B)) if rows is None else list(rows)
    return _rows(q_bits, kv_pages, kv_dtype, block_table, np.arange(B), idx, lens, scale, rows)


def sparse_mla_prefill(q_bits, kv_pages, kv_dtype, block_table, row_req, idx, lens, scale, rows=None):
    """Prefill: query token t uses block-table row ``row_req[t]``.

    Every token is computed on its own (section "Sparse MLA and FlashMLA":
    prefill chunks each request independently rather than by a batch plan).
    """
    T = q_bits.shape[0]
    rows = list(range(T)) if rows is None else list(rows)
    return _rows(q_bits, kv_pages, kv_dtype, block_table, row_req, idx, lens, scale, rows)


def sparse_mla_rows_sink(q_rows, K, scale, sink):
    """Attention of H query rows over n latent rows plus one sink logit per head.

    The sink of head h is a logit ``sink[h]`` (natural-log units, the same
    units as ``scale * q . K``) that joins the softmax denominator with no
    value row; ``-inf`` means no sink:

        out[h, :] = sum_j exp(S[h, j]) V[j, :] / (sum_j exp(S[h, j]) + exp(sink[h]))
        lse[h]    = log(sum_j exp(S[h, j]) + exp(sink[h]))

    A head with no valid entry and no sink gives out = 0 and lse = -inf; with
    a sink and no entry, out = 0 and lse = sink.
    """
    H = q_rows.shape[0]
    sink = np.asarray(sink, dtype=np.float64)
    S = scale * (q_rows @ K.T) if K.shape[0] else np.zeros((H, 0))
    out = np.zeros((H, D_V))
    lse = np.full(H, -np.inf)
    for h in range(H):
        logits = np.concatenate([S[h], [sink[h]]])
        m = logits.max()
        if m == -np.inf:
            continue
        w = np.exp(logits - m)                       # the sink's weight is w[-1]
        denom = w.sum()
        out[h] = (w[:-1] @ K[:, :D_V]) / denom if K.shape[0] else 0.0
        lse[h] = m + np.log(denom)
    return out, lse


def sparse_mla_decode_swa(q_bits, kv_pages, kv_dtype, block_table, idx, lens,
                          swa_pages, swa_block_table, swa_idx, swa_lens, sink, scale, rows=None):
    """Decode over the concatenation [top-k entries of the compressed KV ||
    sliding-window entries of the window KV], with a per-head attention sink.

    "[DeepSeek-V4][Preview][DO NOT MERGE] Batch-invariant kernels for 0-diff
    RL", section "Sparse MLA and FlashMLA": decode gathers compressed and
    sliding-window KV and runs one sparse attention over both; the section
    on model loading keeps -inf padding in the attention sinks. "[Bugfix]
    Make DSV4 sparse MLA work end-to-end ...", section "What is fixed": the
    window index list is padded to a multiple of 64 entries (-1 padding).

    Readings where the pages are silent: the window entries are positions
    in their own paged pool (same row format and element type as the
    compressed pool), looked up through their own block table and valid iff
    ``0 <= swa_idx < swa_lens[row]``; ``sink`` is float [H] in natural-log
    units (``None`` or -inf: no sink). Attention is the plain definition of
    ``sparse_mla_rows_sink`` over all valid entries of both lists.
    """
    B, H = q_bits.shape[0], q_bits.shape[1]
    rows = list(range(B)) if rows is None else list(rows)
    sink = np.full(H, -np.inf) if sink is None else np.asarray(sink, dtype=np.float64)
    out = np.zeros((len(rows), H, D_V))
    lse = np.full((len(rows), H), -np.inf)
    for i, r in enumerate(rows):
        parts = []
        for pages, bt, ix, ln in ((kv_pages, block_table, idx, lens),
                                  (swa_pages, swa_block_table, swa_idx, swa_lens)):
            if pages is None or ix is None:
                continue
            ent = _valid_entries(ix[r], ln[r], bt[r], pages.shape[0])
            if ent:
                parts.append(gather_latent_rows(pages, kv_dtype, bt[r], ent))
        K = np.concatenate(parts) if parts else np.zeros((0, D_QK))
        q = bf16_bits_to_float64(q_bits[r])
        out[i], lse[i] = sparse_mla_rows_sink(q, K, scale, sink)
    return out, lse
