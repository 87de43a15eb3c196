"""Oracle for the indexer scores that feed the top-k (test infrastructure only).

The pages name this step without defining it: "[SM120] Sync DS4 with upstream
main + validated perf backports" routes the indexer's "MQA logits" through a
dedicated kernel and derives a "paged-MQA" warm-up width, and "[Bugfix] Make
DSV4 sparse MLA work end-to-end ...", section "What is fixed", gives the
DSA indexer one context length per query token. So the scores are multi-head
queries against one shared key per context position (MQA), read from a
paged key cache, one row per query token.

The formula is taken from outside the pages: the "lightning indexer" of the
DeepSeek-V3.2-Exp technical report, whose scores the sparse attention's top-k
selects from. For query row r and context position s,

    I[r, s] = sum_j  w[r, j] * max(0, q[r, j, :] . k[s, :])

over the indexer heads j, with per-row head weights w. Readings where the
pages are silent (each stated once more in the function's docstring):

* q and the key cache are bfloat16, w is float32, the score is computed
  exactly (here in float64);
* the key of position s sits at ``k_pages[block_table[req, s // 64], s % 64]``
  (the same paged layout as the latent KV), ``req = row_req[r]`` or r;
* row r scores positions ``0 .. L_r - 1`` with ``L_r = clamp(lens[r], 0,
  64 * bt_stride)`` (signed, as for the top-k); a position whose page id lies
  outside the pool scores -inf;
* positions at or beyond ``L_r`` are not scores: NaN here.

Everything is float64, no blocking or reordering beyond the definition.
"""

import numpy as np

from .fp8 import bf16_bits_to_float64

PAGE = 64


def indexer_row_length(length, bt_stride):
    """Scored positions of a row: ``clamp(length, 0, 64 * bt_stride)``, signed."""
    return max(0, min(int(length), PAGE * int(bt_stride)))


def indexer_logits(q_bits, weights, k_pages_bits, block_table, lens, row_req=None, width=None):
    """Indexer scores, float64 [R, width] (NaN beyond each row's length).

    ``q_bits``: bf16 bit patterns uint16 [R, H_I, d]; ``weights``: float32
    [R, H_I]; ``k_pages_bits``: bf16 bits uint16 [P, 64, d];
    ``block_table``: int [num_requests, bt_stride]; ``lens``: int [R];
    ``row_req``: int [R] or None (row r reads block-table row r);
    ``width``: columns of the result (default: the longest row).
    """
    q = bf16_bits_to_float64(np.asarray(q_bits))                 # [R, H, d]
    w = np.asarray(weights, dtype=np.float32).astype(np.float64)  # [R, H]
    kp = np.asarray(k_pages_bits)
    bt = np.asarray(block_table, dtype=np.int64)
    R = q.shape[0]
    num_pages = kp.shape[0]
    Ls = [indexer_row_length(lens[r], bt.shape[1]) for r in range(R)]
    if width is None:
        width = max(Ls) if Ls else 0
    out = np.full((R, int(width)), np.nan, dtype=np.float64)
    for r in range(R):
        L = Ls[r]
        if L == 0:
            continue
        req = r if row_req is None else int(row_req[r])
        pos = np.arange(L, dtype=np.int64)
        pages = bt[req, pos // PAGE]
        ok = (pages >= 0) & (pages < num_pages)
        scores = np.full(L, -np.inf, dtype=np.float64)
        if ok.any():
            keys = bf16_bits_to_float64(kp[pages[ok], pos[ok] % PAGE])   # [n, d]
            dots = q[r] @ keys.T                                          # [H, n]
            scores[ok] = w[r] @ np.maximum(dots, 0.0)
        out[r, :L] = scores
    return out
