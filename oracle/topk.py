"""Oracle for the deterministic per-row top-k (test infrastructure only).

Follows "[DeepSeek-V4][Preview][DO NOT MERGE] Batch-invariant kernels for
0-diff RL", section "Deterministic sparse top-k": the selector ranks a row's
positions by a composite (score, index) key with a stable tie-break, and the
selected indices are then put in canonical (ascending) order before the
attention step, so equal scores or request offsets never change the result.

The row length and the -1 padding follow "[Bugfix] Make DSV4 sparse MLA work
end-to-end for plain decode, MTP, and DSpark", section "What is fixed": the
length is computed signed and clamped before use, and unused top-k slots hold
-1 rather than 0..k-1.

Readings where the pages are silent (each is a fixed rule so results are
testable bit for bit):

* indices are relative to ``row_start`` (the position within the request's
  context, which is what the page lookup needs);
* -0.0 and +0.0 are equal scores (the lower index wins the tie);
* NaN ranks below every number, -inf included; NaNs tie with one another;
* a row whose ``row_start`` lies outside ``[0, stride]`` is empty;
* rows shorter than k take every position, then -1 up to k.
"""

import numpy as np


def row_length(row_start, row_end, stride):
    """Signed, clamped row length (section "What is fixed", PR 51538).

    ``clamp(row_end - row_start, 0, stride - row_start)`` computed in Python
    integers, so a negative difference can never wrap to a huge unsigned
    value. A start outside ``[0, stride]`` gives an empty row.
    """
    row_start = int(row_start)
    row_end = int(row_end)
    stride = int(stride)
    if row_start < 0 or row_start > stride:
        return 0
    return max(0, min(row_end - row_start, stride - row_start))


def _order(values):
    """Positions of ``values`` in selection order: score desc, index asc.

    ``np.lexsort`` sorts by its last key first. Keys, most significant first:
    NaN flag (numbers before NaN), negated score (larger score first; -0.0 and
    +0.0 compare equal), position (lower first). Ties in every key cannot
    happen because positions are distinct, so the order is total.
    """
    v = np.asarray(values, dtype=np.float64)
    nan = np.isnan(v)
    neg = np.where(nan, 0.0, -v)
    pos = np.arange(v.shape[0], dtype=np.int64)
    return np.lexsort((pos, neg, nan))


def topk_per_row(scores, row_starts, row_ends, k):
    """Deterministic top-k of every row, canonicalised ascending, -1 padded.

    ``scores``: float32 [num_rows, stride]; row ``b`` ranks
    ``scores[b, row_starts[b] : row_starts[b] + L_b]``.
    Returns int32 [num_rows, k]: the selected positions (relative to the row
    start) in ascending order, then -1 in the slots beyond ``min(k, L_b)``.
    """
    scores = np.asarray(scores)
    num_rows, stride = scores.shape
    out = np.full((num_rows, k), -1, dtype=np.int32)
    for b in range(num_rows):
        n = row_length(row_starts[b], row_ends[b], stride)
        if n == 0:
            continue
        start = int(row_starts[b])
        vals = scores[b, start:start + n]
        chosen = np.sort(_order(vals)[: min(k, n)])
        out[b, : chosen.shape[0]] = chosen.astype(np.int32)
    return out


def _better(a, i, b, j):
    """True when (score a at i) precedes (score b at j) in selection order."""
    a_nan = a != a
    b_nan = b != b
    if a_nan != b_nan:
        return b_nan          # a number precedes NaN
    if not a_nan and a != b:
        return a > b          # larger score first (-0.0 == +0.0 here)
    return i < j              # equal scores: lower index first


def topk_rank_bruteforce(values, k):
    """Selected set by the rank definition, O(n^2), pure Python.

    Position i is selected iff fewer than k positions precede it in the
    composite order. Independent of any sort; used to pin ``topk_per_row``.
    Returns the selected positions ascending.
    """
    vals = [float(x) for x in values]
    n = len(vals)
    sel = []
    for i in range(n):
        ahead = 0
        for j in range(n):
            if j != i and _better(vals[j], j, vals[i], i):
                ahead += 1
        if ahead < k:
            sel.append(i)
    return sel

