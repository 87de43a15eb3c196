"""Pins for the top-k oracle (CPU only).

The oracle sorts; these checks do not. They pin it to:

* hand-derived tie tables (tests/golden/topk_ties.json), worked out from the
  rules of "Batch-invariant kernels for 0-diff RL" (vllm PR 54955), section
  "Deterministic sparse top-k", and "Make DSV4 sparse MLA work end-to-end"
  (vllm PR 51538), section "What is fixed";
* the rank definition, counted pair by pair in O(n^2) on every small input
  over a tie-heavy alphabet;
* library routines on inputs where the answer is unique without any
  tie-break (distinct scores: ``heapq.nlargest``, ``torch.topk``);
* the counting invariant on integer scores (everything above the threshold
  value, then the lowest-index positions that hold it);
* offset invariance (the same row at another ``row_start`` gives the same
  relative indices).
"""

import heapq
import itertools
import json
import math
import os
import random

import numpy as np
import pytest
import torch

from oracle import topk_per_row, topk_rank_bruteforce, row_length

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "topk_ties.json")


def _row(scores, start, end, k, stride=None):
    vals = [float(s) for s in scores]
    stride = len(vals) if stride is None else stride
    arr = np.full((1, stride), np.nan, dtype=np.float32)
    arr[0, : len(vals)] = vals
    return topk_per_row(arr, np.array([start]), np.array([end]), k)[0].tolist()


def test_golden_tie_table():
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    assert len(cases) >= 15
    for c in cases:
        got = _row(c["scores"], c["row_start"], c["row_end"], c["k"])
        assert got == c["expected"], c["name"]


def test_row_length_clamp_signed():
    # A padded decode slot: seq_len 0 with next_n 2 gives end - start = -1.
    assert row_length(0, -1, 100) == 0
    assert row_length(5, 3, 100) == 0
    assert row_length(10, 10 ** 9, 100) == 90
    assert row_length(-3, 5, 100) == 0
    assert row_length(101, 105, 100) == 0
    assert row_length(100, 105, 100) == 0
    assert row_length(0, 100, 100) == 100


ALPHABET = [float("-inf"), -1.0, -0.0, 0.0, 0.5, 1.0, float("nan")]


def test_bruteforce_exhaustive_small():
    """Every row of length <= 4 over a tie-heavy alphabet, every k."""
    for n in range(0, 5):
        for vals in itertools.product(ALPHABET, repeat=n):
            for k in range(1, n + 2):
                got = _row(vals, 0, n, k)
                want = topk_rank_bruteforce(vals, k)
                want = want + [-1] * (k - len(want))
                assert got == want, (vals, k)


def test_bruteforce_random_longer():
    rng = random.Random(1234)
    for _ in range(300):
        n = rng.randint(5, 12)
        vals = [rng.choice(ALPHABET) for _ in range(n)]
        k = rng.randint(1, n + 1)
        got = _row(vals, 0, n, k)
        want = topk_rank_bruteforce(vals, k)
        assert got == want + [-1] * (k - len(want))


def test_distinct_scores_match_heapq_and_torch():
    """With distinct scores the selected set needs no tie-break."""
    rng = np.random.default_rng(7)
    for n, k in [(50, 7), (300, 64), (1000, 128), (4096, 2048)]:
        vals = rng.permutation(n).astype(np.float32) * np.float32(0.25) - np.float32(3.0)
        got = _row(vals.tolist(), 0, n, k)
        want_h = sorted(heapq.nlargest(k, range(n), key=lambda i: vals[i]))
        want_t = sorted(torch.topk(torch.from_numpy(vals), k).indices.tolist())
        assert got == want_h == want_t


def test_counting_invariant_integer_scores():
    """Scores 0..7: all positions above threshold t, then the first ones at t."""
    rng = np.random.default_rng(3)
    for n, k in [(100, 10), (1000, 333), (5000, 2048)]:
        vals = rng.integers(0, 8, n).astype(np.float32)
        got = [i for i in _row(vals.tolist(), 0, n, k) if i >= 0]
        desc = sorted(vals.tolist(), reverse=True)
        t = desc[k - 1]
        above = [i for i in range(n) if vals[i] > t]
        at = [i for i in range(n) if vals[i] == t][: k - len(above)]
        assert got == sorted(above + at)
        assert len(got) == k


def test_offset_invariance():
    rng = np.random.default_rng(11)
    base = np.round(rng.standard_normal(200) * 8) / 8
    want = _row(base.tolist(), 0, 200, 37)
    for off in [1, 3, 17, 64]:
        shifted = [float("nan")] * off + base.tolist()
        got = _row(shifted, off, off + 200, 37)
        assert got == want


def test_ascending_and_padding_shape():
    rng = np.random.default_rng(5)
    R, stride, k = 6, 300, 64
    scores = rng.standard_normal((R, stride)).astype(np.float32)
    starts = np.array([0, 10, 0, 5, 0, 299])
    ends = np.array([300, 40, 64, 5, -1, 400])
    idx = topk_per_row(scores, starts, ends, k)
    for b in range(R):
        L = row_length(starts[b], ends[b], stride)
        n = min(k, L)
        row = idx[b].tolist()
        assert all(x == -1 for x in row[n:])
        valid = row[:n]
        assert all(0 <= x < L for x in valid)
        assert all(a < b_ for a, b_ in zip(valid, valid[1:]))
        if L <= k:
            assert valid == list(range(L))


def test_all_equal_row_gives_prefix():
    for n, k in [(10, 3), (2048, 2048), (5000, 2048)]:
        got = _row([2.0] * n, 0, n, k)
        assert got == list(range(min(n, k))) + [-1] * max(0, k - n)


def test_exactness_makes_selection_unique():
    """The total order leaves nothing to chance: shuffling equal keys' storage
    order never changes the answer because the index is part of the key."""
    vals = [1.0, 1.0, 1.0, 2.0, 2.0, 0.0]
    a = _row(vals, 0, 6, 4)
    assert a == [0, 1, 3, 4]
    assert math.isnan(float("nan"))
