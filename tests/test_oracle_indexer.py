"""Pins for the indexer-score oracle (CPU only).

The adopted definition (DeepSeek-V3.2-Exp lightning indexer; the pages name
the indexer's MQA logits without a formula) is I[r, s] = sum_j w_j *
max(0, q_j . k_s). The oracle evaluates it with one matrix product and a
clamp. These checks do not retype that: they pin it to

* a hand-worked example (tests/golden/indexer_small.json): paging, the signed
  length clamp, an out-of-pool page (-inf) and negative weights;
* two identities of the clamp, max(0, x) - max(0, -x) = x and
  max(0, x) + max(0, -x) = |x|, so I(q) - I(-q) is the weighted plain dot
  product and I(q) + I(-q) the weighted absolute one (a dropped or misplaced
  clamp, a wrong sign or a lost weight fails one of them);
* positive homogeneity in q and in w, and invariance under a permutation of
  the pool's pages applied to the block table.
"""

import json
import os

import numpy as np
import pytest

from oracle.indexer import indexer_logits, indexer_row_length

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "indexer_small.json")


def _bf16_bits(x):
    x = np.asarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    # round to nearest even at bit 16 (inputs here are exactly representable)
    assert np.all((bits & 0xFFFF) == 0), "test values must be bf16-exact"
    return (bits >> 16).astype(np.uint16)


def test_golden_worked_example():
    g = json.load(open(GOLDEN))
    H, d, P = g["heads"], g["dim"], g["num_pages"]
    kp = np.zeros((P, 64, d), np.float32)
    for e in g["keys"]:
        kp[e["page"], e["slot"]] = e["k"]
    bt = np.array(g["block_table"], np.int64)
    rows = g["rows"]
    q = np.array([r["q"] for r in rows], np.float32)
    w = np.array([r["w"] for r in rows], np.float32)
    lens = np.array([r["len"] for r in rows], np.int64)
    req = np.array([r["req"] for r in rows], np.int64)
    out = indexer_logits(_bf16_bits(q), w, _bf16_bits(kp), bt, lens, row_req=req, width=200)
    for i, r in enumerate(rows):
        L = indexer_row_length(r["len"], bt.shape[1])
        if "expected" in r:
            assert L == len(r["expected"])
            np.testing.assert_array_equal(out[i, :L], r["expected"])
        if "expected_len" in r:
            assert L == r["expected_len"]
        if "expected_prefix" in r:
            np.testing.assert_array_equal(out[i, :len(r["expected_prefix"])], r["expected_prefix"])
        if "expected_tail" in r:
            tail = [float(x) for x in r["expected_tail"]]
            np.testing.assert_array_equal(out[i, L - len(tail):L], tail)
        if r["req"] == 2:   # positions 3..63 read zero keys
            np.testing.assert_array_equal(out[i, 3:64], 0.0)
        assert np.all(np.isnan(out[i, L:])), i


def _random_case(seed, R=3, H=8, d=32, P=6, width=300):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((R, H, d)).astype(np.float32)
    k = rng.standard_normal((P, 64, d)).astype(np.float32)
    q = (q.view(np.uint32) & 0xFFFF0000).view(np.float32)
    k = (k.view(np.uint32) & 0xFFFF0000).view(np.float32)
    w = rng.standard_normal((R, H)).astype(np.float32)
    bt = rng.permutation(P)[None, :].repeat(R, 0).astype(np.int64)
    lens = np.array([width, 130, 64][:R], np.int64)
    return q, w, k, bt, lens


def _bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _plain_keys(k, bt, r, L):
    pos = np.arange(L)
    return k[bt[r, pos // 64], pos % 64].astype(np.float64)


def test_clamp_identities():
    q, w, k, bt, lens = _random_case(1)
    Ip = indexer_logits(_bits(q), w, _bits(k), bt, lens)
    Im = indexer_logits(_bits(-q), w, _bits(k), bt, lens)
    for r in range(q.shape[0]):
        L = int(lens[r])
        keys = _plain_keys(k, bt, r, L)
        dots = np.einsum("hd,sd->hs", q[r].astype(np.float64), keys)
        wr = w[r].astype(np.float64)
        np.testing.assert_allclose(Ip[r, :L] - Im[r, :L], wr @ dots, rtol=1e-12, atol=1e-9)
        np.testing.assert_allclose(Ip[r, :L] + Im[r, :L], wr @ np.abs(dots), rtol=1e-12, atol=1e-9)


def test_positive_homogeneity():
    q, w, k, bt, lens = _random_case(2)
    I1 = indexer_logits(_bits(q), w, _bits(k), bt, lens)
    I2 = indexer_logits(_bits(2 * q), w, _bits(k), bt, lens)     # exact in bf16
    I3 = indexer_logits(_bits(q), 3 * w, _bits(k), bt, lens)
    fin = ~np.isnan(I1)
    np.testing.assert_allclose(I2[fin], 2 * I1[fin], rtol=1e-12)
    np.testing.assert_allclose(I3[fin], 3 * I1[fin], rtol=1e-6)   # 3w is rounded to float32


def test_page_permutation_invariance():
    q, w, k, bt, lens = _random_case(3)
    perm = np.random.default_rng(4).permutation(k.shape[0])   # new page id of old page p: perm[p]
    k2 = np.empty_like(k)
    k2[perm] = k
    bt2 = perm[bt]
    a = indexer_logits(_bits(q), w, _bits(k), bt, lens)
    b = indexer_logits(_bits(q), w, _bits(k2), bt2, lens)
    np.testing.assert_array_equal(a, b)


def test_row_length_clamp_is_signed():
    assert indexer_row_length(-5, 10) == 0
    assert indexer_row_length(0, 10) == 0
    assert indexer_row_length(639, 10) == 639
    assert indexer_row_length(641, 10) == 640
