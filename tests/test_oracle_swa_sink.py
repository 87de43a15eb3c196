"""Pins of the oracle's decode over [top-k || sliding-window] entries with
attention sinks (oracle/attention.py: sparse_mla_rows_sink,
sparse_mla_decode_swa), against closed forms, a library routine and
invariances.
"""

import math

import numpy as np
import torch

import oracle

D = 576


def _bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _pool(rng, pages):
    return _bits(rng.standard_normal((pages, 64, D)))


def test_one_entry_with_sink_closed_form():
    rng = np.random.default_rng(0)
    K = oracle.bf16_bits_to_float64(_bits(rng.standard_normal((1, D))))
    q = oracle.bf16_bits_to_float64(_bits(rng.standard_normal((3, D))))
    sink = np.array([0.7, -np.inf, 40.0])
    scale = 0.05
    out, lse = oracle.sparse_mla_rows_sink(q, K, scale, sink)
    for h in range(3):
        logit = scale * float(q[h] @ K[0])
        tot = logit if sink[h] == -np.inf else float(np.logaddexp(logit, sink[h]))
        assert math.isclose(lse[h], tot, rel_tol=0, abs_tol=1e-12)
        np.testing.assert_allclose(out[h], K[0, :512] * math.exp(logit - tot), rtol=1e-12,
                                   atol=1e-300)


def test_no_entries():
    out, lse = oracle.sparse_mla_rows_sink(np.ones((2, D)), np.zeros((0, D)), 0.1,
                                           np.array([1.5, -np.inf]))
    assert (out == 0).all() and lse[0] == 1.5 and lse[1] == -np.inf


def test_zero_query_weights_every_entry_equally():
    rng = np.random.default_rng(1)
    K = oracle.bf16_bits_to_float64(_bits(rng.standard_normal((7, D))))
    sink = np.array([0.0, 2.0])
    out, lse = oracle.sparse_mla_rows_sink(np.zeros((2, D)), K, 0.3, sink)
    for h in range(2):
        denom = 7 + math.exp(sink[h])
        np.testing.assert_allclose(out[h], K[:, :512].sum(0) / denom, rtol=1e-12, atol=1e-12)
        assert math.isclose(lse[h], math.log(denom), abs_tol=1e-12)


def test_matches_float64_sdpa_with_a_sink_key():
    rng = np.random.default_rng(2)
    H, n, scale = 8, 50, 1 / math.sqrt(D)
    K = oracle.bf16_bits_to_float64(_bits(rng.standard_normal((n, D))))
    q = oracle.bf16_bits_to_float64(_bits(rng.standard_normal((H, D))))
    sink = rng.standard_normal(H) * 3
    sink[1] = -np.inf
    out, lse = oracle.sparse_mla_rows_sink(q, K, scale, sink)
    # The sink is one more key with a zero value; its logit comes from the mask.
    Kt = torch.from_numpy(np.concatenate([K, np.zeros((1, D))]))
    Vt = torch.from_numpy(np.concatenate([K[:, :512], np.zeros((1, 512))]))
    mask = torch.zeros((H, n + 1), dtype=torch.float64)
    mask[:, n] = torch.from_numpy(sink)
    qt = torch.from_numpy(q)
    want = torch.nn.functional.scaled_dot_product_attention(
        qt[None, :, None, :], Kt[None, None].expand(1, H, n + 1, D),
        Vt[None, None].expand(1, H, n + 1, 512), attn_mask=mask[None, :, None, :],
        scale=scale)[0, :, 0]
    np.testing.assert_allclose(out, want.numpy(), rtol=1e-10, atol=1e-12)
    logits = scale * qt @ Kt.T + mask
    np.testing.assert_allclose(lse, torch.logsumexp(logits, 1).numpy(), rtol=1e-12)


def test_decode_swa_uses_both_pools_and_reduces_to_plain_decode():
    rng = np.random.default_rng(3)
    B, H, k, W = 3, 16, 128, 64
    kv, swa = _pool(rng, 12), _pool(rng, 6)
    bt = np.stack([rng.permutation(12)[:4] for _ in range(B)]).astype(np.int32)
    sbt = np.stack([rng.permutation(6)[:2] for _ in range(B)]).astype(np.int32)
    lens = np.array([250, 0, 100], np.int32)
    slens = np.array([128, 70, 5], np.int32)
    idx = np.stack([rng.permutation(256)[:k] for _ in range(B)]).astype(np.int32)
    sidx = np.full((B, W), -1, np.int32)
    for b in range(B):
        w = min(W, int(slens[b]))
        sidx[b, :w] = np.arange(slens[b] - w, slens[b])   # the last w positions
    q = _bits(rng.standard_normal((B, H, D)))
    scale = 0.04
    sink = rng.standard_normal(H)
    out, lse = oracle.sparse_mla_decode_swa(q, kv, "bf16", bt, idx, lens, swa, sbt, sidx, slens,
                                            sink, scale)
    # Brute force: gather both lists' rows by hand and apply the definition.
    for b in range(B):
        rows = [oracle.bf16_bits_to_float64(kv[bt[b, p // 64], p % 64])
                for p in idx[b] if 0 <= p < lens[b]]
        rows += [oracle.bf16_bits_to_float64(swa[sbt[b, p // 64], p % 64])
                 for p in sidx[b] if 0 <= p < slens[b]]
        K = np.array(rows).reshape(-1, D)
        qb = oracle.bf16_bits_to_float64(q[b])
        S = scale * qb @ K.T
        for h in range(H):
            z = np.concatenate([S[h], [sink[h]]])
            m = z.max()
            w = np.exp(z - m)
            np.testing.assert_allclose(out[b, h], (w[:-1] @ K[:, :512]) / w.sum(), rtol=1e-10,
                                       atol=1e-12)
            assert math.isclose(lse[b, h], m + math.log(w.sum()), abs_tol=1e-10)
    # Without window entries and without sinks it is the plain decode.
    o2, l2 = oracle.sparse_mla_decode_swa(q, kv, "bf16", bt, idx, lens, None, None, None, None,
                                          None, scale)
    o3, l3 = oracle.sparse_mla_decode(q, kv, "bf16", bt, idx, lens, scale)
    np.testing.assert_allclose(o2, o3, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(np.isfinite(l2), np.isfinite(l3))
    # Permuting the window pool's pages (and its block table) changes nothing.
    perm = rng.permutation(6)
    inv = np.argsort(perm)
    o4, l4 = oracle.sparse_mla_decode_swa(q, kv, "bf16", bt, idx, lens, swa[perm], inv[sbt],
                                          sidx, slens, sink, scale)
    np.testing.assert_allclose(o4, out, rtol=1e-12, atol=1e-14)
