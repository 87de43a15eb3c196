"""Pins for the gather + sparse attention oracle and the element decoders (CPU only).

The oracle evaluates softmax(scale * q K^T) V with a float64 matmul. These
checks tie it to facts that do not go through that code:

* closed forms: q = 0 gives the mean of V and lse = ln|J|; one valid entry
  gives its V row and lse = scale * q.K; two entries with a score gap D give
  sigmoid(D) V1 + sigmoid(-D) V2;
* a textbook softmax written with ``math.fsum`` scalar loops on tiny sizes;
* a library routine on a special case: dense attention over every position
  equals ``torch.nn.functional.scaled_dot_product_attention`` in float64;
* page permutation invariance and the page/slot arithmetic of the paged
  layout ("Make DSV4 sparse MLA work end-to-end", vllm PR 51538, section
  "What is fixed": slot = block_id * block_size + offset);
* the FP8 E4M3 and bfloat16 decoders against torch's own dtype conversions
  over every code.
"""

import math

import numpy as np
import torch
import torch.nn.functional as F

from oracle import (bf16_bits_to_float64, e4m3_to_float64, gather_latent_rows,
                    sparse_mla_decode, sparse_mla_prefill, sparse_mla_rows)

PAGE, DQK, DV = 64, 576, 512
SCALE = 1.0 / math.sqrt(DQK)


def _bf16_bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _pool(num_pages, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((num_pages, PAGE, DQK), generator=g)
    return _bf16_bits(x)


def _q(B, H, seed):
    g = torch.Generator().manual_seed(seed)
    return _bf16_bits(torch.randn((B, H, DQK), generator=g))


def test_bf16_decoder_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = bf16_bits_to_float64(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_decoder_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_to_float64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()
    assert e4m3_to_float64(np.array([0x7E], np.uint8))[0] == 448.0
    assert e4m3_to_float64(np.array([0x01], np.uint8))[0] == 2.0 ** -9


def test_gather_page_slot_arithmetic():
    """Each stored row encodes its own (page, slot); gathering returns them."""
    P = 5
    pool = np.zeros((P, PAGE, DQK), dtype=np.float32)
    for p in range(P):
        for s in range(PAGE):
            pool[p, s, 0] = p
            pool[p, s, 1] = s
    bits = _bf16_bits(pool)
    bt = np.array([3, 0, 4, 1, 2])
    pos = np.array([0, 63, 64, 130, 319])
    rows = gather_latent_rows(bits, "bf16", bt, pos)
    assert rows[:, 0].tolist() == [bt[x // PAGE] for x in pos]
    assert rows[:, 1].tolist() == [x % PAGE for x in pos]


def test_uniform_scores_give_mean_of_v():
    pool = _pool(4, 1)
    bt = np.array([[2, 0, 3, 1]])
    idx = np.array([[0, 5, 9, 70, 128, 200, 255, -1]], dtype=np.int32)
    q = np.zeros((1, 8, DQK), dtype=np.uint16)          # bf16 +0.0
    out, lse = sparse_mla_decode(q, pool, "bf16", bt, idx, np.array([256]), SCALE)
    J = [0, 5, 9, 70, 128, 200, 255]
    V = gather_latent_rows(pool, "bf16", bt[0], J)[:, :DV]
    np.testing.assert_allclose(out[0], np.broadcast_to(V.mean(axis=0), (8, DV)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], np.log(len(J)), rtol=0, atol=1e-12)


def test_single_entry_is_exact():
    pool = _pool(3, 2)
    bt = np.array([[1, 2, 0]])
    q = _q(1, 4, 3)
    idx = np.array([[77, -1, -1, -1]], dtype=np.int32)
    out, lse = sparse_mla_decode(q, pool, "bf16", bt, idx, np.array([150]), SCALE)
    K = gather_latent_rows(pool, "bf16", bt[0], [77])[0]
    qf = bf16_bits_to_float64(q[0])
    assert np.array_equal(out[0], np.broadcast_to(K[:DV], (4, DV)))
    for h in range(4):
        want = SCALE * math.fsum(float(a) * float(b) for a, b in zip(qf[h], K))
        assert abs(lse[0, h] - want) < 1e-9


def test_two_entries_closed_form():
    """q picks out one dim; the two K rows differ there by a set gap."""
    K = np.zeros((2, DQK))
    K[0, 3], K[1, 3] = 2.0, 0.5
    K[:, 10:20] = np.arange(20).reshape(2, 10)
    q = np.zeros((1, DQK))
    q[0, 3] = 1.0 / SCALE
    out, lse = sparse_mla_rows(q, K, SCALE)
    d = 1.5
    s1, s2 = 1.0 / (1.0 + math.exp(-d)), 1.0 / (1.0 + math.exp(d))
    np.testing.assert_allclose(out[0], s1 * K[0, :DV] + s2 * K[1, :DV], rtol=1e-14, atol=1e-14)
    assert abs(lse[0] - (2.0 + math.log(1.0 + math.exp(-d)))) < 1e-12


def _fsum_attention(q, K, scale):
    """Textbook softmax attention with compensated scalar sums."""
    H, n = len(q), len(K)
    out = [[0.0] * DV for _ in range(H)]
    lse = [0.0] * H
    for h in range(H):
        s = [scale * math.fsum(q[h][d] * K[j][d] for d in range(DQK)) for j in range(n)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = math.fsum(e)
        lse[h] = m + math.log(z)
        for c in range(DV):
            out[h][c] = math.fsum(e[j] * K[j][c] for j in range(n)) / z
    return out, lse


def test_matches_scalar_textbook_softmax():
    pool = _pool(2, 5)
    bt = np.array([[1, 0]])
    q = _q(1, 2, 6)
    idx = np.array([[1, 4, 66, 100, 127, -1, -1, -1]], dtype=np.int32)
    out, lse = sparse_mla_decode(q, pool, "bf16", bt, idx, np.array([128]), SCALE)
    K = gather_latent_rows(pool, "bf16", bt[0], [1, 4, 66, 100, 127]).tolist()
    want_out, want_lse = _fsum_attention(bf16_bits_to_float64(q[0]).tolist(), K, SCALE)
    np.testing.assert_allclose(out[0], np.array(want_out), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[0], np.array(want_lse), rtol=1e-12, atol=1e-12)


def test_dense_selection_matches_sdpa():
    """k >= context, idx = every position: plain dense attention."""
    ctx, H = 150, 4
    pool = _pool(3, 7)
    bt = np.array([[2, 0, 1]])
    q = _q(1, H, 8)
    idx = np.concatenate([np.arange(ctx), -np.ones(42)]).astype(np.int32)[None]
    out, lse = sparse_mla_decode(q, pool, "bf16", bt, idx, np.array([ctx]), SCALE)
    K = torch.from_numpy(gather_latent_rows(pool, "bf16", bt[0], np.arange(ctx)))
    qt = torch.from_numpy(bf16_bits_to_float64(q[0]))
    ref = F.scaled_dot_product_attention(qt[None, :, None, :],
                                         K[None, None].expand(1, H, ctx, DQK),
                                         K[None, None, :, :DV].expand(1, H, ctx, DV),
                                         scale=SCALE)
    np.testing.assert_allclose(out[0], ref[0, :, 0].numpy(), rtol=1e-10, atol=1e-12)
    ref_lse = torch.logsumexp(SCALE * (qt @ K.T), dim=-1)
    np.testing.assert_allclose(lse[0], ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_page_permutation_invariance():
    pool = _pool(6, 9)
    bt = np.array([[4, 1, 5, 0, 2, 3]])
    q = _q(1, 3, 10)
    idx = np.array([[3, 64, 65, 200, 383, -1]], dtype=np.int32)
    out, lse = sparse_mla_decode(q, pool, "bf16", bt, idx, np.array([384]), SCALE)
    perm = np.array([2, 5, 0, 4, 3, 1])           # new page id of old page p = perm[p]
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    out2, lse2 = sparse_mla_decode(q, pool2, "bf16", perm[bt], idx, np.array([384]), SCALE)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_invalid_entries_are_skipped_and_empty_row():
    pool = _pool(2, 11)
    bt = np.array([[1, 0], [0, 1]])
    q = _q(2, 2, 12)
    idx = np.array([[5, 90, 100, 127, -1, 128, 5000],     # 100,127 >= len 96; 128 has no page
                    [-1, -1, -1, -1, -1, -1, -1]], dtype=np.int32)
    out, lse = sparse_mla_decode(q, pool, "bf16", bt, idx, np.array([96, 128]), SCALE)
    ref, ref_lse = sparse_mla_decode(q, pool, "bf16", bt, np.array([[5, 90]], np.int32),
                                     np.array([96]), SCALE, rows=[0])
    assert np.array_equal(out[0], ref[0]) and np.array_equal(lse[0], ref_lse[0])
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


def test_prefill_uses_row_req_block_table():
    pool = _pool(4, 13)
    bt = np.array([[0, 1], [2, 3]])
    q = _q(3, 2, 14)
    idx = np.array([[0, 1, 70], [0, 1, 70], [3, -1, -1]], dtype=np.int32)
    lens = np.array([100, 100, 4])
    out, lse = sparse_mla_prefill(q, pool, "bf16", bt, np.array([1, 0, 1]), idx, lens, SCALE)
    a, la = sparse_mla_decode(q[[0]], pool, "bf16", bt[[1]], idx[[0]], lens[[0]], SCALE)
    b, lb = sparse_mla_decode(q[[1]], pool, "bf16", bt[[0]], idx[[1]], lens[[1]], SCALE)
    assert np.array_equal(out[0], a[0]) and np.array_equal(out[1], b[0])
    assert np.array_equal(lse[0], la[0]) and np.array_equal(lse[1], lb[0])


def test_fp8_rows_decode_layout():
    """656-byte row: 512 E4M3 codes, 4 float32 group scales, 64 bf16 rope."""
    row = np.zeros((1, 1, 656), dtype=np.uint8)
    row[0, 0, :512] = 0x38                                # e4m3 1.0
    row[0, 0, 512:528] = np.array([0.5, 2.0, 4.0, 8.0], "<f4").view(np.uint8)
    row[0, 0, 528:656] = np.full(64, 0x3F80, "<u2").view(np.uint8)   # bf16 1.0
    K = gather_latent_rows(row, "fp8", np.array([0]), [0])[0]
    assert K[:128].tolist() == [0.5] * 128 and K[128:256].tolist() == [2.0] * 128
    assert K[256:384].tolist() == [4.0] * 128 and K[384:512].tolist() == [8.0] * 128
    assert K[512:].tolist() == [1.0] * 64


def test_fp8_generator_roundtrip_within_e4m3_step():
    """The generator's packing dequantises back to within half an E4M3 step."""
    from synthetic import quantize_fp8_rows
    g = torch.Generator().manual_seed(21)
    x = torch.randn((8, DQK), generator=g)
    rope = x[:, 512:].to(torch.bfloat16)
    raw = quantize_fp8_rows(x[:, :512], rope).numpy().reshape(8, 1, 656)
    bt = np.arange(8)
    K = gather_latent_rows(raw, "fp8", bt, np.arange(8) * PAGE)
    err = np.abs(K[:, :512] - x[:, :512].double().numpy())
    amax = x[:, :512].abs().reshape(8, 4, 128).amax(-1).repeat_interleave(128, -1).double().numpy()
    assert np.all(err <= amax / 448.0 * 16.0 + 1e-12)      # half an ulp of the top binade (ulp 32)
    assert np.array_equal(K[:, 512:], rope.double().numpy())
