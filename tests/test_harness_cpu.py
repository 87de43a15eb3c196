"""The parity check itself, on the CPU: what it accepts and what it rejects.

Outputs of the decode shape used by the benchmarks (top-k 2048 over
contexts of several thousand) are about N(0, 1/750) per element, so the
per-element bound (atol 2e-2 + 1e-2 |ref|) alone is about half of a typical
value. The harness adds a per-(row, head) bound on max |err| / RMS(ref).
These tests plant the mistakes in a copy of the oracle's own output: an 8 %
scaling error passes the per-element bound but not the scale-aware one, and
a plain bf16 rounding of the exact result passes both.
"""

import numpy as np
import pytest
import torch

import oracle
from harness import ATOL, RTOL, assert_close, q_bits, kv_np
from synthetic import decode_case


@pytest.fixture(scope="module")
def exact():
    c = decode_case("harness", [6000, 4096, 2500], 16, 2048, "bf16", seed=41, device="cpu")
    idx = oracle.topk_per_row(c.np_scores(), c.np_int("row_starts"), c.np_int("row_ends"), c.k)
    out, lse = oracle.sparse_mla_decode(q_bits(c.q), kv_np(c.kv_pages, "bf16"), "bf16",
                                        c.block_table.numpy(), idx, c.lens.numpy(), c.scale)
    return out, lse


def test_bf16_rounding_of_the_exact_result_passes(exact):
    out, lse = exact
    got = torch.from_numpy(out).to(torch.bfloat16)
    assert_close(got, torch.from_numpy(lse.astype(np.float32)), out, lse, "bf16", "rounded")


def test_eight_percent_scaling_error_is_caught(exact):
    out, lse = exact
    wrong = out * 1.08
    # The per-element bound alone would let it through ...
    assert np.all(np.abs(wrong - out) <= ATOL["bf16"] + RTOL * np.abs(out))
    # ... the scale-aware one does not.
    with pytest.raises(AssertionError, match="RMS"):
        assert_close(torch.from_numpy(wrong).to(torch.bfloat16),
                     torch.from_numpy(lse.astype(np.float32)), out, lse, "bf16", "scaled")
