"""CPU oracle for the deterministic sparse top-k and sparse MLA attention path.

TEST INFRASTRUCTURE ONLY. This package is the slow, plain, obviously-correct
definition that the CUDA path is checked against. Only the test suite, the
smoke check in ``__graft_entry__`` and the ``cpu_baseline`` / ``--impl
reference`` legs of ``bench.py`` may import it. The product path (the C-ABI
library and its Python binding) never imports, calls or links anything here,
and this package never imports the product path.

Everything is NumPy, computed in float64 where floating point is involved.
Each function cites the passage of the source pages it follows:

* "[DeepSeek-V4][Preview][DO NOT MERGE] Batch-invariant kernels for 0-diff RL"
  (vllm-project/vllm PR 54955), sections "Deterministic sparse top-k" and
  "Sparse MLA and FlashMLA".
* "[Bugfix] Make DSV4 sparse MLA work end-to-end for plain decode, MTP, and
  DSpark" (vllm-project/vllm PR 51538), section "What is fixed".
* "[JJ] Preallocate DeepSeek V4 padded-query output" (local-inference-lab/vllm
  PR 671), section "Operation contract" (caller-owned outputs).
* "[SM120] Sync DS4 with upstream main + validated perf backports" (jasl/vllm
  PR 47), which names the indexer's MQA logits; their formula is the
  DeepSeek-V3.2-Exp lightning indexer (outside the pages; see indexer.py).

Where the pages are silent the oracle takes one plain reading and states it
in the function's docstring.

Parity status: every public function here is pinned by ``tests/test_oracle_*``
against brute force, closed forms, hand-built tie tables, library routines on
special cases, or identities (uniform scores give the mean of V; a single
valid entry returns its V row exactly).
"""

from .topk import row_length, topk_per_row, topk_rank_bruteforce  # noqa: F401
from .fp8 import (  # noqa: F401
    e4m3_to_float64,
    bf16_bits_to_float64,
    e4m3_encode,
    quantize_latent_rows,
    kv_cache_write,
)
from .indexer import indexer_logits, indexer_row_length  # noqa: F401
from .attention import (  # noqa: F401
    gather_latent_rows,
    sparse_mla_rows,
    sparse_mla_decode,
    sparse_mla_prefill,
    sparse_mla_rows_sink,
    sparse_mla_decode_swa,
)
