"""GPU parity of ds_topk_per_row against the oracle: bit-exact indices.

Covers the named workloads (tiny decode with ties, the TP2-shaped and TP1
decode batches, sampled rows of the chunked-prefill score matrix), and the
edge cases of "Deterministic sparse top-k" (PR 54955) and "What is fixed"
(PR 51538): heavy ties, signed zeros, NaN and -inf, negative and oversized
lengths, offsets that break 16-byte alignment, rows shorter than, equal to
and one longer than k, and empty batches. Row widths and batch sizes are
chosen so that every kernel behind ds_topk_per_row runs: whole rows in
shared memory (16 or more rows of width <= 32768), the streaming grid (256
or more rows of up to 65536), the grid kernel that spreads every row over
the whole GPU (the remaining shapes of up to 1024 rows, 131072 wide and
2^24 scores, when a workspace is given) and a cluster per row (the same
shapes without a workspace).
"""

import numpy as np
import pytest
import torch

import oracle
from harness import ensure_built
from synthetic import workload_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def ds():
    return ensure_built()


def run(ds, scores, starts, ends, k, workspace=None):
    s = torch.as_tensor(scores, dtype=torch.float32).to(DEV).contiguous()
    a = torch.as_tensor(starts, dtype=torch.int32).to(DEV)
    b = torch.as_tensor(ends, dtype=torch.int32).to(DEV)
    got = ds.topk_per_row(s, a, b, k, workspace=workspace)
    torch.cuda.synchronize()
    return got.cpu().numpy()


def check(ds, scores, starts, ends, k):
    scores = np.asarray(scores, dtype=np.float32)
    got = run(ds, scores, starts, ends, k)
    want = oracle.topk_per_row(scores, np.asarray(starts), np.asarray(ends), k)
    assert np.array_equal(got, want), (
        f"rows differ: {np.nonzero((got != want).any(1))[0][:10].tolist()}")
    return got


@pytest.mark.parametrize("name", ["tiny_decode", "tp2_decode"])
def test_named_workloads_exact(ds, name):
    c = workload_case(name, device="cpu")
    check(ds, c.np_scores(), c.np_int("row_starts"), c.np_int("row_ends"), c.k)


def test_tp1_decode_scores_exact(ds):
    c = workload_case("tp1_fp8_decode", device="cuda")
    got = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k).cpu().numpy()
    want = oracle.topk_per_row(c.np_scores(), c.np_int("row_starts"), c.np_int("row_ends"), c.k)
    assert np.array_equal(got, want)


def test_chunked_prefill_scores_sampled(ds):
    # 4096 x 65536 fp32 scores (1 GiB) on the device; the oracle checks a
    # seeded sample of rows, the kernel runs on the full matrix.
    T, ctx = 4096, 65536
    g = torch.Generator(device="cuda").manual_seed(3)
    pos = torch.arange(ctx - T, ctx, dtype=torch.int32, device=DEV)
    scores = torch.randn((T, ctx), generator=g, device=DEV)
    col = torch.arange(ctx, device=DEV)[None, :]
    scores = torch.where(col < (pos + 1)[:, None], scores, torch.full_like(scores, float("nan")))
    starts = torch.zeros(T, dtype=torch.int32, device=DEV)
    idx = ds.topk_per_row(scores, starts, pos + 1, 2048).cpu().numpy()
    rows = np.random.default_rng(0).choice(T, 24, replace=False).tolist() + [0, T - 1]
    sub = scores[rows].cpu().numpy()
    want = oracle.topk_per_row(sub, np.zeros(len(rows)), (pos + 1).cpu().numpy()[rows], 2048)
    assert np.array_equal(idx[rows], want)
    # Properties that hold for every row: ascending, in range, exactly k.
    assert (idx >= 0).all() and (np.diff(idx, axis=1) > 0).all()
    assert (idx < (pos + 1).cpu().numpy()[:, None]).all()


def test_heavy_ties_integer_scores(ds):
    rng = np.random.default_rng(1)
    for L, k in [(100, 10), (5000, 2048), (32768, 2048), (70000, 2048)]:
        s = rng.integers(0, 8, (3, L)).astype(np.float32)
        check(ds, s, [0, 0, 0], [L, L, L], k)


def test_all_equal_and_two_values(ds):
    s = np.full((2, 9000), 1.5, dtype=np.float32)
    s[1, ::3] = 2.5
    got = check(ds, s, [0, 0], [9000, 9000], 2048)
    assert got[0].tolist() == list(range(2048))


def test_special_values(ds):
    rng = np.random.default_rng(2)
    L = 6000
    s = rng.choice(np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan], np.float32), (4, L))
    check(ds, s, [0] * 4, [L] * 4, 700)
    check(ds, s, [0] * 4, [L] * 4, 64)
    s2 = np.full((1, 3000), np.nan, np.float32)
    s2[0, 1000:1010] = -np.inf
    check(ds, s2, [0], [3000], 2048)


def test_lengths_clamped_and_padded(ds):
    rng = np.random.default_rng(3)
    stride = 5000
    s = rng.standard_normal((8, stride)).astype(np.float32)
    starts = [0, 10, 0, 100, 4000, 5000, -3, 7]
    ends = [-1, 5, 2048, 2149, 9999, 5001, 100, 2056]
    got = check(ds, s, starts, ends, 2048)
    assert (got[0] == -1).all() and (got[1] == -1).all() and (got[5] == -1).all()
    assert got[2].tolist() == list(range(2048))
    assert (got[4][1000:] == -1).all()


def test_k_boundaries(ds):
    rng = np.random.default_rng(4)
    for k in [1, 2, 63, 64, 2047, 2048, 2049, 4096]:
        for L in [k - 1, k, k + 1, 3 * k + 5]:
            if L <= 0:
                continue
            s = np.round(rng.standard_normal((2, L)) * 8).astype(np.float32) / 8
            check(ds, s, [0, 0], [L, L], k)


def test_unaligned_offsets_and_strides(ds):
    rng = np.random.default_rng(5)
    for stride in [4097, 10001]:
        s = (np.round(rng.standard_normal((6, stride)) * 4) / 4).astype(np.float32)
        starts = [1, 2, 3, 5, 0, 17]
        ends = [stride, stride - 1, 4000, stride, 3001, 9000]
        check(ds, s, starts, ends, 512)


def test_offset_invariance(ds):
    rng = np.random.default_rng(6)
    base = (np.round(rng.standard_normal(20000) * 8) / 8).astype(np.float32)
    ref = run(ds, base[None], [0], [20000], 2048)[0]
    for off in [1, 3, 64, 1000]:
        s = np.full((1, 20000 + off), np.nan, np.float32)
        s[0, off:] = base
        assert np.array_equal(run(ds, s, [off], [20000 + off], 2048)[0], ref)


def test_batch_invariance_of_indices(ds):
    from synthetic import invariance_batch
    ref = None
    for B in [1, 7, 64, 256]:
        slot = (B * 5) // 7
        c = invariance_batch(B, slot, device="cuda")
        idx = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)[slot].cpu().numpy()
        if ref is None:
            ref = idx
            want = oracle.topk_per_row(c.scores[slot:slot + 1].cpu().numpy(), [0],
                                       [c.meta["ctx"][slot]], c.k)[0]
            assert np.array_equal(ref, want)
        assert np.array_equal(idx, ref), B


def test_empty_batch(ds):
    s = torch.zeros((0, 128), dtype=torch.float32, device=DEV)
    z = torch.zeros(0, dtype=torch.int32, device=DEV)
    assert ds.topk_per_row(s, z, z, 16).shape == (0, 16)


def test_run_to_run_deterministic(ds):
    c = workload_case("tp2_decode", device="cuda")
    a = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    b = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    assert torch.equal(a, b)


def _mixed_rows(rng, R, stride, k):
    """R rows cycling through the cases that stress each refinement pass."""
    s = np.empty((R, stride), np.float32)
    starts, ends = np.zeros(R, np.int64), np.full(R, stride, np.int64)
    specials = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan], np.float32)
    for r in range(R):
        case = r % 9
        if case == 0:
            s[r] = np.round(rng.standard_normal(stride) * 8) / 8
        elif case == 1:  # eight values: the threshold bucket is unresolved at 32 bits
            s[r] = rng.integers(0, 8, stride)
        elif case == 2:
            s[r] = 1.5
        elif case == 3:
            s[r] = rng.choice(specials, stride)
        elif case == 4:  # every score shares its top 16 key bits
            s[r] = 1.0 + rng.random(stride) * 2.0 ** -7
        elif case == 5:  # shared top 16 bits, ties in the low 8 bits
            s[r] = 1.0 + rng.integers(0, 64, stride) * 2.0 ** -14
        elif case == 6:  # row no longer than k: no score is read
            s[r] = rng.standard_normal(stride)
            ends[r] = int(rng.integers(0, k + 1))
        elif case == 7:  # odd start and end
            s[r] = rng.standard_normal(stride)
            starts[r] = int(rng.integers(1, 40))
            ends[r] = stride - int(rng.integers(0, 40))
        else:
            s[r] = rng.standard_normal(stride) * 1e-3
    return s, starts, ends


@pytest.mark.parametrize("stride,k", [(20000, 2048), (20001, 700), (9000, 64), (32768, 2048),
                                      (40001, 2048), (50000, 700)])
def test_many_rows_mixed_cases_exact(ds, stride, k):
    # Rows of up to 32K scores are held whole in shared memory; batches of at
    # least 256 longer rows (up to 64K) are streamed by a persistent grid.
    rng = np.random.default_rng(stride + k)
    s, a, b = _mixed_rows(rng, 288, stride, k)
    check(ds, s, a, b, k)


def test_many_rows_longest_rows_sampled(ds):
    rng = np.random.default_rng(11)
    R, stride, k = 256, 65536, 2048
    s, a, b = _mixed_rows(rng, R, stride, k)
    got = run(ds, s, a, b, k)
    rows = list(range(18)) + rng.choice(R, 12, replace=False).tolist()
    want = oracle.topk_per_row(s[rows], a[rows], b[rows], k)
    assert np.array_equal(got[rows], want)


def test_kernel_choice_never_changes_indices(ds):
    # The same rows alone in a 40000-wide matrix (a cluster per row), in a
    # batch of 300 such rows (the streaming kernel) and in a 30000-wide
    # matrix (whole row in shared memory) give identical indices.
    rng = np.random.default_rng(12)
    s, a, b = _mixed_rows(rng, 300, 30000, 2048)
    wide = np.full((300, 40000), np.nan, np.float32)
    wide[:, :30000] = s
    narrow = run(ds, s, a, b, 2048)
    big = run(ds, wide, a, b, 2048)
    assert np.array_equal(big, narrow)
    for r in [0, 1, 3, 4, 5, 7, 8, 299]:
        one = run(ds, wide[r:r + 1], a[r:r + 1], b[r:r + 1], 2048)[0]
        assert np.array_equal(one, big[r]), r


@pytest.mark.parametrize("k", [2048, 8192, 16384])
def test_rows_wider_than_128k_exact(ds, k):
    # Rows wider than 131072 scores take the kernel whose histogram passes
    # read global memory; every refinement case of _mixed_rows on 200003-wide
    # rows.
    rng = np.random.default_rng(k + 1)
    s, a, b = _mixed_rows(rng, 9, 200003, k)
    check(ds, s, a, b, k)


@pytest.mark.parametrize("k", [8192, 16384])
@pytest.mark.parametrize("rows,stride", [(16, 32768), (256, 40000), (8, 100000)])
def test_large_k_on_every_kernel_exact(ds, rows, stride, k):
    # k above 4096 on the whole-row kernel (16 rows of 32K), the streaming
    # grid (256 rows of 40000) and the cluster kernel (8 rows of 100000).
    rng = np.random.default_rng(rows * 7 + k)
    s, a, b = _mixed_rows(rng, rows, stride, k)
    check(ds, s, a, b, k)


def _grid_run(ds, s, a, b, k, base_offset=0):
    """Runs the grid kernel with an explicit workspace of stale contents,
    checking its error word afterwards. base_offset shifts the score matrix
    by that many floats from a 16-byte boundary; such a matrix takes the
    kernels that need no workspace (the grid kernel's copies need a 16-byte
    aligned start)."""
    R, stride = s.shape
    need = ds.topk_workspace_size(R, stride, k)
    assert need > 0, (R, stride)
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device=DEV)   # stale contents
    flat = torch.empty(R * stride + 4, dtype=torch.float32, device=DEV)
    dev_s = flat[base_offset:base_offset + R * stride].view(R, stride)
    dev_s.copy_(torch.as_tensor(s))
    got = ds.topk_per_row(dev_s, torch.as_tensor(a, dtype=torch.int32).to(DEV),
                          torch.as_tensor(b, dtype=torch.int32).to(DEV), k, workspace=ws)
    torch.cuda.synchronize()
    if base_offset % 4 == 0:
        assert int(ws[8:12].view(torch.int32).item()) == 0, "a grid wait gave up"
    return got.cpu().numpy()


@pytest.mark.parametrize("rows,stride,k", [(9, 40001, 2048), (8, 100000, 700), (5, 131072, 2048),
                                           (12, 33000, 64), (15, 32768, 2048), (1, 16384, 2048),
                                           (40, 70000, 2048), (3, 131072, 16384)])
def test_grid_kernel_exact(ds, rows, stride, k):
    # Every refinement case of _mixed_rows, plus ascending and descending rows
    # and a constant row: lists far longer than one resolve tile.
    rng = np.random.default_rng(rows * 13 + stride + k)
    s, a, b = _mixed_rows(rng, rows, stride, k)
    s[0] = np.arange(stride, dtype=np.float32)
    if rows > 2:
        s[2] = -np.arange(stride, dtype=np.float32)
        a[2], b[2] = 3, stride - 5
    got = _grid_run(ds, s, a, b, k)
    want = oracle.topk_per_row(s, a, b, k)
    assert np.array_equal(got, want), np.nonzero((got != want).any(1))[0][:10].tolist()


@pytest.mark.parametrize("base_offset", [1, 2, 3])
def test_grid_shape_unaligned_score_pointer(ds, base_offset):
    # A score matrix starting 4, 8 or 12 bytes past a 16-byte boundary, with
    # a workspace given: the call takes a kernel that reads the scores with
    # plain loads, and the indices are the same.
    rng = np.random.default_rng(base_offset)
    s, a, b = _mixed_rows(rng, 9, 50001, 2048)
    got = _grid_run(ds, s, a, b, 2048, base_offset=base_offset)
    assert np.array_equal(got, oracle.topk_per_row(s, a, b, 2048))


def test_grid_kernel_equals_workspace_free_kernels(ds):
    # The TP1 batch shape (128 rows of up to 131072 scores) with and without a
    # workspace: the grid kernel and the cluster kernel give identical indices,
    # and the grid kernel repeats bit for bit.
    c = workload_case("tp1_fp8_decode", device="cuda")
    assert ds.topk_workspace_size(c.scores.shape[0], c.scores.shape[1], c.k) > 0
    grid1 = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    grid2 = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k)
    free = ds.topk_per_row(c.scores, c.row_starts, c.row_ends, c.k, workspace=False)
    assert torch.equal(grid1, grid2)
    assert torch.equal(grid1, free)


def test_grid_kernel_batch_of_one_row_in_many(ds):
    # One row alone and inside batches of 7 and 64 neighbours of random
    # lengths: bitwise the same indices (the rest of the batch changes which
    # CTAs hold which segments of the row, never the result).
    rng = np.random.default_rng(21)
    stride, k = 65536, 2048
    row = (np.round(rng.standard_normal(stride) * 4) / 4).astype(np.float32)
    ref = _grid_run(ds, row[None], [0], [60001], k)[0]
    assert np.array_equal(ref, oracle.topk_per_row(row[None], [0], [60001], k)[0])
    for B in [7, 64, 255]:
        s = rng.standard_normal((B, stride)).astype(np.float32)
        slot = B // 2
        s[slot] = row
        a = np.zeros(B, np.int64)
        b = rng.integers(0, stride + 1, B)
        b[slot] = 60001
        got = _grid_run(ds, s, a, b, k)
        assert np.array_equal(got[slot], ref), B


def test_grid_kernel_bound_edge_cases(ds):
    # Rows built against the bound each CTA takes from the first segment of
    # its part of a row: a first segment of NaN (the bound drops to the
    # bottom: everything after it is listed), the largest scores at the end
    # of the row (early bounds low, lists long but complete), +inf first and
    # falling after (the bound lies above most of the top k, so the row is
    # taken whole), every score tied, and a row one longer than k.
    rng = np.random.default_rng(33)
    R, stride, k = 10, 100000, 2048
    s = rng.standard_normal((R, stride)).astype(np.float32)
    a = np.zeros(R, np.int64)
    b = np.full(R, stride, np.int64)
    s[0, :9000] = np.nan
    s[1] = np.sort(s[1])                       # ascending: the top k is the row's end
    s[2, :3000] = np.inf
    s[2, 3000:] = -np.sort(-s[2, 3000:])       # descending after the infinities
    s[3] = 7.0                                 # all tied
    b[4] = k + 1
    s[5, ::2] = np.nan                         # half NaN
    s[6] = np.where(rng.random(stride) < 0.5, 0.0, -0.0).astype(np.float32)
    s[6, 50000:50010] = 1.0
    s[7, :8192] = -np.inf
    a[8], b[8] = 1, stride - 1                 # odd start and end
    s[9, -5000:] = 100.0 + rng.standard_normal(5000).astype(np.float32)
    got = _grid_run(ds, s, a, b, k)
    want = oracle.topk_per_row(s, a, b, k)
    assert np.array_equal(got, want), np.nonzero((got != want).any(1))[0][:10].tolist()


def test_grid_kernel_in_a_cuda_graph(ds):
    # The cooperative launch and the workspace header's zero fill capture into
    # a CUDA graph; replays on new scores in the same buffers give the
    # oracle's indices each time.
    rng = np.random.default_rng(41)
    R, stride, k = 24, 90000, 2048
    s0, a, b = _mixed_rows(rng, R, stride, k)
    scores = torch.as_tensor(s0).to(DEV)
    starts = torch.as_tensor(a, dtype=torch.int32).to(DEV)
    ends = torch.as_tensor(b, dtype=torch.int32).to(DEV)
    ws = torch.empty(ds.topk_workspace_size(R, stride, k), dtype=torch.uint8, device=DEV)
    idx = torch.empty((R, k), dtype=torch.int32, device=DEV)
    side = torch.cuda.Stream(DEV)
    with torch.cuda.stream(side):
        ds.topk_per_row(scores, starts, ends, k, idx_out=idx, workspace=ws)   # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        ds.topk_per_row(scores, starts, ends, k, idx_out=idx, workspace=ws)
    for it in range(3):
        s = rng.standard_normal((R, stride)).astype(np.float32) if it else s0
        scores.copy_(torch.as_tensor(s))
        g.replay()
        torch.cuda.synchronize()
        assert int(ws[8:12].view(torch.int32).item()) == 0
        assert np.array_equal(idx.cpu().numpy(), oracle.topk_per_row(s, a, b, k)), it


def test_grid_kernel_k1_and_short_workspace(ds):
    rng = np.random.default_rng(42)
    R, stride = 6, 70000
    s, a, b = _mixed_rows(rng, R, stride, 1)
    assert np.array_equal(_grid_run(ds, s, a, b, 1), oracle.topk_per_row(s, a, b, 1))
    # One byte short of the grid kernel's workspace: a workspace-free kernel
    # runs instead, with the same indices.
    k = 700
    s, a, b = _mixed_rows(rng, R, stride, k)
    need = ds.topk_workspace_size(R, stride, k)
    short = torch.empty(need - 1, dtype=torch.uint8, device=DEV)
    got = run(ds, s, a, b, k, workspace=short)
    assert np.array_equal(got, oracle.topk_per_row(s, a, b, k))


def test_grid_kernel_random_shapes(ds):
    # Seeded random shapes, bounds and score distributions (normal, few
    # distinct integers, special values, eighths with NaN holes, sorted rows,
    # a narrow band of shared high bits), each against the oracle.
    rng = np.random.default_rng(2027)
    specials = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan], np.float32)
    done = 0
    while done < 24:
        R = int(rng.choice([1, 3, 8, 15, 40, 100]))
        stride = int(rng.integers(max(8192 // R + 1, 64), 131073))
        if R * stride > (1 << 20):
            stride = (1 << 20) // R
        k = int(rng.choice([1, 7, 100, 700, 2048, 2049, 8192]))
        if ds.topk_workspace_size(R, stride, k) == 0:
            continue
        kind = done % 6
        if kind == 0:
            s = rng.standard_normal((R, stride)).astype(np.float32)
        elif kind == 1:
            s = rng.integers(0, int(rng.integers(1, 50)), (R, stride)).astype(np.float32)
        elif kind == 2:
            s = rng.choice(specials, (R, stride))
        elif kind == 3:
            s = (np.round(rng.standard_normal((R, stride)) * 8) / 8).astype(np.float32)
            s[rng.random((R, stride)) < 0.1] = np.nan
        elif kind == 4:
            s = np.sort(rng.standard_normal((R, stride)).astype(np.float32), axis=1)
            if rng.random() < 0.5:
                s = s[:, ::-1].copy()
        else:
            s = (1.0 + rng.random((R, stride)) * 2.0 ** -int(rng.integers(5, 20))).astype(np.float32)
        a = rng.integers(-3, stride // 3, R)
        b = a + rng.integers(-5, stride + 10, R)
        got = _grid_run(ds, s, a, b, k)
        assert np.array_equal(got, oracle.topk_per_row(s, a, b, k)), (R, stride, k, kind)
        done += 1
