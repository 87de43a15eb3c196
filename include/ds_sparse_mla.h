/*
 * ds_sparse_mla.h -- C ABI of the GB300 (sm_103a) deterministic sparse top-k
 * and sparse MLA attention library (libds_sparse_mla.so).
 *
 * What the library computes
 * -------------------------
 * The two steps of DeepSeek-V4-style sparse MLA described on the pages
 * "[DeepSeek-V4][Preview][DO NOT MERGE] Batch-invariant kernels for 0-diff
 * RL" (vllm-project/vllm PR 54955), sections "Deterministic sparse top-k" and
 * "Sparse MLA and FlashMLA", and "[Bugfix] Make DSV4 sparse MLA work
 * end-to-end for plain decode, MTP, and DSpark" (vllm-project/vllm PR 51538),
 * section "What is fixed":
 *
 *   1. ds_topk_per_row: for every row, the k positions with the largest
 *      indexer scores under the total order (score descending, position
 *      ascending), written in ascending position order, -1 in unused slots.
 *   2. ds_sparse_mla_decode / ds_sparse_mla_prefill: gather the selected
 *      entries of a paged latent KV cache (64 entries per page, 576 = 512
 *      latent + 64 rope dims, one latent row shared by every head) and
 *      compute out = softmax(scale * q K^T) V with V = the first 512 dims of
 *      the same rows, plus lse = ln(sum exp(scale * q K^T)).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer (cudaMalloc'd or otherwise
 *    device-accessible) unless stated otherwise. Nothing is allocated or
 *    freed inside; outputs and workspaces are owned by the caller, as in the
 *    caller-owned-output contract of "[JJ] Preallocate DeepSeek V4
 *    padded-query output" (local-inference-lab/vllm PR 671, section
 *    "Operation contract").
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Every call only enqueues work on it and never synchronises the
 *    host, so calls may be captured into a CUDA graph.
 *  - Arguments are validated on the host before anything is launched.
 *    Unsupported shapes are a hard error (PR 54955: "missing kernel support
 *    is a hard error rather than a silent fallback"); ds_last_error() names
 *    the offending parameter and the allowed set (PR 51538, "SM120 gate").
 *  - Row lengths are computed signed and clamped at 0 before any decision,
 *    so a negative length from a padded request is an empty row, never a
 *    huge unsigned value (PR 51538, "What is fixed").
 *  - Offsets inside the kernels are 64-bit: tensors may exceed 2^31
 *    elements (PR 54955, the 64-bit offset fix).
 *  - Results never depend on the rest of the batch: every row's output is
 *    bit-identical whether it runs alone or inside any batch, because each
 *    row's work is split and reduced in an order fixed by k alone.
 *  - Return value: DS_OK, or a ds_status error code. Any code other than
 *    DS_OK or DS_ERR_CUDA means nothing was launched; DS_ERR_CUDA means a
 *    launch failed (cudaGetLastError() reported an error).
 */
#ifndef DS_SPARSE_MLA_H
#define DS_SPARSE_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DS_OK = 0,
  DS_ERR_NULL = 1,         /* a required pointer is NULL                      */
  DS_ERR_SHAPE = 2,        /* a size is negative or inconsistent              */
  DS_ERR_UNSUPPORTED = 3,  /* a size is outside the supported set             */
  DS_ERR_DTYPE = 4,        /* unknown kv_dtype                                */
  DS_ERR_ALIGN = 5,        /* a pointer is not aligned as required            */
  DS_ERR_WORKSPACE = 6,    /* workspace missing or smaller than required      */
  DS_ERR_CUDA = 7          /* the CUDA runtime reported an error at launch    */
} ds_status;

typedef enum {
  DS_KV_BF16 = 0,          /* kv row = 576 bfloat16 (1152 bytes)              */
  DS_KV_FP8_E4M3 = 1       /* kv row = 656 bytes, layout below                */
} ds_kv_dtype;

/*
 * FP8 KV row layout (656 bytes, 16-byte aligned): bytes [0, 512) are the
 * 512 latent dims as OCP FP8 E4M3 codes; bytes [512, 528) are four
 * little-endian float32 scales, one per 128-dim group (dims 0-127, 128-255,
 * 256-383, 384-511), kept contiguous as in the FP8 KV cache of
 * "MooreThreads/vllm-musa PR 178" (optimisation table, contiguous FP32 scale
 * groups); bytes [528, 656) are the 64 rope dims as bfloat16. A latent value
 * is code * scale of its group.
 */
#define DS_PAGE_BLOCK_SIZE 64
#define DS_D_QK 576
#define DS_D_V 512
#define DS_KV_ROW_BYTES_BF16 1152
#define DS_KV_ROW_BYTES_FP8 656
#define DS_INDEXER_HEAD_DIM 128

/* Device-side error bits ORed into *err_flag (when err_flag != NULL). */
#define DS_DEVERR_IDX 1      /* an idx entry other than -1 outside [0, lens[row]) */
#define DS_DEVERR_PAGE 2     /* a block-table slot beyond bt_stride, or a page id
                                outside [0, num_pages)                            */
#define DS_DEVERR_ROWREQ 4   /* prefill: row_req[t] outside [0, num_requests)     */
#define DS_DEVERR_TIMEOUT 8  /* an internal pipeline wait gave up (library bug)   */

/*
 * Message of the last error on the calling host thread ("" if none). The
 * string is thread-local and stays valid until the next call on this thread.
 */
const char* ds_last_error(void);

/*
 * 1 if (num_heads, topk, page_block_size, d_qk, d_v, kv_dtype) is a shape the
 * attention entry points accept, else 0 with ds_last_error() naming the first
 * parameter that missed and the values that are available. Lets a caller
 * validate a model configuration at init time instead of at its first decode
 * (PR 51538, "SM120 gate"). Supported: num_heads in {16, 32, 64, 128}; topk a
 * multiple of 64 in [64, 2048]; page_block_size 64; d_qk 576; d_v 512;
 * kv_dtype DS_KV_BF16 or DS_KV_FP8_E4M3.
 */
int ds_supported_config(int num_heads, int topk, int page_block_size, int d_qk, int d_v,
                        int kv_dtype);

/*
 * Workspace bytes that let ds_topk_per_row spread every row of this shape
 * over the whole GPU (the grid kernel), or 0 for shapes that another kernel
 * serves without one. Nonzero for batches of at most 256 rows of at most
 * 131072 scores (8192 to 2^24 scores in all) that are neither 16 or more rows
 * of at most 32768 nor 256 or more rows of at most 65536: 256 header bytes,
 * then 64 KiB of candidate list and 8 bytes of bookkeeping for each of the
 * ceil((row_stride + 255) / 8192) segments a row may have, per row. k does
 * not change it.
 */
size_t ds_topk_workspace_size(int64_t num_rows, int64_t row_stride, int k);

/*
 * Workspace bytes ds_sparse_mla_decode / ds_sparse_mla_prefill need for
 * num_rows query rows (decode requests or prefill tokens), num_heads heads
 * and top-k width k: the per-split partial results (the unnormalised output
 * rounded to bfloat16, the running maximum and sum in float32). The number
 * of splits is a function of k alone. Returns 0 for an unsupported shape.
 */
size_t ds_sparse_mla_workspace_size(int64_t num_rows, int num_heads, int k);

/*
 * Deterministic per-row top-k ("Deterministic sparse top-k", PR 54955; length
 * clamp and -1 padding from PR 51538, "What is fixed").
 *
 *  scores      float32, row-major [num_rows, row_stride]; 4-byte aligned.
 *  row_stride  elements between consecutive rows, 1 <= row_stride <= 2^28.
 *  num_rows    >= 0 (0 launches nothing).
 *  row_starts  int32 [num_rows]; row_ends int32 [num_rows]. Row b ranks the
 *              scores at positions [row_starts[b], row_starts[b] + L_b) with
 *              L_b = clamp(row_ends[b] - row_starts[b], 0,
 *                          row_stride - row_starts[b]),
 *              computed signed; a row_starts[b] outside [0, row_stride] gives
 *              L_b = 0.
 *  k           1 <= k <= 16384.
 *  idx_out     int32 [num_rows, k], written fully: the selected positions
 *              RELATIVE to row_starts[b], ascending, then -1 in slots
 *              [min(k, L_b), k). Rows with L_b <= k select every position.
 *
 * Order: larger score first; equal scores (-0.0 equals +0.0) by lower
 * position; NaN ranks below -inf and NaNs tie with one another. The selected
 * set is therefore unique and the output is bit-exact and independent of the
 * batch.
 *
 *  workspace   NULL, or 256-byte aligned device memory of workspace_bytes.
 *              With at least ds_topk_workspace_size() bytes (when that is
 *              nonzero) and scores 16-byte aligned, the grid kernel runs:
 *              one cooperative launch whose CTAs are all resident, preceded
 *              by a zero fill of the workspace's first 256 bytes (so its
 *              contents need no initialisation); otherwise a kernel that
 *              needs no workspace runs. The output is identical either way.
 *              After the grid kernel, the int32 at byte offset 8 of the
 *              workspace is 0; a nonzero value means one of its bounded
 *              waits gave up (not expected: the launch keeps every CTA
 *              resident) and idx_out is unspecified. Concurrent calls need
 *              separate workspaces.
 */
int ds_topk_per_row(const float* scores, int64_t row_stride, int64_t num_rows,
                    const int32_t* row_starts, const int32_t* row_ends, int k,
                    int32_t* idx_out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Sparse MLA decode over a paged latent KV cache ("Sparse MLA and FlashMLA",
 * PR 54955: decode gathers the selected KV and runs sparse attention; slot
 * arithmetic slot = block_id * block_size + offset from PR 51538).
 *
 *  q            bfloat16 [num_rows, num_heads, 576], 16-byte aligned.
 *  kv_pages     DS_KV_BF16: bfloat16 [num_pages, 64, 576];
 *               DS_KV_FP8_E4M3: uint8 [num_pages, 64, 656]. 16-byte aligned.
 *  num_pages    >= 1.
 *  block_table  int32 [num_rows, bt_stride]: page id of each 64-position
 *               block of row b's context.
 *  idx          int32 [num_rows, k]: context positions to attend to (the
 *               output of ds_topk_per_row); -1 entries are skipped.
 *  lens         int32 [num_rows]: context length of each row.
 *  scale        softmax scale applied to q.K (e.g. 1/sqrt(576)).
 *  out          bfloat16 [num_rows, num_heads, 512], 16-byte aligned.
 *  lse          float32 [num_rows, num_heads]: natural-log sum of
 *               exp(scale * q.K) over the valid entries (-inf if none).
 *  workspace    >= ds_sparse_mla_workspace_size(num_rows, num_heads, k)
 *               bytes, 256-byte aligned; contents need no initialisation.
 *  err_flag     optional int32 device word (NULL = no report). Entries with
 *               an idx outside [0, lens[b]) (other than -1), or whose page
 *               lookup misses, are skipped and a DS_DEVERR_* bit is ORed in;
 *               the kernels never trap.
 *
 * Entry j of row b is valid iff 0 <= idx[b,j] < lens[b], idx[b,j]/64 <
 * bt_stride and the page id lies in [0, num_pages). A row with no valid entry
 * gives out = 0 and lse = -inf.
 */
int ds_sparse_mla_decode(const void* q, const void* kv_pages, int kv_dtype, int64_t num_pages,
                         const int32_t* block_table, int64_t bt_stride,
                         const int32_t* idx, const int32_t* lens,
                         int64_t num_rows, int num_heads, int k, float scale,
                         void* out, float* lse, void* workspace, size_t workspace_bytes,
                         int32_t* err_flag, void* stream);

/*
 * Sparse MLA prefill: as decode, with one query row per token. Token t reads
 * block-table row row_req[t] (int32 [num_tokens], in [0, num_requests)) and
 * is computed on its own, never through a batch-level plan ("Batch-invariant
 * prefill chunks each request independently", PR 54955). block_table is
 * int32 [num_requests, bt_stride]; idx, lens, q, out and lse are indexed by
 * token. A row_req outside [0, num_requests) gives out = 0, lse = -inf and
 * sets DS_DEVERR_ROWREQ.
 */
int ds_sparse_mla_prefill(const void* q, const void* kv_pages, int kv_dtype, int64_t num_pages,
                          const int32_t* block_table, int64_t bt_stride, int64_t num_requests,
                          const int32_t* row_req, const int32_t* idx, const int32_t* lens,
                          int64_t num_tokens, int num_heads, int k, float scale,
                          void* out, float* lse, void* workspace, size_t workspace_bytes,
                          int32_t* err_flag, void* stream);

/*
 * Allocation-free variant of ds_sparse_mla_decode. The pages have no
 * counterpart to this entry point; it exists for callers that cannot provide
 * device scratch memory: code running under a memory manager that owns all
 * device memory, code in the middle of recording a CUDA graph (where a plain
 * cudaMalloc is not allowed), and loops that cannot afford cudaMalloc's
 * implicit device synchronisation.
 *
 * Arguments, results and errors are those of ds_sparse_mla_decode, minus the
 * workspace. The scratch is a built-in 32 MiB device array of this library
 * (each GPU holds it from the time the library's module is first loaded there
 * until the process exits). Calls whose ds_sparse_mla_workspace_size() exceeds
 * 32 MiB return DS_ERR_WORKSPACE with a message; nothing is launched. The call
 * itself performs no cudaMalloc/cudaFree or other allocation.
 *
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture. A
 * lookup that fails returns DS_ERR_CUDA and is not remembered: the next call
 * tries again.
 * Every call shares the one array, and each call overwrites what the
 * previous one left there: calls that can overlap on the GPU (on different
 * streams without ordering between them) race on it and must not be issued.
 */
int ds_sparse_mla_decode_noalloc(const void* q, const void* kv_pages, int kv_dtype,
                                 int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                                 const int32_t* idx, const int32_t* lens, int64_t num_rows,
                                 int num_heads, int k, float scale, void* out, float* lse,
                                 int32_t* err_flag, void* stream);

/*
 * Sparse MLA decode over the concatenation [top-k entries of the compressed
 * KV || sliding-window entries of the window KV], with per-head attention
 * sinks ("[DeepSeek-V4][Preview][DO NOT MERGE] Batch-invariant kernels for
 * 0-diff RL", section "Sparse MLA and FlashMLA": decode gathers compressed
 * and sliding-window KV and runs one sparse attention over both; attention
 * sinks keep -inf padding. "[Bugfix] Make DSV4 sparse MLA work end-to-end
 * ...", section "What is fixed": the window index list is padded to a
 * multiple of 64 entries).
 *
 * The first ten arguments and q, out, lse, workspace, err_flag and stream
 * are those of ds_sparse_mla_decode (k is the top-k width). The window:
 *  swa_pages        the window pool, same row format and kv_dtype as
 *                   kv_pages, 16-byte aligned; swa_num_pages >= 1.
 *  swa_block_table  int32 [num_rows, swa_bt_stride]: page id of each
 *                   64-position block of the row's window context.
 *  swa_idx          int32 [num_rows, swa_width]: window positions (-1 =
 *                   padding); an entry is valid iff 0 <= swa_idx < swa_lens[row]
 *                   and its page lookup hits, like a top-k entry.
 *  swa_lens         int32 [num_rows].
 *  swa_width        0 (no window; the window arguments may be NULL) or a
 *                   multiple of 64 in [64, 512].
 *  attn_sink        optional float32 [num_heads] (NULL = no sinks): the sink
 *                   logit of each head, in the units of scale * q.K (natural
 *                   log). It joins the softmax denominator with no value row:
 *                   out = sum_j exp(S_j) V_j / (sum_j exp(S_j) + exp(sink)),
 *                   lse = log(sum_j exp(S_j) + exp(sink)); -inf = no sink.
 *                   A head with no valid entry gives out = 0 and lse = sink.
 *  workspace        >= ds_sparse_mla_swa_workspace_size(num_rows, num_heads,
 *                   k, swa_width) bytes, 256-byte aligned.
 *
 * The concatenated list is cut into 64-entry tiles spread evenly over
 * max(ceil(k / 512), ceil((k + swa_width) / 768)) splits, so the reduction
 * order depends on k and swa_width only, never on the batch.
 */
int ds_sparse_mla_decode_swa(const void* q, const void* kv_pages, int kv_dtype, int64_t num_pages,
                             const int32_t* block_table, int64_t bt_stride, const int32_t* idx,
                             const int32_t* lens, int k, const void* swa_pages,
                             int64_t swa_num_pages, const int32_t* swa_block_table,
                             int64_t swa_bt_stride, const int32_t* swa_idx,
                             const int32_t* swa_lens, int swa_width, const float* attn_sink,
                             int64_t num_rows, int num_heads, float scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t* err_flag,
                             void* stream);

/* Workspace bytes of ds_sparse_mla_decode_swa (0 for an unsupported shape). */
size_t ds_sparse_mla_swa_workspace_size(int64_t num_rows, int num_heads, int k, int swa_width);

/*
 * Indexer scores (the "MQA logits" that the top-k selects from). "[SM120]
 * Sync DS4 with upstream main + validated perf backports" routes these
 * logits through their own kernel and sizes a paged-MQA warm-up; "[Bugfix]
 * Make DSV4 sparse MLA work end-to-end ...", section "What is fixed", gives
 * the indexer one signed context length per query token. The pages give no
 * formula; this library computes the lightning indexer of the
 * DeepSeek-V3.2-Exp technical report: for query row r and position s,
 *
 *   logits[r, s] = sum_j weights[r, j] * max(0, q[r, j, :] . k[s, :])
 *
 * (multi-head queries, one shared key per position), with fp32 accumulation
 * and the heads summed in order j = 0, 1, ...
 *
 *  q              bfloat16 [num_rows, num_heads, 128], 16-byte aligned.
 *  weights        float32 [num_rows, num_heads].
 *  k_pages        bfloat16 [num_pages, 64, 128] key cache, 16-byte aligned;
 *                 the key of position s of a row is
 *                 k_pages[block_table[req, s / 64], s % 64].
 *  block_table    int32 [num_requests, bt_stride]; req = row_req[r], or r
 *                 when row_req is NULL (then num_requests >= num_rows).
 *  lens           int32 [num_rows]: row r scores positions 0 .. L_r - 1 with
 *                 L_r = clamp(lens[r], 0, 64 * bt_stride), computed signed.
 *  logits         float32 [num_rows, logits_stride], logits_stride >=
 *                 64 * bt_stride; positions at or beyond L_r are not written.
 *                 Feed it to ds_topk_per_row with row_starts = 0 and
 *                 row_ends = lens (the same clamp applies there).
 *  err_flag       optional int32 device word: DS_DEVERR_PAGE for a page id
 *                 outside [0, num_pages) (its 64 positions score -inf),
 *                 DS_DEVERR_ROWREQ for a row_req outside [0, num_requests)
 *                 (the row scores nothing).
 *
 * Supported: num_heads 16, 32 or 64; head dim 128. A row's scores depend on
 * that row's q, weights and keys alone (bitwise the same in any batch).
 * Asynchronous on `stream`; allocates nothing.
 */
int ds_indexer_logits(const void* q, const float* weights, const void* k_pages,
                      int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                      int64_t num_requests, const int32_t* row_req, const int32_t* lens,
                      int64_t num_rows, int num_heads, int head_dim, float* logits,
                      int64_t logits_stride, int32_t* err_flag, void* stream);

/*
 * KV cache write: new latent rows into the paged cache, as bf16 rows or
 * quantised to the FP8 layout above (MooreThreads/vllm-musa PR 178,
 * optimisation table: the FP8 attention cache write, with each row's FP32
 * scale groups kept contiguous).
 *
 *  latent     bfloat16 [num_rows, 576] (512 latent dims, then 64 rope dims),
 *             16-byte aligned.
 *  slots      int64 [num_rows], 8-byte aligned: row i goes to slot
 *             page * 64 + offset ("[Bugfix] Make DSV4 sparse MLA work
 *             end-to-end ...", section "What is fixed": slot =
 *             block_id * block_size + offset). A negative slot is a padding
 *             row and writes nothing (never into page 0); a slot at or past
 *             num_pages * 64 writes nothing and ORs DS_DEVERR_PAGE into
 *             err_flag.
 *  kv_dtype   DS_KV_BF16: the row is copied. DS_KV_FP8_E4M3: per group of
 *             128 latent dims, scale = amax / 448 (1 for an all-zero group),
 *             code = E4M3(x / scale) rounded to nearest, ties to even,
 *             saturating at +-448 (float32 division); the four float32
 *             scales and the 64 bf16 rope dims follow the codes.
 *  kv_pages   the pool (layout as for ds_sparse_mla_decode), 16-byte aligned;
 *             only the written slots change.
 *  err_flag   optional int32 device word (NULL = no report).
 *
 * Rows are independent: a row's bytes depend on that row alone. num_rows = 0
 * is a no-op. Slots that repeat are written in an unspecified order.
 */
int ds_kv_cache_write(const void* latent, int64_t num_rows, const int64_t* slots, int kv_dtype,
                      void* kv_pages, int64_t num_pages, int32_t* err_flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DS_SPARSE_MLA_H */
