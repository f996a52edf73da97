/*
 * mlafold.h -- C ABI of the folded, KV-balanced FP8 MLA decode for GB300 (sm_103a).
 *
 * What the library computes (pages: "vllm...specialized_decode.drafter.attention",
 * module overview and `folded_decode`; "vllm...specialized_decode.cutedsl.mla.balanced",
 * module overview and `BalancedMla.plan` / `BalancedMla.decode`):
 *
 *   Absorbed Multi-head Latent Attention decode is MQA over one shared latent
 *   KV head of 576 dims (512 latent + 64 rope); the value is the 512-dim latent
 *   slice of the same cache row. The k query tokens of a non-causal draft block
 *   are folded into the head axis, [R*k, H, 576] -> [R, k*H, 576], so each
 *   request's cache is read once instead of k times. Every one of the M = k*H
 *   (token, head) rows of request r gets its own softmax over keys
 *   j < seq_lens[r]:
 *
 *     s[m][j]  = bmm1_scale * dot(q[r][m][0:576], kv[page(r,j)][j%64][0:576])
 *     out[r][m] = bmm2_scale * sum_j softmax_j(s[m]) * kv[page(r,j)][j%64][0:512]
 *     lse[r][m] = log2 sum_j 2^(s[m][j] * log2(e))         (base-2 LSE)
 *
 *   with page(r, j) = block_table[r][j / 64]. bmm1_scale = sm_scale * q_scale *
 *   kv_scale and bmm2_scale = kv_scale are the stock decode's scales
 *   (drafter-attention page, `_scales`). Folded and stock layouts are the same
 *   memory: row m = t*H + h of request r is token r*k + t, head h.
 *
 * Pipeline per decode step: mla_plan_splits (once per step, reused by every
 * layer) -> mla_folded_decode (per layer) -> mla_split_combine (per layer).
 *
 * Conventions for every entry point:
 *   - The caller owns all memory and the stream. The library never allocates
 *     device memory, never synchronises the stream and never frees.
 *   - Device pointers must point to memory of the current CUDA device. Calls
 *     are asynchronous on `stream` (NULL = the legacy default stream).
 *   - Arguments are validated on the host before any launch; a bad argument
 *     returns a negative mla_status and launches nothing. No C++ exception
 *     crosses the ABI and nothing aborts the process.
 *   - A launch failure returns MLA_ERR_CUDA (the CUDA error is left for the
 *     caller to read with cudaGetLastError).
 *   - Kernels are chained with programmatic dependent launch: each reads its
 *     predecessor's outputs only after the grid dependency is resolved.
 *   - Nothing is prepared lazily at call time beyond host-side descriptor
 *     encoding, so the calls can be captured into a CUDA graph once the
 *     buffers exist (the pages prepare their plans before capture:
 *     balanced-MLA page, `BalancedMla.require`).
 */
#ifndef MLAFOLD_H
#define MLAFOLD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle: pass a cudaStream_t (or NULL). */
typedef struct CUstream_st *mla_stream_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_NULL = -1,        /* a required pointer is NULL                        */
  MLA_ERR_SHAPE = -2,       /* a size is out of range (see mla_shape)            */
  MLA_ERR_WORKSPACE = -3,   /* workspace_bytes < mla_workspace_bytes()          */
  MLA_ERR_LIST = -4,        /* list_len < mla_plan_list_len()                    */
  MLA_ERR_UNSUPPORTED = -5, /* page_size != 64, or the device is not sm_103      */
  MLA_ERR_CUDA = -6,        /* a CUDA runtime or driver call failed              */
  MLA_ERR_ALIGN = -7,       /* a pointer is not aligned as documented            */
  MLA_ERR_SCRATCH_LIMIT = -8 /* the shape needs more split-KV scratch than the
                               library's fixed array holds (see
                               mla_folded_decode_noalloc)                         */
} mla_status;

typedef enum {
  /* Split counts planned from the KV lengths: the longest requests split the
   * most, so one wave of persistent CTAs finishes together (balanced-MLA page,
   * module overview). */
  MLA_POLICY_BALANCED = 0,
  /* Every request gets the same split count, fixed by the batch shape
   * (the uniform tokenspeed schedule the balanced-MLA page compares against). */
  MLA_POLICY_UNIFORM = 1
} mla_policy;

/* Problem shape and plan parameters. All fields are host values. */
typedef struct {
  int32_t R;                /* requests in the batch (distinct KV), >= 1                   */
  int32_t k;                /* query tokens per request (draft block), >= 1                */
  int32_t H;                /* heads per token, >= 1; M = k*H rows per request, <= 4096    */
  int32_t page_size;        /* tokens per cache page; must be 64                           */
  int32_t max_pages;        /* entries per block_table row (row pitch), 1 .. 2^25 - 1      */
  int32_t num_pages;        /* pages in the cache, >= 1, < 2^25                            */
  int32_t num_ctas;         /* persistent CTAs the plan targets and the decode launches;
                               normally the device's SM count, 1..2048                     */
  int32_t min_split_tokens; /* smallest split a long request is cut into, >= 1 (e.g. 256)  */
  int32_t max_splits;       /* largest split count of one request, 1..4096 (e.g. 64)       */
  int32_t policy;           /* mla_policy                                                   */
  int32_t groups;           /* row groups per request, dividing k (0 is read as 1): the k
                               tokens of a request form `groups` decode rows of k/groups
                               tokens x H heads that all read the request's one KV (its
                               block_table row and seq_lens entry). 1 = full fold; k = the
                               stock unfolded layout; in between = the partial fold of the
                               drafter-attention page's `fold_plan`. Memory layouts of q,
                               out and lse do not change. R * groups <= 1024.              */
} mla_shape;

/* Length, in int32 words, of the plan buffer `work` that mla_plan_splits
 * fills for this shape (layout at mla_plan_splits): E entries (E = units +
 * R*groups for the balanced policy, R*groups x the uniform split count for the
 * uniform one; units = max(1, num_ctas / ceil(Mg / row block)), Mg = (k /
 * groups) * H rows per row group, row block 32 for Mg <= 32 else 64), two job
 * counters, 2E range words and 8 x units unit-table words. Returns the length
 * or a negative mla_status. Host only; launches nothing. */
int32_t mla_plan_list_len(const mla_shape *shape);

/* Bytes of split-KV workspace mla_folded_decode and mla_split_combine need for
 * this shape: FP32 partial outputs [slots][M][512] followed by FP32 log2 LSEs
 * [slots][M], where `slots` bounds the work items of requests that get two or
 * more splits (the pages size the same thing as rows x splits x heads x
 * (512 + 1) x 4 bytes: drafter-attention page, `tier_workspace_bytes`).
 * Writes the size to *bytes (0 when no request can be split). Host only. */
int32_t mla_workspace_bytes(const mla_shape *shape, size_t *bytes);

/* Plan the step's splits on the device (one CTA), from the KV lengths.
 *   seq_lens [R] int32, device: keys per request (negative is read as 0).
 *   counts   [R*groups] int32, device, written: pieces of each decode row group (>= 1).
 *   work     [list_len] int32, device, written (-1 where unused, except as noted):
 *            [0, E)      entries (row group << 12 | piece, plus 1 << 30 in
 *                        every entry of a packed plan): row groups with two
 *                        or more pieces first, then the others, each longest
 *                        first (ties: lower index first), pieces in ascending
 *                        order; a multi-piece entry's index is its partial slot.
 *                        Row group g reads request g / groups.
 *            [E, E+2)    the decode's job counters (-1).
 *            [E+2, 3E+2) packed plans: entry e's first and end page within
 *                        its row group's keys, at E+2+2e and E+3+2e.
 *            [3E+2, ...) packed plans: 8 x units words, the entries each unit
 *                        processes, in order, slot-major (unit u's j-th entry
 *                        at 3E+2 + j * units + u; -1 padded).
 *            Otherwise neither is written, and piece s of n covers pages
 *            [floor(s p / n), floor((s+1) p / n)) of the row group's p pages.
 *            Words past mla_plan_list_len(shape) are not written.
 *   list_len must be >= mla_plan_list_len(shape).
 * Balanced policy: a chunk of c pages per split, c the even share of all pages
 * over the units, raised until one wave of items fits when every request fits
 * in one wave; equal page-aligned splits of each request. In that one-wave
 * case, when the largest item would still exceed the even share by more than
 * 1/8, the plan is packed instead: the row groups' pages, longest first, are
 * laid end to end and cut into segments of the even share, one per unit
 * (kept when no row group has more than max_splits pieces and no unit more
 * than 8). Uniform policy: min(ceil(units / R), max_splits, pages) equal splits.
 * Integer arithmetic only; the result is a pure function of the lengths and
 * the shape (the project's CPU planner reproduces it bit for bit). */
int32_t mla_plan_splits(const mla_shape *shape, const int32_t *seq_lens, int32_t *counts,
                        int32_t *work, int32_t list_len, mla_stream_t stream);

/* Split-KV decode of the planned work list. Persistent CTAs take one job
 * each (a work item's block of query rows), then claim further jobs in list
 * order from a counter kept in the two words after the entries in `work`
 * (the plan leaves them at -1; the decode counts them down and its last CTA
 * puts them back to -1), so one plan serves any number of decodes in stream
 * order; with a packed plan CTA b (row block b % nb of unit b / nb,
 * nb = ceil(M / row block)) walks unit b / nb's entries instead.
 * Decodes that share one `work` array must not run concurrently.
 *   q           [R*k, H, 576] FP8 E4M3, device, 16-byte aligned: the queries in the
 *               stock token-major layout (= the folded [R, M, 576] view).
 *   kv          [num_pages, 64, 576] FP8 E4M3, device, 16-byte aligned: the
 *               paged latent cache (cols 0..511 latent = value, 512..575 rope).
 *   block_table [R, max_pages] int32, device: page ids; only the first
 *               ceil(seq_lens[r] / 64) entries of row r are read.
 *   seq_lens    [R] int32, device: the same lengths that were planned.
 *   bmm1_scale  sm_scale * q_scale * kv_scale, finite and > 0; bmm2_scale: kv_scale.
 *   counts/work the plan of mla_plan_splits for these lengths; list_len its size.
 *   workspace   >= mla_workspace_bytes(shape) bytes, device, 256-byte aligned;
 *               scratch for split partials (contents need not be initialised).
 *   out         [R, M, 512] BF16, device, 16-byte aligned, written for requests
 *               with one split (the others are written by mla_split_combine).
 *   lse         [R, M] FP32 base-2 LSE, device, written like `out`; or NULL for
 *               the route without an LSE (drafter-attention page, `fold_plan`
 *               and `draft_forward_mqa` with return_lse off): nothing is
 *               written for it (split partials still carry their own LSEs).
 *   status      optional int32 device word (may be NULL); the kernel ORs in
 *               MLA_FAULT_* bits for conditions it detects instead of trapping.
 * Numerics: FP8 QK^T and PV on the tensor cores with FP32 accumulation; FP32
 * online softmax in base 2 whose running max is kept while a new score
 * exceeds it by at most 8 (2^8, balanced-MLA page, module overview) and, when
 * it moves, is set 2 below the new maximum (P's small values then stay in
 * E4M3's normal range); P is fed
 * to the PV product as FP8 E4M3, unscaled, as the sum of two E4M3 terms built
 * from p rounded to FP16 (p16 = fp16(p), hi = e4m3(p16), lo = e4m3(p16 - hi),
 * each rounding to nearest even: hi + lo is p to about 2^-8 relative, the
 * FP16 step adding at most 2^-11); the normaliser is the FP32 sum of p. */
int32_t mla_folded_decode(const mla_shape *shape, const void *q, const void *kv,
                          const int32_t *block_table, const int32_t *seq_lens,
                          float bmm1_scale, float bmm2_scale, const int32_t *counts,
                          int32_t *work, int32_t list_len, void *workspace,
                          size_t workspace_bytes, void *out, float *lse, int32_t *status,
                          mla_stream_t stream);

/* Failure detection, for tests: mla_folded_decode with every pipeline wait
 * bounded by wait_limit_ns (1 ms .. 2 s; the regular call uses 2 s) and with
 * the first KV tile copy of CTA 0 never issued, so that a wait on it runs out
 * (the DSA prepared-layers page, `held`, records a CUDA graph that hung when a
 * kernel read its inputs before its dependency wait; every wait here is
 * bounded instead, so a lost input stops the CTA). The CTA then ORs
 * MLA_FAULT_WAIT_TIMEOUT into *status (required here), stops, lets its copies
 * and MMAs in flight finish, frees its tensor memory and returns; the other
 * CTAs finish the rest of the plan, and the job counters in `work` are back at
 * their planned state afterwards, so a regular decode of the same plan may
 * follow. The jobs the stopped CTA had taken are not computed: `out`, `lse`
 * and the workspace hold unspecified values for them. No trap, no fault. */
int32_t mla_folded_decode_wait_test(const mla_shape *shape, const void *q, const void *kv,
                                    const int32_t *block_table, const int32_t *seq_lens,
                                    float bmm1_scale, float bmm2_scale, const int32_t *counts,
                                    int32_t *work, int32_t list_len, void *workspace,
                                    size_t workspace_bytes, void *out, float *lse,
                                    int32_t *status, uint64_t wait_limit_ns,
                                    mla_stream_t stream);

/* LSE reduction of the split partials into `out` and `lse` for the requests
 * with two or more splits: out = bmm2_scale * sum_s w_s O_s / sum_s w_s, with
 * w_s = 2^(lse_s - max_s lse_s), rounded once to BF16; lse = max + log2 sum w
 * (drafter-attention page, `DraftDcp`: exp2(lse - max) / sum in FP32, one
 * BF16 rounding). Arguments as for mla_folded_decode, same plan and workspace
 * (lse may be NULL: no LSE written).
 * Rows whose splits are all empty get out = 0 and lse = -inf.
 * Ordering: launch it after that mla_folded_decode on the same stream (the
 * decode between the two is what makes the plan complete when this kernel
 * starts reading counts and work; it reads them while the decode finishes). */
int32_t mla_split_combine(const mla_shape *shape, const int32_t *counts, const int32_t *work,
                          int32_t list_len, const void *workspace, size_t workspace_bytes,
                          float bmm2_scale, void *out, float *lse, mla_stream_t stream);

/* The split reduction fused with the W_UV up-projection (drafter-attention
 * page, `DraftDcp`: the head owner merges its heads' partial rows by
 * exp2(lse - max) / sum in FP32 with one BF16 rounding and applies W_UV as a
 * BF16 MMA with FP32 accumulation; `latent_major` for the weight layout):
 *   y[t, h, :] = bf16( bf16(o(t, h)) . W_UV[h] ),   W_UV[h] is [512, 128],
 * where o(t, h) is the merged 512-dim row of token t (of R*k, token-major) and
 * head h, as mla_split_combine would write it: from the split partials in the
 * workspace for a request with two or more splits, else the row `out` already
 * holds. The merged rows themselves are not written anywhere.
 *   counts, work, list_len, workspace, workspace_bytes, bmm2_scale: the plan,
 *               workspace and scale of the mla_folded_decode call before it.
 *   out   [R, k*H, 512] BF16, device, 16-byte aligned: that decode's output
 *         (read for one-split requests only).
 *   w_uv  [H, 128, 512] BF16, device, 16-byte aligned: W_UV[h] transposed, row j
 *         holding W_UV[h, :, j] (latent-contiguous).
 *   y     [R*k, H, 128] BF16, device, 16-byte aligned, written.
 *   status optional int32 device word: MLA_FAULT_* bits (a malformed plan, a
 *         wait that timed out), as for mla_folded_decode.
 * The pages run this step after the DCP exchange; here it follows the
 * single-GPU decode. */
int32_t mla_uv_combine(const mla_shape *shape, const int32_t *counts, const int32_t *work,
                       int32_t list_len, const void *workspace, size_t workspace_bytes,
                       float bmm2_scale, const void *out, const void *w_uv, void *y,
                       int32_t *status, mla_stream_t stream);

/* Merge of S partial results of the same rows over disjoint key sets, e.g.
 * the S shards of a decode-context-parallel KV cache each decoded on its own
 * (drafter-attention page, `DraftDcp`: each head's rows are merged over the
 * DCP sources by exp2(lse - max) / sum in FP32 with one BF16 rounding):
 *   w_s = 2^(lse_s - max_s lse_s), out = sum_s w_s out_s / sum_s w_s,
 *   lse = max + log2 sum_s w_s; rows whose sources are all empty get 0, -inf.
 *   parts_out [S, rows, 512] BF16, device, 16-byte aligned: each source's out.
 *   parts_lse [S, rows] FP32 base-2 LSE, device.
 *   out [rows, 512] BF16 (16-byte aligned), lse [rows] FP32, device, written
 *   (lse may be NULL: no LSE written).
 * S in 1..4096, rows >= 1. Moving the sources between GPUs is the caller's. */
int32_t mla_lse_merge(int32_t S, int32_t rows, const void *parts_out, const float *parts_lse,
                      void *out, float *lse, mla_stream_t stream);

/* The tiered launch (drafter-attention page, `balanced_decode`): instead of
 * one persistent decode over a device-balanced plan, the longest decode rows
 * move out of one unsplit launch into "tiers" of a few rows each, every tier a
 * decode launch of its own whose rows are split, on streams of lower priority.
 * The two calls below are its data steps; the launches themselves are plain
 * mla_plan_splits / mla_folded_decode / mla_split_combine calls.
 *
 * mla_tier_plan -- which rows move (drafter-attention page, `_balanced_tables`
 * and `_plan_kernel`), one CTA on the device: rank the `rows` decode rows by
 * length, longest first (ties: lower row first); a row of rank r < split_rows
 * moves when len * move_den * pairs > move_num * sum(len) ("longer than MOVE
 * of a pair's share of the batch's keys").
 *   seq_lens   [rows] int32, device (negative is read as 0).
 *   rest_lens  [rows] int32, device, written: each row's length in the
 *              unsplit launch, 0 for a moved row.
 *   tier_rows  [split_rows] int32, device, written: the batch row of rank r
 *              if it moved, else `rows`.
 *   tier_lens  [split_rows] int32, device, written: its length if it moved,
 *              else 0.
 *   1 <= rows <= 1024, 0 <= split_rows <= rows, 1 <= pairs <= 4096,
 *   1 <= move_num, move_den <= 65536. Integer arithmetic only; the project's
 *   CPU rule reproduces it bit for bit. */
int32_t mla_tier_plan(int32_t rows, int32_t split_rows, int32_t pairs, int32_t move_num,
                      int32_t move_den, const int32_t *seq_lens, int32_t *rest_lens,
                      int32_t *tier_rows, int32_t *tier_lens, mla_stream_t stream);

/* mla_row_copy -- whole rows of `row_bytes` bytes (a multiple of 4) between
 * two row-major buffers, for the target rows whose index lies in [0, bound)
 * (drafter-attention page, `_row_copy_kernel`): with gather = 1 dst row i
 * receives src row index[i]; with gather = 0 src row i goes to dst row
 * index[i]. i runs over 0 .. targets-1; other rows are not touched.
 *   src, dst: device, 4-byte aligned (16-byte aligned rows copy in 16-byte
 *   pieces); gather: src holds `bound` rows, dst `targets`; scatter: the
 *   reverse. index [targets] int32, device. targets = 0 launches nothing. */
int32_t mla_row_copy(const void *src, void *dst, const int32_t *index, int32_t targets,
                     int32_t bound, int64_t row_bytes, int32_t gather, mla_stream_t stream);

/* The decode of mla_folded_decode followed by mla_split_combine, for callers
 * that cannot allocate device memory (a host application or plugin whose
 * allocator owns the device, or code running while a memory pool is sized):
 * instead of a caller workspace, the split-KV partials live in a fixed array
 * of device memory that the library itself defines, MLA_NOALLOC_SCRATCH_BYTES
 * (64 MiB) per GPU, held from the moment the library's device code is loaded
 * on that GPU until the process exits. The pages have no counterpart; it is
 * an addition of this library.
 *   Arguments, layouts and results are those of mla_folded_decode (which also
 *   writes the multi-split rows here, as mla_split_combine would); the plan
 *   (counts, work) comes from mla_plan_splits as usual.
 *   Returns MLA_ERR_SCRATCH_LIMIT, launching nothing, when
 *   mla_workspace_bytes(shape) exceeds MLA_NOALLOC_SCRATCH_BYTES.
 *   Calls no cudaMalloc, cudaFree or other allocating routine.
 *   The first call on a device looks the array's device address up
 *   (cudaGetSymbolAddress) with that device current and caches it. With the
 *   CUDA runtime's lazy module loading that first lookup is also when the
 *   64 MiB are committed on the device, so make the first call (a warm-up
 *   will do) before sizing memory pools and before any stream capture. The
 *   cached address does not survive cudaDeviceReset: do not call this entry
 *   point on a device after resetting it in the same process.
 *   Every call on a device uses the same array: two calls whose work overlaps
 *   on the GPU (different streams, no ordering between them) race and corrupt
 *   each other's results. Nothing in the array needs clearing between calls. */
#define MLA_NOALLOC_SCRATCH_BYTES (64u << 20)
int32_t mla_folded_decode_noalloc(const mla_shape *shape, const void *q, const void *kv,
                                  const int32_t *block_table, const int32_t *seq_lens,
                                  float bmm1_scale, float bmm2_scale, const int32_t *counts,
                                  int32_t *work, int32_t list_len, void *out, float *lse,
                                  int32_t *status, mla_stream_t stream);

/* Bits the decode kernel ORs into *status. */
#define MLA_FAULT_WAIT_TIMEOUT 0x1 /* a pipeline wait gave up; the CTA stopped early */
#define MLA_FAULT_PAGE_RANGE 0x2   /* a block-table entry was outside [0, num_pages) */
#define MLA_FAULT_WORK_ITEM 0x4    /* a work item named a request or split out of range */

#ifdef __cplusplus
}
#endif

#endif /* MLAFOLD_H */
