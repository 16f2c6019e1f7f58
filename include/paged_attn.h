/*
 * paged_attn.h -- attention over a paged (block-table) KV cache on GB300
 * (sm_103a): varlen causal paged prefill, split-KV paged decode, and a mixed
 * call that routes each row of a serving batch to one of the two.
 *
 * Plain C ABI: every argument is a plain pointer (host or device, as stated)
 * or a size; no C++ or framework types cross it.  The library never allocates
 * or frees memory and never synchronizes the stream inside a compute call.
 *
 * ------------------------------------------------------------------------
 * The operation (all three compute entry points compute the same thing)
 * ------------------------------------------------------------------------
 * A batch holds num_rows sequences ("rows").  Row b brings q_b new query
 * tokens, q_b = cu_seqlens_q[b+1] - cu_seqlens_q[b], packed one row after
 * another in q; its KV length L_b = seq_lens[b] counts every key of the row,
 * the new tokens included, so the new tokens are the LAST q_b keys (bottom-
 * right causal alignment).  Query token i of row b (0 <= i < q_b) in query
 * head h attends to keys j = 0 .. L_b - q_b + i of KV head h / (Hq / Hkv):
 *
 *     x_j = s * (q . k_j) * k_scale,   out = sum_j softmax(x)_j * v_j * v_scale
 *
 * Key j of row b is slot j % P of physical page block_table[b][j / P].
 * A token with no visible key (L_b - q_b + i < 0; in particular every token of
 * a row with L_b = 0, an empty row) produces exact zeros.
 *
 * Sources: vllm-rlt PR #128 ("Purpose": the packed interface with
 * cu_seqlens_q, one block table per sequence, bottom-right causal alignment,
 * tiles with online softmax, K/V gathered through the block table, GQA; the
 * split-KV decode with 16 equal tile-aligned parts per row, fp32 partial
 * softmax states merged by a second kernel, a partition that depends on the
 * row's own length only, a static grid; "Memory": the fp32 workspace of
 * rows x heads x 16 x (head_dim + 2) x 4 bytes).  1Cat-vLLM PR #616 (original
 * description, "Purpose": small-query rows -- q = 1 decode and q = K+1
 * speculative-verify rows -- sent to the paged decode kernel instead of the
 * per-sequence prefill loop; the page size as a kernel argument, any
 * multiple of 16, with bit-identical results; an fp8_e5m2 KV cache).
 * 1Cat-vLLM PR #1279 (commit 1: GQA-packed query rows per CTA; commit 5:
 * key-range splits merged by log-sum-exp).
 *
 * ------------------------------------------------------------------------
 * Layouts (all row-major and contiguous)
 * ------------------------------------------------------------------------
 *   q, out        [total_q, Hq, head_dim]      element type q_dtype
 *   k_cache,
 *   v_cache       [num_pages, page_size, Hkv, head_dim]   element type kv_dtype
 *                 (PA_E5M2: one byte per element)
 *   block_table   int32 [num_rows, max_pages_per_row]; entries past a row's
 *                 ceil(L_b / P) pages are never read
 *   cu_seqlens_q  int32 [num_rows + 1], non-decreasing, cu_seqlens_q[0] = 0
 *   seq_lens      int32 [num_rows]
 * Query head h uses KV head h / (Hq / Hkv) (consecutive query heads share a
 * KV head).  Byte offsets into the caches are 64-bit.
 *
 * ------------------------------------------------------------------------
 * Ownership, streams and errors
 * ------------------------------------------------------------------------
 * All buffers are caller-owned.  q, caches, tables and workspace are device
 * memory; out is device memory and is fully written (every token of every
 * row).  The *_host mirrors in pa_batch are optional host copies; when given
 * they are used for argument checks and tighter grids (never stored).
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  They keep no state between calls except a per-device cache of
 * launch attributes, and are safe to call from several host threads with
 * distinct workspaces.  Results are deterministic: the same call gives the
 * same bits; a row's output does not depend on the other rows of the batch
 * (prefill rows under PA_PREFILL_PARTS_AUTO excepted), on the page size or
 * on which physical pages hold it.
 *
 * Every entry point returns a pa_status.  Host-detectable problems
 * (null pointers, bad sizes, unsupported types, a small workspace, and --
 * when host mirrors are given -- negative lengths, L_b > max_pages_per_row * P
 * or a decode row with q_b > max_decode_q) return an error before any launch.
 * Problems only the device can see (without host mirrors: a block-table entry
 * outside [0, num_pages) for a page that is needed, a row longer than its
 * block-table row, a decode row with q_b > max_decode_q) are never
 * dereferenced: such a slot reads as zeros, such a row is skipped, and a
 * sticky flag is set in the workspace header, readable with
 * paged_attn_read_errors().
 */
#ifndef PAGED_ATTN_H_
#define PAGED_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pa_stream_t;

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,          /* null pointer, inconsistent sizes or lengths */
  PA_ERR_UNSUPPORTED = 2,          /* head_dim / dtype combination not built */
  PA_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < paged_attn_workspace_size() */
  PA_ERR_CUDA = 4,                 /* a CUDA runtime call or launch failed */
  PA_ERR_NO_DEVICE = 5             /* no sm_103 device is current */
} pa_status;

typedef enum pa_dtype {
  PA_F32 = 0,
  PA_F16 = 1,
  PA_BF16 = 2,
  PA_E5M2 = 3   /* fp8 E5M2 (KV cache only), value = code * scale */
} pa_dtype;

/* Problem parameters.  Zero-initialise, then set what you need. */
typedef struct pa_params {
  int32_t num_q_heads;    /* Hq > 0 */
  int32_t num_kv_heads;   /* Hkv > 0, Hq % Hkv == 0 */
  int32_t head_dim;       /* 64, 128 or 256 */
  int32_t page_size;      /* P > 0 and a multiple of 16 */
  int32_t q_dtype;        /* pa_dtype of q and out: PA_BF16, PA_F16 or PA_F32 */
  int32_t kv_dtype;       /* pa_dtype of the caches: same as q_dtype, or PA_E5M2
                             with a 16-bit q_dtype */
  float softmax_scale;    /* s; 0 selects 1/sqrt(head_dim) */
  float k_scale;          /* per-tensor scale of K; 0 selects 1 */
  float v_scale;          /* per-tensor scale of V; 0 selects 1 */
  int32_t max_decode_q;   /* mixed: rows with 1 <= q_b <= max_decode_q go to the
                             split-KV decode path; 0 selects 16.  decode: the
                             largest q_b allowed. */
  int32_t num_splits;     /* split-KV parts per decode row: 0 or 16, or
                             PA_SPLITS_BY_LENGTH, see below */
  int32_t verify_mode;    /* decode rows with q_b > 1: PA_VERIFY_PACKED (0) or
                             PA_VERIFY_TOKENWISE (1), see below */
  int32_t prefill_kv_parts; /* prefill work items cut into key-range parts:
                               0 or 1 = not cut, 2..16 = at most this many
                               parts, PA_PREFILL_PARTS_AUTO = chosen per
                               call, see below */
  int32_t merge_mode;     /* split-KV merge of paged_attn_decode: PA_MERGE_AUTO
                             (0), PA_MERGE_SEPARATE or PA_MERGE_SAME_LAUNCH,
                             see below */
} pa_params;

/*
 * Where the split-KV merge of paged_attn_decode (and _decode_static) runs
 * (vllm-rlt PR #128, Test Result: a follow-up merges inside the decode
 * launch, bitwise identical to the two-kernel path, to save host time per
 * call).  PA_MERGE_SEPARATE: a second kernel.  PA_MERGE_SAME_LAUNCH: the
 * decode kernel itself, after a grid-wide barrier (its CTAs, at most one per
 * SM, wait for each other with the clock bound every wait has).
 * PA_MERGE_AUTO: the same launch when the decode grid is smaller than the
 * GPU (small batches, where the second launch costs more than the merge),
 * otherwise separate.  The result is the same bits either way.  Applies to
 * the TMA decode kernel (16-bit q) without PA_SPLITS_BY_LENGTH; other
 * decode paths, and the mixed call, always merge in a separate kernel.  The
 * same-launch merge needs every CTA of the decode grid resident at once: on
 * a device whose SMs are partitioned between contexts (fewer SMs available
 * than the device has), choose PA_MERGE_SEPARATE -- otherwise the barrier
 * can only end by running out (PA_DEVERR_TIMEOUT, the merge skipped).
 */
enum { PA_MERGE_AUTO = 0, PA_MERGE_SEPARATE = 1, PA_MERGE_SAME_LAUNCH = 2 };

/*
 * Decode rows with q_b > 1 (speculative-verify rows):
 *  PA_VERIFY_PACKED     the row's q_b * g query rows share one pass over the
 *                       row's keys, split by the row's L_b (K/V read once).
 *  PA_VERIFY_TOKENWISE  token i of the row is computed as a decode row of its
 *                       own, q = 1 over the first L_b - q_b + 1 + i keys and
 *                       split by that length: each token's result is bitwise
 *                       equal to decoding the tokens one at a time (1Cat-vLLM
 *                       PR #616, "Purpose": a verify row expanded into single
 *                       tokens; vllm-rlt PR #128, "Purpose": packed rows equal
 *                       serial decode only where the kernel makes them so).
 *                       The row's K/V is read once per token.  Supported for
 *                       16-bit q (same-type or E5M2 caches); other dtypes
 *                       return PA_ERR_UNSUPPORTED.
 */
enum { PA_VERIFY_PACKED = 0, PA_VERIFY_TOKENWISE = 1 };

/*
 * Prefill key-range parts (prefill_kv_parts = K in 2..16; 1Cat-vLLM PR #1279,
 * commit 5: a CTA's key range split into whole-tile ranges merged by
 * log-sum-exp).  A prefill work item (a block of GQA-packed query rows of one
 * row and KV head) whose rows see k_end keys runs as
 *     parts = min(K, ceil(ceil(k_end / 128) / 128))
 * CTAs, each over an equal run of whole 128-key units (the last one takes the
 * rest), chosen from k_end alone; each part writes an fp32 partial state
 * (acc[d], m, l) per query token and head, and a merge kernel combines the
 * parts in fixed order.  Items with at most 16384 keys are not cut.  The
 * work list runs longest part first, so long rows fill the GPU in many
 * short waves instead of a few long ones.  Results stay deterministic, and
 * independent of the rest of the batch, the page size and the physical
 * pages; a cut item equals the uncut one to rounding only.  Applies to the
 * tcgen05 prefill (16-bit q with a same-type cache, or an E5M2 cache at
 * head_dim 128 or 256); other prefill paths ignore it.  The workspace grows by
 * total_q * Hq * K * (head_dim + 2) * 4 bytes; paged_attn_decode ignores the
 * field.  Values outside 0..16 and PA_PREFILL_PARTS_AUTO return
 * PA_ERR_INVALID_ARG.
 *
 * PA_PREFILL_PARTS_AUTO (-1): the part count (1 to 4) is chosen per call, the
 * one whose work list -- items cut into equal runs of whole 128-key units,
 * at least 1024 keys each, handed out longest first, one CTA per SM --
 * finishes first on this device (1Cat-vLLM PR #1279, commit 5: the split
 * count that takes the fewest full-CTA times); launches with four or more
 * waves, or whose longest item has fewer than 8192 keys, are not cut.  It
 * needs the host mirrors and applies to calls without decode rows, and to
 * mixed calls whose decode rows use num_splits = PA_SPLITS_BY_LENGTH with
 * their long parts on the tile kernel (head_dim 256, a 16-bit q and a
 * same-type cache: those parts are short items that take a small share of
 * the SMs); other mixed calls with decode rows, and calls without mirrors,
 * are not cut.
 * The count depends on the whole batch, so a prefill row's bits may differ
 * between batches (still independent of the page size and the pages); the
 * workspace is sized for 4 parts.
 */
enum { PA_PREFILL_PARTS_AUTO = -1 };

/*
 * Length-only split count for long decode rows (num_splits =
 * PA_SPLITS_BY_LENGTH).  vllm-rlt PR #128 ("Purpose", decode bullets) fixes
 * the partition as a function of the row's own length -- what keeps a row's
 * bits independent of the batch -- and its review thread leaves the count of
 * 16 untuned.  In this mode a row of at most 32768 keys keeps the 16 parts of
 * the default (bitwise the same result); a longer row is cut into parts of
 * 2048 keys (whole 128-key tiles), at most 128 of them (longer parts past
 * 262144 keys).  At head_dim 256 with a 16-bit q and a same-type cache those
 * parts run on the tcgen05 tile kernel with all of the row's q_b * g
 * GQA-packed query rows in one 128-row tile, so each part's K/V is read
 * once; otherwise on the decode kernel, whose many more, shorter work items
 * then spread evenly over the GPU.  Still a function of the row's length
 * alone: results stay batch-invariant, page-size- and page-order-independent.
 * The partial states take 128 slots per decode token and query head: the
 * workspace is sized for that (8x the default's partial-state bytes), and the
 * merge always runs as a separate kernel.  Needs packed verify rows and a
 * 16-bit q (the decode kernel's cases); fp32 and one-token verify rows return
 * PA_ERR_UNSUPPORTED from the decode and mixed calls.  Without host mirrors
 * the decode kernel walks 128 split indices per row and KV head (most of
 * them empty for short rows).
 */
enum { PA_SPLITS_BY_LENGTH = -1 };

typedef struct pa_batch {
  int32_t num_rows;             /* B >= 0 */
  int32_t total_q;              /* cu_seqlens_q[B], the rows of q and out */
  int32_t num_pages;            /* pages in each cache */
  int32_t max_pages_per_row;    /* columns of block_table */
  const int32_t* cu_seqlens_q;  /* device [B + 1] */
  const int32_t* seq_lens;      /* device [B] */
  const int32_t* block_table;   /* device [B, max_pages_per_row] */
  const int32_t* cu_seqlens_q_host;  /* optional host mirror [B + 1] (or NULL) */
  const int32_t* seq_lens_host;      /* optional host mirror [B] (or NULL) */
} pa_batch;

/*
 * Bytes of device workspace the three compute calls need for a batch of at
 * most num_rows rows and total_q query tokens (an upper bound, so one buffer
 * serves every batch up to those sizes).  It holds a 256-byte header (error
 * flags, work counts), the mixed call's row plan, and the fp32 split-KV
 * partial states, (acc[d], m, l) per decode token, query head and split --
 * the vllm-rlt PR #128 "Memory" figure of heads x 16 x (head_dim + 2) x 4
 * bytes per decode token -- plus, with prefill_kv_parts = K > 1, the prefill
 * parts' states (K per query token and head).  Returns 0 for invalid
 * parameters.
 * The workspace must be zero-filled once before its first use (the header's
 * error word is sticky); the calls never require it to be zeroed again.
 */
size_t paged_attn_workspace_size(const pa_params* params, int32_t num_rows, int32_t total_q);

/*
 * Defined by: vllm-rlt PR #128, "Purpose", prefill bullets (the packed varlen
 * interface: cu_seqlens_q, one block table per sequence, bottom-right causal
 * alignment, tiled online softmax over K/V gathered through the block table).
 *
 * Varlen causal paged prefill: every row with q_b > 0, whatever its length,
 * on the prefill kernel (GQA-packed query tiles, online softmax over key
 * tiles, bottom-right causal mask).  Short rows are correct but slow here;
 * use paged_attn_mixed for serving batches.
 */
pa_status paged_attn_prefill(const pa_params* params, const pa_batch* batch, const void* q,
                             const void* k_cache, const void* v_cache, void* out,
                             void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * Defined by: vllm-rlt PR #128, "Purpose", decode bullets (each row's keys cut
 * into 16 equal, tile-aligned parts chosen from the row's length alone, fp32
 * partial softmax states, a second kernel that merges them, a static grid).
 *
 * Split-KV paged decode: every row (1 <= q_b <= max_decode_q; q_b > 1 are
 * speculative-verify rows) split into num_splits (16) contiguous parts of
 * whole 64-key tiles, chosen from L_b alone.  Each (row, KV head, split,
 * 16-row block of GQA-packed query rows) is one work item; persistent warps
 * take the items (rows with the longest splits first) and write fp32 partial
 * states; a second kernel merges them in fixed split order.  Batch-invariant
 * bitwise: a row's result depends on its own data and length only.
 */
pa_status paged_attn_decode(const pa_params* params, const pa_batch* batch, const void* q,
                            const void* k_cache, const void* v_cache, void* out,
                            void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * Defined by: 1Cat-vLLM PR #616, original description, "Purpose" (decode and
 * speculative-verify rows of a mixed batch sent to one paged decode launch
 * instead of the per-sequence prefill loop).
 *
 * Mixed serving batch: rows with 1 <= q_b <= max_decode_q go to the split-KV
 * decode path, longer rows to the prefill kernel, rows with q_b = 0 are
 * skipped.  The routing is computed on the device from cu_seqlens_q, so the
 * call needs no host mirrors and its grids depend only on num_rows and
 * total_q (capturable in a CUDA graph).  Each token's result is bitwise equal
 * to the one the corresponding single-path call gives.  When the batch has
 * both kinds of rows, the decode rows run on a second stream the library
 * keeps per host thread and device, forked from `stream` after the routing
 * and joined back before the call returns (event record / wait; all of the
 * call's work is ordered before later work on `stream`, also under graph
 * capture).
 */
pa_status paged_attn_mixed(const pa_params* params, const pa_batch* batch, const void* q,
                           const void* k_cache, const void* v_cache, void* out,
                           void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * Split-KV decode that allocates nothing and takes no workspace.
 *
 * No counterpart on the pages: this is an addition for callers that cannot
 * allocate device memory -- for example a plugin loaded into a program that
 * has already reserved all device memory for its own pool, or a plain C host
 * that must keep its device memory use fixed after start-up and has no
 * allocator to own a workspace's lifetime.
 *
 * Same arguments, layouts and results as paged_attn_decode minus the
 * workspace.  The scratch it needs (the fp32 partial states and a small
 * header) is one array of PA_STATIC_SCRATCH_BYTES that the library keeps in
 * device memory: every GPU that loads the library holds it until the process
 * exits.  A batch whose paged_attn_workspace_size() exceeds that size is
 * rejected with PA_ERR_WORKSPACE_TOO_SMALL before anything is launched (use
 * paged_attn_decode with a workspace of your own for larger batches).  The
 * call never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * The first call on a device (and the first after its context was torn down
 * and made again) does a one-time set-up: it looks up the array's device
 * address with that device current; make that first call before any stream
 * capture.  Every call shares the one array: calls whose work overlaps on the
 * GPU (different streams, or different host threads) race and may corrupt
 * each other's results -- serialize them.  Each call clears the array's work
 * counters; its device-side error flags are sticky, like a workspace's, and
 * paged_attn_read_errors(NULL, ...) reads and clears them.
 */
#define PA_STATIC_SCRATCH_BYTES (16u << 20)
pa_status paged_attn_decode_static(const pa_params* params, const pa_batch* batch, const void* q,
                                   const void* k_cache, const void* v_cache, void* out,
                                   pa_stream_t stream);

/* Error flags the kernels may set in the workspace header (sticky). */
#define PA_DEVERR_BAD_PAGE   0x1u  /* a needed block-table entry outside [0, num_pages),
                                      or a key past the row's block-table columns */
#define PA_DEVERR_DECODE_Q   0x4u  /* a decode-path row with q_b > max_decode_q */
#define PA_DEVERR_TIMEOUT    0x8u  /* a bounded in-kernel wait ran out; that CTA's rows
                                      are incomplete (never expected; reported, not hung) */

/*
 * Copies the workspace header's error flags to *flags (host) and clears
 * them.  workspace = NULL reads the flags of the array that
 * paged_attn_decode_static uses on the current device.  Synchronizes
 * `stream`.  Not a compute call.
 */
pa_status paged_attn_read_errors(void* workspace, pa_stream_t stream, uint32_t* flags);

/* Static description of a status code. */
const char* paged_attn_status_string(pa_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t paged_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H_ */
