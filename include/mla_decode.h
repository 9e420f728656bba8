/*
 * mla_decode.h — C ABI of the GB300 (sm_103a) paged-latent MLA decode library.
 *
 * The library computes Multi-head Latent Attention decode in its absorbed
 * ("data-movement friendly", MQA) form: each of N query heads carries
 * q = [ql_nope (512) | q_pe (64)] and attends over one shared latent row
 * [kv_c (512) | k_pe (64)] per context token, with V = kv_c
 * ("mla_attention.py · tduncan/Nvidia-Optimization-Stack-VLLM", module
 * docstring, section "Data-Movement Friendly Approach"). The interface follows
 * the FlashMLA statement of the problem — a host planner that turns
 * cache_seqlens into tile-scheduler metadata and split counts, then a decode
 * call over (q, paged k_cache, block_table, cache_seqlens, softmax_scale,
 * causal, indices) returning (out, softmax_lse)
 * ("Implementation:Sgl project Sglang Flash MLA", Signature and I/O Contract) —
 * and the HALOps conventions of caller-owned buffers, in-place outputs and one
 * workspace ("MLA" API page of HALOps, mla_attention / mla_workspace).
 *
 * Conventions (all entry points):
 *  - Return 0 on success or a negative MLA_ERR_* code; no exception crosses the
 *    ABI. mla_last_error() returns a thread-local message for the last failure.
 *  - "device" pointers are CUDA device (or managed) memory owned by the caller;
 *    "host" pointers are ordinary host memory. Nothing is freed or kept.
 *  - Device work is enqueued on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream) and is asynchronous. mla_decode,
 *    mla_combine, mla_combine_v_up, mla_combine_inv_rope, mla_kv_write,
 *    mla_kv_write_norm_rope and mla_kv_gather perform no host synchronisation and
 *    no device allocation.
 *  - bf16 = IEEE bfloat16 bit patterns (uint16); all row-major, contiguous.
 *
 * KV layouts (one page = page_size rows, page_size a power of two >= 8):
 *  MLA_KV_BF16_576      row = [kv_c 512 | k_pe 64] bf16 (1152 B);
 *                       page_bytes = page_size * 1152. K = row[0:576], V = row[0:512].
 *  MLA_KV_FP8_448_UE8M0 row = [448 e4m3 NoPE | 64 bf16 RoPE] (576 B); after the
 *                       rows, page_size 8-byte scale slots (7 ue8m0 bytes, one per
 *                       64 NoPE elements, + 1 zero byte); page_bytes = page_size*584
 *                       rounded up to a multiple of 576 ("MLA" API page of HALOps,
 *                       mla_attention, kv_cache parameter). K = V = the 512-wide row.
 *  MLA_KV_FP8_512_UE8M0 the same with 512 e4m3 NoPE (640 B rows, 8 scale bytes);
 *                       page_bytes = page_size*648 rounded up to a multiple of 640.
 *                       K = [dequantised 512 | RoPE 64], V = K[0:512].
 *  A NoPE value is e4m3(byte) * 2^(scale_byte - 127).
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_OK 0
#define MLA_ERR_INVALID_ARG (-1)          /* null pointer, bad size, misalignment */
#define MLA_ERR_UNSUPPORTED (-2)          /* valid but outside what the kernels handle */
#define MLA_ERR_WORKSPACE_TOO_SMALL (-3)
#define MLA_ERR_CUDA (-4)                 /* a CUDA runtime/driver call failed */
#define MLA_ERR_DEVICE_CHECK (-5)         /* a kernel reported a bad input or a timed-out wait */
#define MLA_ERR_CAPACITY (-6)             /* a caller-provided host array is too short */

/* Bits of the device status word (mla_read_status). */
#define MLA_STATUS_WAIT_TIMEOUT 1u        /* a pipeline wait gave up after ~2 s */
#define MLA_STATUS_BAD_PAGE 2u            /* a block_table entry needed for a row < L is outside [0, num_pages) */
#define MLA_STATUS_BAD_SLOT 4u            /* a KV write slot's page is outside [0, num_pages): row not written */
#define MLA_STATUS_BAD_POSITION 8u        /* a fused write's position is outside [0, max_pos): row not written */

typedef enum {
  MLA_KV_BF16_576 = 0,
  MLA_KV_FP8_448_UE8M0 = 1,
  MLA_KV_FP8_512_UE8M0 = 2
} mla_kv_layout;

/* Sizes the kernels are built for. */
#define MLA_DV 512              /* value / output width per head */
#define MLA_BLOCK_ROWS 64       /* KV rows per tile (planner block) */
#define MLA_GROUP_ROWS 64       /* query rows (token x head) per CTA work item */
#define MLA_WORKSPACE_HEADER 256
#define MLA_DECODE_SKIP_COMBINE 1u  /* mla_decode flag: leave split partials in the workspace */
/* A dense bf16 decode whose query rows per request (q_tokens_per_req x num_heads) come in
 * groups of 128 (for example 128 heads) runs on the CTA-pair kernel: two SMs per group of
 * 128 query rows share each KV tile through one tensor-core pair. mla_decode flag: run it on
 * the single-SM kernel instead (same results within the stated tolerances; for comparison
 * and testing). Ignored for other decodes. */
#define MLA_DECODE_SINGLE_SM 2u
/* mla_decode flag, for testing failure detection only: the decode kernel withholds
 * the signal that its first score tile is complete, so the softmax's bounded wait
 * runs out; every role then leaves its loop, the call completes, and the workspace
 * status word reports MLA_STATUS_WAIT_TIMEOUT (~2 s later). Outputs are undefined. */
#define MLA_DECODE_TEST_WITHHOLD_SIGNAL 0x80000000u

typedef struct {
  int32_t num_partitions;   /* rows of sched produced */
  int32_t groups;           /* query-row groups per request = ceil(q_tokens*heads / 64) */
  int32_t total_splits;     /* num_splits[batch]: sum over requests of their split counts */
  int32_t max_splits;       /* largest split count of one request */
  size_t workspace_bytes;   /* device workspace mla_decode needs for this plan */
} mla_plan_info;

/* Page size in bytes of a layout (see above). Host only. */
int mla_page_bytes(mla_kv_layout layout, int32_t page_size, int64_t* page_bytes);

/*
 * Split-KV planner (host). The pages fix its inputs and outputs
 * (get_mla_metadata: cache_seqlens, query tokens x heads, topk ->
 * tile_scheduler_metadata, num_splits; "Implementation:Sgl project Sglang
 * Flash MLA", Signature); the rule is this library's own:
 *  - G = ceil(q_tokens_per_req*num_heads / 64) query-row groups per request;
 *    P = max(1, num_sms / G) partitions share the SMs.
 *  - request b has nb_b = max(1, ceil(K_b / 64)) KV blocks, K_b = topk if
 *    topk > 0 else cache_seqlens[b]; its cost is nb_b + 3.
 *  - payload = the smallest p >= p0 = max(ceil(sum cost / P), 4) with which the
 *    greedy fill below opens at most P partitions (p0 + 6 always does, so only
 *    p0 .. p0 + 6 are tried).
 *  - with min_splits = k > 1, let n = the fewest blocks of a request that has
 *    >= k blocks; cap = max(1, (n - 1) / (k - 1)) + 3 (integer division) cuts
 *    every such request into >= k splits. If cap < payload, the payload becomes
 *    the p in (cap - 64, cap], p > 3, with the fewest ceil(partitions(p) / P) * p
 *    (ties: the larger p), partitions(p) being the count the fill opens.
 *  - partitions are filled greedily in request order; a partition that cannot
 *    take the rest of a request takes (budget - 3) blocks of it and closes.
 * Outputs (host arrays):
 *  sched [num_partitions][8] int32: begin_req, begin_blk, end_req, end_blk
 *        (exclusive, request-major order), first_split (split index of the first
 *        segment within begin_req), 0, 0, 0.
 *  num_splits [batch + 1] int32: prefix sums of per-request split counts.
 * Pass sched == NULL to only fill *info. Returns MLA_ERR_CAPACITY (with *info
 * filled) if sched_capacity < info->num_partitions.
 * cache_seqlens: host [batch]; batch >= 1; q_tokens_per_req >= 1; num_heads
 * >= 1; topk >= 0; min_splits >= 1; num_sms >= 1 (the SM count of the device
 * mla_decode will run on).
 */
int mla_decode_plan(const int32_t* cache_seqlens, int32_t batch, int32_t q_tokens_per_req, int32_t num_heads,
                    int32_t topk, int32_t min_splits, int32_t num_sms, int32_t* sched, int32_t sched_capacity,
                    int32_t* num_splits, mla_plan_info* info);

/*
 * Decode (device). out[t, n, :] and lse[t, n] for every query token t of every
 * request and head n: softmax over the request's candidate KV rows of
 * sm_scale * <q[t, n, :], K_j>, applied to V_j
 * ("mla_attention.py · tduncan/Nvidia-Optimization-Stack-VLLM", module docstring,
 * "Data-Movement Friendly Approach"; "Implementation:Sgl project Sglang Flash
 * MLA", I/O Contract).
 *  q            device bf16 [T = batch*q_tokens_per_req, num_heads, Dqk]
 *               (Dqk = 576, or 512 for MLA_KV_FP8_448_UE8M0), 16-byte aligned.
 *  kv_cache     device uint8 [num_pages, page_bytes(layout, page_size)], 16-B aligned.
 *  block_table  device int32 [batch, max_pages]: page of each page-sized block.
 *  cache_seqlens device int32 [batch]: L_b, context rows including the query
 *               tokens' own new rows (seq_len = context_len + query_len,
 *               "mla_attention.py", MLACommonMetadata).
 *  sm_scale     softmax scale of the scores (positive, finite).
 *  sink         device float [num_heads] per-head sink logit added to the
 *               softmax denominator only, or NULL ("MLA" API page of HALOps,
 *               mla_attention, attn_sink). lse does not include it.
 *  indices      device int32 [T, topk] request-local KV positions, or NULL for
 *               dense decode; entries outside [0, L_b) are skipped, duplicates
 *               count twice; causal is ignored with indices. With indices and
 *               q_tokens_per_req > 1, num_heads must be a multiple of 64.
 *  causal       nonzero: query token i of a request sees rows j <= L_b - s_q + i
 *               (draft tokens at consecutive positions, "MLA" API page of
 *               HALOps, mla_attention, draft_tokens).
 *  sched, num_splits, num_partitions, total_splits: from mla_decode_plan with
 *               the same cache_seqlens/topk/heads/tokens, copied to the device.
 *  workspace    device, >= info.workspace_bytes, 256-B aligned; its first 256
 *               bytes hold the status word and must be zeroed once
 *               (mla_workspace_init) before first use.
 *  out          device bf16 [T, num_heads, 512]; lse device float [T, num_heads]
 *               (natural log; -inf and out = 0 for an empty candidate set).
 * num_heads >= 1 and q_tokens_per_req*num_heads <= 4096. Requests split by the
 * plan are merged by mla_combine on the same stream inside this call unless
 * flags has MLA_DECODE_SKIP_COMBINE, in which case the caller runs mla_combine
 * on the workspace partials (layout: MLA_WORKSPACE_HEADER bytes of status, then
 * part_lse float [total_splits, R] padded to a multiple of 256 bytes, then
 * part_out float [total_splits, R, 512], R = q_tokens_per_req * num_heads, then the
 * partial max logits of mla_sparse_prefill, float [total_splits, R] padded to 256 bytes).
 */
int mla_decode(const void* q, const void* kv_cache, mla_kv_layout layout, int64_t num_pages, int32_t page_size,
               const int32_t* block_table, int32_t max_pages, const int32_t* cache_seqlens, int32_t batch,
               int32_t q_tokens_per_req, int32_t num_heads, float sm_scale, const float* sink,
               const int32_t* indices, int32_t topk, int32_t causal, const int32_t* sched,
               const int32_t* num_splits, int32_t num_partitions, int32_t total_splits, void* workspace,
               size_t workspace_bytes, void* out, float* lse, uint32_t flags, void* stream);

/*
 * Sparse prefill (device): "Implementation:Sgl project Sglang Flash MLA", Signature and
 * I/O Contract of flash_mla_sparse_fwd (q, kv, indices, sm_scale, d_v = 512 -> out,
 * max_logits, lse). Every token attends over its own top-k list of rows of one unpaged
 * latent run.
 *  q        device bf16 [num_tokens, num_heads, 576] (16-B aligned).
 *  kv       device bf16 [s_kv, 576]: the latent rows [kv_c 512 | k_pe 64] (16-B aligned);
 *           K = row, V = row[0:512].
 *  indices  device int32 [num_tokens, topk]: positions in kv; entries outside
 *           [0, s_kv) are skipped, duplicates count twice.
 *  sched, num_splits, num_partitions, total_splits: a plan from mla_decode_plan with
 *           cache_seqlens = s_kv for each of num_tokens requests, q_tokens_per_req = 1,
 *           num_heads and topk (copied to the device); workspace as for mla_decode.
 *  out      device bf16 [num_tokens, num_heads, 512]; lse device float [num_tokens,
 *           num_heads] (natural log over the listed rows); max_logits device float
 *           [num_tokens, num_heads]: the largest sm_scale * <q, K_j> over the listed
 *           rows. A token with no valid entry gets out = 0, lse = -inf, max_logits = -inf.
 * flags: MLA_DECODE_SKIP_COMBINE is not accepted here (split partials are always merged).
 * Errors as mla_decode.
 */
int mla_sparse_prefill(const void* q, const void* kv, int32_t s_kv, const int32_t* indices, int32_t topk,
                       int32_t num_tokens, int32_t num_heads, float sm_scale, const int32_t* sched,
                       const int32_t* num_splits, int32_t num_partitions, int32_t total_splits, void* workspace,
                       size_t workspace_bytes, void* out, float* max_logits, float* lse, uint32_t flags,
                       void* stream);

/*
 * No-allocation decode (device). The pages have no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory — a host that
 * gives its whole GPU memory budget to its own pool and forbids extensions to
 * call cudaMalloc, a latency-critical loop that must not pay for an allocation
 * (cudaMalloc may synchronise the device), or a language binding with no way to
 * allocate CUDA memory. It does exactly what mla_decode does (same arguments,
 * same results) but uses a workspace the library keeps in a static device array
 * of MLA_STATIC_WORKSPACE_BYTES, held on every GPU that loads the library until
 * the process exits. Plans needing more (info.workspace_bytes larger than that)
 * are rejected with MLA_ERR_WORKSPACE_TOO_SMALL. It allocates nothing.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any stream
 *    capture.
 *  - All calls share the one array: calls that overlap on the GPU (several
 *    streams or host threads) race with each other.
 *  - Each call clears the status word first. status_out, if not NULL, is a
 *    device uint32 that receives this call's MLA_STATUS_* bits (stream-ordered).
 *    It is the only way to see this call's device-side checks (a bad page, a
 *    pipeline wait that ran out): the static status word is not exposed, and
 *    the next call clears it. Pass NULL only when those checks are not needed.
 */
#define MLA_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)
int mla_decode_static_workspace(const void* q, const void* kv_cache, mla_kv_layout layout, int64_t num_pages,
                                int32_t page_size, const int32_t* block_table, int32_t max_pages,
                                const int32_t* cache_seqlens, int32_t batch, int32_t q_tokens_per_req,
                                int32_t num_heads, float sm_scale, const float* sink, const int32_t* indices,
                                int32_t topk, int32_t causal, const int32_t* sched, const int32_t* num_splits,
                                int32_t num_partitions, int32_t total_splits, void* out, float* lse,
                                uint32_t* status_out, void* stream);

/*
 * Sliding-window runs (device): compress each token's window of cache slots into at
 * most two runs of consecutive slots ("MLA" API page of HALOps, mla_attention_plan).
 *  kv_indices   device int32 [num_tokens, topk]: the window's cache slots
 *               (page * page_size + offset); columns past a token's length are ignored.
 *  topk_lengths device int32 [num_tokens] or NULL (every window has topk rows); clamped
 *               to [0, topk].
 *  kv_run_step  1 or -1: the slot step between consecutive window rows.
 *  runs         device int32 [num_tokens, 4], 16-byte aligned: (slot0, len0, slot1, rows).
 * A run continues while the next slot equals the previous one plus kv_run_step and lies on
 * the same page. A window of more than two runs is cut to its first row (rows = 1). Each
 * run is stored from its lowest slot upwards: row g < len0 is slot slot0 + g, row g >= len0
 * is slot slot1 + g - len0, for g < rows. An empty window gives (0, 0, 0, 0).
 */
int mla_swa_plan(const int32_t* kv_indices, const int32_t* topk_lengths, int32_t num_tokens, int32_t topk,
                 int32_t page_size, int32_t kv_run_step, int32_t* runs, void* stream);

/*
 * Decode over window runs (device): as mla_decode, with each query token attending over
 * the rows of its runs (mla_swa_plan) instead of a request's context. Slots address the
 * cache directly (no block_table, no cache_seqlens); a slot outside the cache is skipped
 * and counted in the status word like a bad page. `window` is the largest rows value
 * (the topk of mla_swa_plan) and is the topk given to mla_decode_plan for the schedule.
 * Requests are independent tokens' windows: q_tokens_per_req > 1 needs num_heads % 64 == 0.
 */
int mla_decode_runs(const void* q, const void* kv_cache, mla_kv_layout layout, int64_t num_pages, int32_t page_size,
                    const int32_t* runs, int32_t window, int32_t batch, int32_t q_tokens_per_req, int32_t num_heads,
                    float sm_scale, const float* sink, const int32_t* sched, const int32_t* num_splits,
                    int32_t num_partitions, int32_t total_splits, void* workspace, size_t workspace_bytes, void* out,
                    float* lse, uint32_t flags, void* stream);

/*
 * Split combine (device): for every request whose split count
 * (num_splits[b+1] - num_splits[b]) is at least 2, merge its partials by
 * log-sum-exp — lse = ln sum_s e^(lse_s), out = sum_s e^(lse_s - lse) o_s, a
 * partial with lse_s = -inf carrying no weight ("mla_attention.py", Chunked
 * Prefill: merge_attn_states; neutralize_empty_context_partials) — then apply
 * the sink once: out *= 1 / (1 + e^(sink - lse)). Requests with one split are
 * left untouched.
 *  part_out device float [total_splits, rows_per_req, 512]; part_lse device
 *  float [total_splits, rows_per_req]; split s of request b is row block
 *  num_splits[b] + s. rows_per_req = q_tokens_per_req * num_heads; the head of
 *  row r is r % num_heads.
 */
int mla_combine(const float* part_out, const float* part_lse, const int32_t* num_splits, int32_t batch,
                int32_t rows_per_req, int32_t num_heads, const float* sink, void* out, float* lse, void* stream);

/*
 * Split combine fused with the value up-projection (device): the step after the
 * decode in the absorbed form. Every query row's latent output x (512 wide) is
 * mapped to its head's value space, o_v = x W_UV[n] ("mla_attention.py ·
 * tduncan/Nvidia-Optimization-Stack-VLLM": _v_up_proj multiplies the (N, B, L)
 * latent output by W_UV (N, L, V)).
 *  part_out, part_lse, num_splits, sink: as for mla_combine. part_out and part_lse
 *         may be NULL (both): then no row is merged and every row of out is taken as
 *         written (for a plan in which no request has two or more splits).
 *  w_uv   device bf16 [num_heads, 512, 128] (value head dim 128), 16-byte aligned.
 *  out    device bf16 [T, N, 512]: read for requests with one split (the decode
 *         wrote it); for split requests the merged row is written here first,
 *         exactly as mla_combine writes it (and lse with it).
 *  o_v    device bf16 [T, N, 128]: o_v[t, n, :] = bf16(sum_l x[t, n, l] W_UV[n, l, :]),
 *         x being the bf16 latent row, products summed in fp32.
 *  status optional device uint32 (NULL or a workspace): bit 0 is set when a
 *         bounded wait ran out (the call then leaves o_v incomplete).
 */
int mla_combine_v_up(const float* part_out, const float* part_lse, const int32_t* num_splits, int32_t batch,
                     int32_t q_tokens_per_req, int32_t num_heads, const float* sink, const void* w_uv, void* out,
                     float* lse, void* o_v, uint32_t* status, void* stream);

/*
 * Split combine fused with the inverse RoPE of the output (device): the step after
 * the decode for rows whose value part carries RoPE (the DSV4 row: value dim 512 =
 * 448 NoPE + 64 RoPE, whose O still carries the rotation; "MLA" API page of HALOps,
 * mla_output_proj, which merges the split-KV partials by LSE and then undoes the RoPE).
 * Every row of out [T, N, 512] (bf16, in place) is first merged as mla_combine
 * merges it when its request has two or more splits and part_out / part_lse are
 * given (writing lse too), or taken as the decode wrote it; then elements [rope0, rope0 + 64) are rotated back: pair i =
 * (u, v) -> (u c + v s, v c - u s) with (c, s) = freqs[positions[t], 2i .. 2i + 1],
 * in fp32, and rounded to bf16. Rows of a token whose position is outside
 * [0, max_pos) are merged but not rotated.
 *  positions device int32 [T]; freqs device float [max_pos, 64]; rope0 a multiple
 *  of 4 with rope0 + 64 <= 512 (448 for the DSV4 row).
 */
int mla_combine_inv_rope(const float* part_out, const float* part_lse, const int32_t* num_splits, int32_t batch,
                         int32_t q_tokens_per_req, int32_t num_heads, const float* sink, const int32_t* positions,
                         const float* freqs, int32_t max_pos, int32_t rope0, void* out, float* lse, void* stream);

/*
 * KV-row write (device): scatter n new rows into their pages ("MLA" API page of
 * HALOps, mla_attention: its cache-write step and kv_cache parameter).
 *  rows   device bf16 [n, row_elems], already RMSNorm'd (and RoPE'd);
 *         row_elems = 576 (layouts 0 and 2) or 512 (layout 1: 448 NoPE | 64 RoPE).
 *  slots  device int32 [n]: page * page_size + offset; negative slots are skipped.
 * Layout 0 copies the bits. fp8 layouts: per 64-element NoPE group,
 * amax = max(max|x|, 1e-10f), e = the smallest integer with 448 * 2^e >= amax,
 * scale byte = e + 127, code = e4m3 round-to-nearest-even, saturating, of
 * x * 2^-e; the RoPE part is copied as bf16. A NaN element takes no part in its
 * group's amax (the maximum is taken over the numbers) and is stored as the
 * E4M3 NaN code 0x7F; an infinite one makes amax infinite (scale byte 254) and
 * is stored as +-448.
 *  status device uint32 or NULL: a row whose slot's page is >= num_pages is not
 *         written and ORs MLA_STATUS_BAD_SLOT into *status.
 */
int mla_kv_write(const void* rows, const int32_t* slots, int32_t n, void* kv_cache, mla_kv_layout layout,
                 int64_t num_pages, int32_t page_size, uint32_t* status, void* stream);

/*
 * Normalise, rotate and write new KV rows (device): the step that produces a
 * cache row from the latent projection, fused with mla_kv_write ("MLA" API page
 * of HALOps, mla_attention: the step that normalises and rotates q and kv before the
 * cache write; its kv_norm_weight, kv_eps, positions and freqs_real parameters).
 *  raw     device bf16 [n, row_elems], the un-normalised rows; row_elems = 576
 *          for layouts 0 and 2 ([kv_c 512 | k_pe 64]) and 512 for layout 1 (the
 *          DSV4 row: 448 NoPE | 64 RoPE).
 *  slots   device int32 [n] as for mla_kv_write (negative slots are skipped).
 *  positions device int32 [n]: the token position that selects the RoPE row;
 *          rows whose position is outside [0, max_pos) are skipped (not written).
 *  norm_weight device bf16 [512]: the RMSNorm gain; eps: the RMSNorm epsilon.
 *  freqs   device float [max_pos, 64]: per position 32 interleaved (cos, sin) pairs.
 * For every row, in fp32:
 *  - RMSNorm of the 512 latent elements (elements 0..511):
 *    y = x * (1 / sqrt(sum(x^2) / 512 + eps)) * w;
 *  - RoPE of the 64 RoPE elements, pair i = (x[2i], x[2i+1]) of that part, with
 *    (c, s) = (freqs[pos, 2i], freqs[pos, 2i+1]): (x0 c - x1 s, x0 s + x1 c).
 *    Layouts 0 and 2 rotate the raw k_pe (elements 512..575, not normalised);
 *    layout 1 rotates elements 448..511 after the normalisation;
 *  - the row is rounded to bf16 (nearest even) and written exactly as
 *    mla_kv_write writes that bf16 row.
 * status (device uint32, or NULL) is OR-ed with MLA_STATUS_BAD_POSITION for a
 * row skipped for its position and MLA_STATUS_BAD_SLOT for a row whose slot's
 * page is out of range (as for mla_kv_write).
 */
int mla_kv_write_norm_rope(const void* raw, const int32_t* slots, const int32_t* positions, const void* norm_weight,
                           float eps, const float* freqs, int32_t max_pos, int32_t n, void* kv_cache,
                           mla_kv_layout layout, int64_t num_pages, int32_t page_size, uint32_t* status,
                           void* stream);

/*
 * Page gather (device, a test export): out[j, :] = decoded K row j of one
 * request (block_table_row device int32 [max_pages]) for j < length, as float
 * [length, Dqk]. Rows whose page is out of range are written as NaN.
 */
int mla_kv_gather(const void* kv_cache, mla_kv_layout layout, int64_t num_pages, int32_t page_size,
                  const int32_t* block_table_row, int32_t max_pages, int32_t length, float* out, void* stream);

/* Zero the workspace status header (enqueued on stream). */
int mla_workspace_init(void* workspace, void* stream);

/* Synchronise `stream`, read the status word into *status (MLA_STATUS_* bits);
 * clear it if reset != 0. Returns MLA_ERR_DEVICE_CHECK when a bit is set. */
int mla_read_status(void* workspace, uint32_t* status, int32_t reset, void* stream);

/* Thread-local message describing the last nonzero return of this thread. */
const char* mla_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DECODE_H_ */
