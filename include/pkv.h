/*
 * pkv — the per-layer paged-KV attention step on NVIDIA GB300 (sm_103a).
 *
 * Two calls make one layer's step:
 *   pkv_write      scatters the step's new K/V rows into the block-paged cache;
 *   pkv_attention  runs causal varlen attention for a packed batch of prefill
 *                  chunks and decodes over that cache.
 * Call pkv_write before pkv_attention on the same stream: the step's own
 * tokens must be in the cache when attention reads it.
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers of the current CUDA device.
 *   - bf16 tensors are passed as raw bit storage (2 bytes per element).
 *   - Row strides are counted in elements, not bytes.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on `stream` and returns; none
 *     synchronises except pkv_get_error.  Work is stream ordered as usual:
 *     the write and attention calls (not pkv_prepare_step) launch their
 *     kernels with programmatic dependent launch,
 *     so a kernel may begin its set-up while the work before it on the
 *     stream is finishing, but it writes no global memory, and reads none
 *     that that work produces, until that work has finished.  One
 *     refinement: the step plan of pkv_attention, pkv_attention_int8,
 *     pkv_attention_noalloc and pkv_plan reads query_start_loc and seq_lens
 *     as soon as its kernel starts, which is after the kernel before it on
 *     the stream has finished, or, when that kernel is pkv_write's (or
 *     pkv_write_int8's) or another plan's, after everything before that
 *     kernel has finished: so enqueue the metadata before the write (as a
 *     step does), or from a kernel launched without programmatic
 *     serialisation.  Within a bf16 attention call that has prefill work,
 *     the decode kernel leaves some SMs to the prefill kernel, whose items
 *     run there beside the decode units.
 *   - The caller owns every buffer it passes; the library keeps no pointer to
 *     any of them after the call returns.  The library owns one grow-only
 *     device workspace per device (step plan, split-KV partial results and
 *     the device error word).  It is allocated on first use, or beforehand by
 *     pkv_reserve_workspace (needed before CUDA-graph capture, since no
 *     allocation may happen while a stream is being captured).
 *   - Errors found on the host (null pointers, sizes, geometry, alignment)
 *     return a negative PKV_ERR_* code before anything is enqueued: no buffer
 *     is touched.  pkv_last_error_string() describes the last such error of
 *     the calling thread.
 *   - Errors in the VALUES of device-resident metadata (a slot past the pool,
 *     a block id outside the pool, seq_len < query_len, decreasing
 *     query_start_loc, a block-table row too short) cannot be seen by the host
 *     without a device-to-host copy.  The kernels skip the offending item,
 *     never trap, and OR a PKV_DEV_ERR_* bit into a per-device error word that
 *     pkv_get_error reads and clears.
 *
 * Geometry supported: head_size 128, block_size 16, num_heads a multiple of
 * num_kv_heads (MHA: equal; GQA: num_kv_heads > 1; MQA: num_kv_heads = 1),
 * num_heads / num_kv_heads <= 32.  Anything else returns PKV_ERR_UNSUPPORTED.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side status codes. */
#define PKV_OK 0
#define PKV_ERR_ARG (-1)         /* null pointer, negative size, bad stride   */
#define PKV_ERR_UNSUPPORTED (-2) /* geometry outside the supported set        */
#define PKV_ERR_ALIGN (-3)       /* pointer or row stride not 16-byte aligned */
#define PKV_ERR_CUDA (-4)        /* a CUDA runtime call failed                */
#define PKV_ERR_NO_DEVICE (-5)   /* no usable sm_103 device current           */

/* Device error word bits (pkv_get_error). */
#define PKV_DEV_ERR_SLOT_RANGE 1 /* pkv_write: slot >= num_blocks*block_size  */
#define PKV_DEV_ERR_QSL 2        /* query_start_loc decreasing or > q_rows    */
#define PKV_DEV_ERR_SEQ_LEN 4    /* seq_len < query_len (or negative)         */
#define PKV_DEV_ERR_BT_WIDTH 8   /* ceil(seq_len/block_size) > row width      */
#define PKV_DEV_ERR_BLOCK_ID 16  /* block id outside [0, num_blocks)          */
#define PKV_DEV_ERR_TIMEOUT 32   /* an on-chip pipeline wait gave up          */
#define PKV_DEV_ERR_INT8_PREFILL 64 /* pkv_attention_int8: a request too long for
                                       the decode path (its rows are skipped)  */
#define PKV_DEV_ERR_CAPACITY 128 /* the step plan outgrew the workspace: the
                                    whole step was skipped (no output row
                                    written).  The library sizes the workspace
                                    so that this does not happen; the bit
                                    reports a broken bound, never truncation */

/*
 * pkv_write — the cache-write scatter.
 *
 * Defined by "vLLM 推理全流程深度解析" (vLLM inference deep dive),
 * reshape_and_cache section, and "Tour: One forward pass", stop 4 (slot =
 * block_number * block_size + offset; padding tokens at PAD_SLOT_ID = -1) and
 * stop 10 (the separate cache-update op before attention).
 *
 * For t in [0, n_tokens): s = slot_mapping[t]; if s < 0 the token is padding
 * and is skipped; otherwise the [num_kv_heads, head_size] rows k[t] and v[t]
 * are copied bit for bit to key_cache[s / block_size][s % block_size] and
 * value_cache[s / block_size][s % block_size].  No other cache byte changes.
 *
 *   k, v          bf16 [n_tokens, num_kv_heads, head_size]; token t starts at
 *                 element t * k_row_stride (v_row_stride); each token's
 *                 num_kv_heads * head_size elements are contiguous.  Strided
 *                 rows let k and v be column slices of a fused qkv tensor.
 *   key_cache,    bf16 [num_blocks, block_size, num_kv_heads, head_size],
 *   value_cache   contiguous.  Written in place.
 *   slot_mapping  int64 [n_tokens].  Non-negative slots within one call must
 *                 be distinct (the result is otherwise unspecified).  A slot
 *                 >= num_blocks * block_size is skipped and reported as
 *                 PKV_DEV_ERR_SLOT_RANGE.
 *   n_tokens      >= 0; 0 enqueues nothing.
 * Alignment: k, v, both caches 16-byte aligned; row strides * 2 bytes a
 * multiple of 16.
 */
int pkv_write(const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride,
              void* key_cache, void* value_cache, int64_t num_blocks, int32_t block_size,
              int32_t num_kv_heads, int32_t head_size, const int64_t* slot_mapping,
              int64_t n_tokens, void* stream);

/*
 * pkv_attention — varlen causal attention over the paged cache for a packed
 * batch that mixes prefill chunks and decodes.
 *
 * Defined by "Tour: One forward pass", stop 3 (query_start_loc, seq_lens =
 * num_computed + query_len), stop 5 (the attention metadata) and stop 10
 * (cu_seqlens_q = query_start_loc, seqused_k = seq_lens, block_table; causal;
 * only the first query_start_loc[num_reqs] output rows are written); "vLLM
 * MHA Code Path: From QKV to Paged KV Cache", sections "One Path Covers MHA,
 * GQA, and MQA" and "Worked Trace: One Decode Token" (the current token
 * attends to itself); "vLLM 推理全流程深度解析", paged_attention_v1 section
 * (gather through block_tables, softmax, weighted sum of V).
 *
 * For request r: q0 = query_start_loc[r], n = query_start_loc[r+1] - q0,
 * L = seq_lens[r], ctx = L - n.  Query row i (absolute position ctx + i) of
 * head h reads KV head h / (num_heads / num_kv_heads) and keys 0 .. ctx + i,
 * key j living at key_cache[block_table[r][j / 16]][j % 16]:
 *   out[q0+i][h] = sum_j softmax_j(scale * q[q0+i][h] . K_j) * V_j,
 * computed with bf16 inputs, fp32 accumulation and a bf16 result.  Any n
 * works; requests whose n * (num_heads / num_kv_heads) fits 16 rows (32 for
 * groups above 16), single-token decodes and short multi-token (speculative)
 * steps, take the split-KV decode path, longer ones the prefill path; both
 * compute the formula above.
 *
 *   q               bf16 [q_rows, num_heads, head_size], row stride
 *                   q_row_stride elements (>= num_heads * head_size).
 *   key_cache,      bf16 [num_blocks, block_size, num_kv_heads, head_size],
 *   value_cache     contiguous; read only.
 *   query_start_loc int32 [num_reqs + 1], non-decreasing, last <= q_rows.
 *   seq_lens        int32 [num_reqs].
 *   block_table     int32 [num_reqs, block_table_width], rows contiguous.
 *                   Entries past ceil(seq_len / 16) are never read.
 *   num_reqs        >= 0.
 *   scale           softmax scale (1/sqrt(head_size) for standard attention).
 *   out             bf16 [q_rows, num_heads, head_size], row stride
 *                   out_row_stride.  Rows >= query_start_loc[num_reqs], and
 *                   rows of requests that fail a metadata check, are not
 *                   written.  (A request with a block id outside the pool is
 *                   reported as PKV_DEV_ERR_BLOCK_ID; its rows are then
 *                   unspecified.)
 * Alignment: q, out, caches 16-byte aligned; row strides * 2 bytes multiples
 * of 16.
 */
int pkv_attention(const void* q, int64_t q_row_stride, int64_t q_rows, int32_t num_heads,
                  const void* key_cache, const void* value_cache, int64_t num_blocks,
                  int32_t block_size, int32_t num_kv_heads, int32_t head_size,
                  const int32_t* query_start_loc, const int32_t* seq_lens,
                  const int32_t* block_table, int64_t block_table_width, int32_t num_reqs,
                  float scale, void* out, int64_t out_row_stride, void* stream);

/*
 * pkv_plan / pkv_attention_planned — one step plan serving every layer.
 *
 * "Tour: One forward pass", stop 5: one attention-metadata object is built per
 * step and shared by all layers; stop 7: the 32-layer loop.  pkv_attention
 * builds its plan (the work lists: decode units, split pairs, prefill tiles)
 * on every call; pkv_plan builds it once per step and pkv_attention_planned
 * runs one layer on it, so a step of L layers pays for one plan.
 *
 * pkv_plan(q_rows, num_heads, num_kv_heads, query_start_loc, seq_lens,
 *          block_table_width, num_reqs, stream): the metadata arguments of
 *   pkv_attention, with its checks.  The plan is a snapshot: the work lists
 *   hold every request's query rows and lengths, and no later call reads
 *   query_start_loc or seq_lens again.  The plan lives in this device's
 *   workspace (grown here if needed, so reserve it before a graph capture)
 *   and replaces the previous one; pkv_attention, pkv_attention_int8 and a
 *   workspace reallocation (a call needing more room, pkv_reserve_workspace)
 *   replace or drop it too.  Requests whose metadata fail a check are
 *   reported in the error word when the plan kernel runs.
 *
 * pkv_attention_planned(q, q_row_stride, num_heads, key_cache, value_cache,
 *          num_blocks, block_size, num_kv_heads, head_size, block_table,
 *          scale, out, out_row_stride, stream): pkv_attention for the current
 *   plan: the same result as a pkv_attention call with the plan's metadata
 *   and these buffers (q and out hold the plan's q_rows rows; block_table is
 *   read again, so a layer may point at its own table of the same width).
 *   num_heads and num_kv_heads must equal the plan's; with no valid plan on
 *   the current device the call returns PKV_ERR_ARG.  Calls are stream
 *   ordered: the plan must be enqueued before, on the same stream (or one
 *   ordered after it).
 */
int pkv_plan(int64_t q_rows, int32_t num_heads, int32_t num_kv_heads,
             const int32_t* query_start_loc, const int32_t* seq_lens, int64_t block_table_width,
             int32_t num_reqs, void* stream);
int pkv_attention_planned(const void* q, int64_t q_row_stride, int32_t num_heads,
                          const void* key_cache, const void* value_cache, int64_t num_blocks,
                          int32_t block_size, int32_t num_kv_heads, int32_t head_size,
                          const int32_t* block_table, float scale, void* out,
                          int64_t out_row_stride, void* stream);

/*
 * pkv_prepare_step — the step-side metadata the two calls read, computed on
 * the device from the request state (no host round trip).
 *
 * Defined by "Tour: One forward pass", stop 3 (prepare_pos_seq_lens: token t
 * of request r sits at num_computed[r] + (t - query_start_loc[r]); seq_len =
 * num_computed + query_len; padding rows of positions are not written) and
 * stop 4 (gather_block_tables: each request's persistent row, idx_mapping,
 * copied into batch order; compute_slot_mappings: slot = block_number *
 * block_size + offset; rows past the last request's tokens get -1).
 *
 *   query_start_loc       int32 [num_reqs + 1], non-decreasing.
 *   num_computed          int32 [num_reqs]: tokens already in the cache.
 *   idx_mapping           int32 [num_reqs]: persistent row of each batch row
 *                         (NULL: batch row r uses persistent row r).
 *   persistent_block_table int32 [persistent_rows, block_table_width].
 *   positions (out)       int64 [num_tokens_padded]; rows of scheduled tokens.
 *   seq_lens (out)        int32 [num_reqs].
 *   slot_mapping (out)    int64 [num_tokens_padded]; -1 for padding rows.
 *   block_table (out)     int32 [num_reqs, block_table_width] in batch order,
 *                         or NULL to skip the gather.
 * A position past the row width, or a persistent row outside the table,
 * gives slot -1 for that token and PKV_DEV_ERR_BT_WIDTH in the error word.
 */
int pkv_prepare_step(const int32_t* query_start_loc, const int32_t* num_computed,
                     const int32_t* idx_mapping, const int32_t* persistent_block_table,
                     int64_t persistent_rows, int64_t block_table_width, int32_t num_reqs,
                     int64_t num_tokens_padded, int64_t* positions, int32_t* seq_lens,
                     int64_t* slot_mapping, int32_t* block_table, void* stream);

/*
 * pkv_write_int8 — the cache-write scatter into int8 caches.
 *
 * "vLLM 推理全流程深度解析", the closing note of the paged_attention section,
 * names KV-cache int8 quantisation as a decode speed-up without giving a
 * format.  This library's format: one fp32 scale per cache (per layer) and
 * symmetric codes, code = clamp(rne(x / scale), -127, 127), x the bf16 value
 * widened to fp32 and the division the IEEE fp32 one (a NaN value gives
 * code 0); the cached value stands for code * scale.
 *
 * Placement, padding, slot checks, arguments and alignment are those of
 * pkv_write; key_cache and value_cache are int8 [num_blocks, block_size,
 * num_kv_heads, head_size], contiguous, 16-byte aligned.  k_scale and
 * v_scale must be finite and positive (else PKV_ERR_ARG).
 */
int pkv_write_int8(const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride,
                   void* key_cache, void* value_cache, float k_scale, float v_scale,
                   int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                   int32_t head_size, const int64_t* slot_mapping, int64_t n_tokens,
                   void* stream);

/*
 * pkv_attention_int8 — pkv_attention over int8 caches written by
 * pkv_write_int8: the same formula with K_j = k_scale * code and V_j =
 * v_scale * code.  The products run on fp16 operands: the codes are exact
 * fp16 integers, the query is multiplied by scale * log2(e) * k_scale and
 * rounded to fp16 (so |q| * scale * k_scale * 1.4427 must stay below 65504,
 * the fp16 range; a larger product gives inf), the probabilities are fp16,
 * accumulation is fp32, and v_scale is applied to the output.  The codes
 * enter the products as code + 1152 (exact in fp16): the constant this adds
 * to a row's scores leaves its softmax unchanged, and the one it adds to the
 * output sums is subtracted at the end, both in fp32.
 *
 * Requests on the decode path only: a request whose query_len * (num_heads /
 * num_kv_heads) is at most 16 (32 when the group is larger than 16) —
 * single-token and short multi-token decodes.  A longer request is skipped
 * (its output rows are not written) and reported as
 * PKV_DEV_ERR_INT8_PREFILL.  Other arguments, layouts, checks and errors are
 * those of pkv_attention; k_scale and v_scale must be finite and positive.
 */
int pkv_attention_int8(const void* q, int64_t q_row_stride, int64_t q_rows, int32_t num_heads,
                       const void* key_cache, const void* value_cache, float k_scale,
                       float v_scale, int64_t num_blocks, int32_t block_size,
                       int32_t num_kv_heads, int32_t head_size, const int32_t* query_start_loc,
                       const int32_t* seq_lens, const int32_t* block_table,
                       int64_t block_table_width, int32_t num_reqs, float scale, void* out,
                       int64_t out_row_stride, void* stream);

/*
 * pkv_attention_noalloc — pkv_attention for callers that cannot allocate
 * device memory.  The pages this library follows have no counterpart to it.
 *
 * Some callers cannot call cudaMalloc: services that fix their device-memory
 * footprint at start-up and may not grow it later, hosts whose device memory
 * is handed out by an allocator of their own that the library must not
 * bypass, and latency-critical loops that cannot take the device-wide
 * synchronisation a cudaMalloc / cudaFree pair brings.  pkv_attention grows
 * its workspace with cudaMalloc on first use; this call runs the same kernels
 * but keeps the scratch (step plan, work lists, split-KV partials) in one
 * statically sized device array inside the library (32 MiB; every GPU that
 * loads the library holds it until the process exits), and allocates
 * nothing.
 *
 * Arguments, layouts, checks and results are those of pkv_attention.  A
 * batch whose scratch bound (the bound pkv_attention sizes its workspace by:
 * with S = ceil(16 * block_table_width / 256) splits and G = num_heads /
 * num_kv_heads, num_reqs * num_kv_heads * S split units of 32 bytes, plus
 * S * num_kv_heads * min(q_rows * G, num_reqs * (G <= 16 ? 16 : 32)) partial
 * rows of 520 bytes, plus the prefill and pair lists) exceeds 32 MiB is
 * refused with PKV_ERR_UNSUPPORTED before anything is enqueued.  Where the
 * array also holds pkv_attention's extra room for a small batch's one-wave
 * split (pkv_workspace_size), both calls make the same plan and give the same
 * bits; otherwise a small batch may be split into fewer, longer pieces and
 * the result agrees with pkv_attention's up to fp32 rounding.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture.
 * Every call shares the one array: calls whose kernels overlap on the GPU
 * (e.g. on two streams) race, and must be serialised by the caller.
 * Device-side metadata errors are skipped as in pkv_attention and reported in
 * an error word of this call's own, which pkv_get_error reads and clears
 * along with the other; pkv_last_error_string is not set: the return code
 * alone says which host check failed.
 */
int pkv_attention_noalloc(const void* q, int64_t q_row_stride, int64_t q_rows, int32_t num_heads,
                          const void* key_cache, const void* value_cache, int64_t num_blocks,
                          int32_t block_size, int32_t num_kv_heads, int32_t head_size,
                          const int32_t* query_start_loc, const int32_t* seq_lens,
                          const int32_t* block_table, int64_t block_table_width,
                          int32_t num_reqs, float scale, void* out, int64_t out_row_stride,
                          void* stream);

/*
 * pkv_reserve_workspace — sizes the current device's workspace for
 * pkv_attention calls with up to max_reqs requests, max_q_rows query rows,
 * block-table rows of up to block_table_width entries and this head
 * geometry, so that such calls allocate nothing (required before capturing
 * them in a CUDA graph: no allocation may happen while a stream is being
 * captured).  Also allocates the device error word.  Synchronous.  Returns
 * PKV_OK or an error code.
 */
int pkv_reserve_workspace(int32_t max_reqs, int64_t max_q_rows, int64_t block_table_width,
                          int32_t num_heads, int32_t num_kv_heads);

/*
 * pkv_workspace_size — what pkv_reserve_workspace would hold for these sizes
 * on a device with num_sms SMs (pkv_num_sms()), computed on the host alone
 * (no device is touched, nothing is allocated): the workspace's bytes and the
 * capacities of the step plan kept in it.  A plan never holds more than these
 * (the plan kernel reports PKV_DEV_ERR_CAPACITY and runs nothing if it
 * would); the split-KV chunk the plan chooses is sized for decode_workers
 * independent decode workers (decode_workers_int8 for int8 caches).
 * Returns PKV_OK, or PKV_ERR_ARG for negative sizes, a head count that is not
 * a multiple of num_kv_heads or num_sms <= 0.
 */
typedef struct {
  int64_t bytes;            /* device bytes of the workspace                   */
  int64_t decode_units;     /* split-KV decode work units                     */
  int64_t prefill_tiles;    /* prefill work entries (128-row query tiles)     */
  int64_t split_pairs;      /* (request, KV head) pairs whose splits merge    */
  int64_t partial_rows;     /* split-KV partial rows (130 fp32 values each)   */
  int32_t decode_workers;   /* decode workers of a bf16 call                  */
  int32_t decode_workers_int8; /* decode workers of an int8 call              */
} pkv_workspace_info;
int pkv_workspace_size(int32_t max_reqs, int64_t max_q_rows, int64_t block_table_width,
                       int32_t num_heads, int32_t num_kv_heads, int32_t num_sms,
                       pkv_workspace_info* info);

/*
 * pkv_get_error — synchronises `stream`, then returns the current device's
 * error words (an OR of PKV_DEV_ERR_* bits accumulated since the last read:
 * the allocating calls' word and pkv_attention_noalloc's) in *bits and
 * clears them.  Allocates nothing (a device no allocating call has used has
 * no word of its own yet and reports only pkv_attention_noalloc's).  Returns
 * PKV_OK or a host error code.
 */
int pkv_get_error(void* stream, int32_t* bits);

/* Text of the calling thread's last host-side error ("" if none). */
const char* pkv_last_error_string(void);

/* Number of SMs the library sizes its persistent grids for (current device). */
int pkv_num_sms(void);

/*
 * Tracing.  Not part of the step itself: a timing facility for benchmarks.
 * While tracing is on, every kernel the library launches is bracketed by a
 * pair of CUDA events recorded on the launch stream (do not capture traced
 * calls in a CUDA graph).  pkv_trace_read waits for those events, adds each
 * launch's duration to its kernel kind, copies up to n kinds of totals into
 * ms[] and launches[] (either may be NULL), clears the record and returns the
 * number of kinds (PKV_TRACE_KINDS).  Kinds: 0 cache write, 1 step plan,
 * 2 decode attention, 3 prefill attention, 4 split-KV merge, 5 step metadata.
 */
#define PKV_TRACE_KINDS 6
int pkv_trace_enable(int on);
int pkv_trace_read(double* ms, int64_t* launches, int n);

/* Total kernel launches issued by the library in this process. */
int64_t pkv_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
