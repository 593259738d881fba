/*
 * pkv.h -- C ABI of libpkv.so: attention over a paged KV cache on GB300 (sm_103a).
 *
 * The three operations are the attention block of a nano-vLLM style engine,
 * as the pages walk through it:
 *   - "vLLM 学习笔记 02：nano-vllm 源码逐段精读", layers/attention.py listing
 *     (store_kvcache, then flash_attn_varlen_func for prefill or
 *     flash_attn_with_kvcache for decode) and engine/model_runner.py listing
 *     (how slot_mapping, cu_seqlens, block_tables and context_lens are built);
 *   - "Nano-vLLM代码手撕笔记", sections "请求执行 – 输入序列预处理与context构建"
 *     and "请求执行 – run model" (the same steps with a worked example).
 *
 * Conventions shared by every entry point
 *   - Element type: bf16 for q, k, v, caches and outputs; the *_f16 entry
 *     points take IEEE fp16 for all of them instead (the experiment code in
 *     "Nano-vLLM代码手撕笔记", section "目录结构概览", builds the engine with
 *     dtype=torch.float16). Arithmetic is fp32 for both. pkv_store_kvcache
 *     copies 16-bit patterns and serves both types. Index arrays int32.
 *   - Supported shape: head_dim = 128, block_size = 256; prefill and decode
 *     also need num_kv_heads = 8 and num_heads = 16 (Qwen3-0.6B attention:
 *     16 query heads grouped 2 per kv head). Query head h reads kv head
 *     h / (num_heads / num_kv_heads).
 *   - Cache layout: k_cache, v_cache are [num_blocks, 256, num_kv_heads, 128]
 *     contiguous; token slot s is the row starting at element s*num_kv_heads*128.
 *   - Pointers are DEVICE pointers owned by the caller unless stated. The
 *     library allocates no memory, never synchronises a stream (except
 *     pkv_device_error) and launches only on the stream it is given, so every
 *     compute call can be captured in a CUDA graph.
 *   - Return value: PKV_OK (0) or a negative PKV_ERR_* detected on the host
 *     before anything is launched (then nothing is launched). Launch failures
 *     return PKV_ERR_CUDA.
 *   - Problems only visible on the device (a slot or block id outside the
 *     pool, inconsistent cu_seqlens, a context longer than max_context_len)
 *     never cause an out-of-bounds access: the offending work is skipped and a
 *     bit is OR-ed into a per-device error word that pkv_device_error reads.
 *     Outputs touched by skipped work are unspecified.
 *   - Every device-side wait is bounded in time; a wait that runs out sets
 *     PKV_DEVERR_TIMEOUT and the kernel returns instead of hanging.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side status codes. */
#define PKV_OK 0
#define PKV_ERR_NULL_POINTER (-1)      /* a required pointer is NULL */
#define PKV_ERR_UNSUPPORTED (-2)       /* head_dim/block_size/head counts outside the supported shape */
#define PKV_ERR_BAD_STRIDE (-3)        /* a row stride smaller than the row */
#define PKV_ERR_ALIGNMENT (-4)         /* pointer or stride not 16-byte aligned where a kernel needs it */
#define PKV_ERR_WORKSPACE (-5)         /* workspace NULL or smaller than the *_workspace_bytes query */
#define PKV_ERR_BAD_SIZE (-6)          /* a negative count or a size beyond the library's limits */
#define PKV_ERR_CUDA (-7)              /* a CUDA call or kernel launch failed */
#define PKV_ERR_DEVICE (-8)            /* current device is not a compute capability 10.3 GPU */
#define PKV_ERR_SCRATCH_LIMIT (-9)     /* pkv_decode_noalloc: the sizes need more than its built-in scratch */

/* Device-side error bits (pkv_device_error). */
#define PKV_DEVERR_BAD_SLOT 0x1u       /* slot_mapping entry not -1 and outside [0, num_slots) */
#define PKV_DEVERR_BAD_BLOCK 0x2u      /* block_tables entry outside [0, num_blocks) where it is read */
#define PKV_DEVERR_BAD_SEQLEN 0x4u     /* cu_seqlens not monotone, seqlen_k < seqlen_q, lengths above the
                                          declared maxima, or a context longer than the block table */
#define PKV_DEVERR_TIMEOUT 0x8u        /* a bounded device wait ran out */

/* Human-readable text for a PKV_* status. Never NULL. */
const char* pkv_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
int pkv_version(void);

/*
 * pkv_store_kvcache -- store_kvcache from layers/attention.py
 * ("vLLM 学习笔记 02：nano-vllm 源码逐段精读"; explained in
 * "Nano-vLLM代码手撕笔记", section "请求执行 – run model").
 *
 * For each token i < num_tokens with slot = slot_mapping[i] != -1:
 *   k_cache[slot, :, :] = k[i, :, :]   and   v_cache[slot, :, :] = v[i, :, :]
 * (num_kv_heads*head_dim elements each, a bit-exact copy). Tokens with
 * slot -1 (padding) are skipped.
 *
 *   k, v            [num_tokens, num_kv_heads, head_dim] 16-bit elements
 *                   (bf16 or fp16: the copy is bit-exact either way); heads and
 *                   dims contiguous within a row, rows k_row_stride /
 *                   v_row_stride ELEMENTS apart (>= num_kv_heads*head_dim;
 *                   e.g. 4096 for views of a fused qkv projection).
 *   k_cache,v_cache [num_slots, num_kv_heads, head_dim], same type, contiguous
 *                   (num_slots = num_blocks * block_size).
 *   slot_mapping    [num_tokens] int32.
 * Any head_dim and num_kv_heads are accepted. When every pointer is 16-byte
 * aligned and both row strides and the row length are multiples of 8
 * elements, 16-byte vector copies are used; otherwise 2-byte copies.
 * Duplicate slots in one call race (the pages never produce them); k/v must
 * not overlap the caches. Slots outside [0, num_slots) set PKV_DEVERR_BAD_SLOT.
 */
int pkv_store_kvcache(const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride,
                      void* k_cache, void* v_cache, const int32_t* slot_mapping, int32_t num_tokens,
                      int32_t num_kv_heads, int32_t head_dim, int64_t num_slots, cudaStream_t stream);

/*
 * pkv_prefill_varlen -- causal variable-length prefill attention, the
 * flash_attn_varlen_func call of layers/attention.py with causal=True.
 *
 * Sequence b owns query rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) of q and
 * Lk_b = cu_seqlens_k[b+1] - cu_seqlens_k[b] keys. Query row i of sequence b
 * sits at position Lk_b - Lq_b + i (prefix-cache hits and chunked prefill put
 * the new tokens at the end, engine/model_runner.py prepare_prefill) and
 * attends to keys 0..that position:
 *   out[row, h, :] = softmax(softmax_scale * q[row, h, :] . K[0..p, h/G, :]^T) V[0..p, h/G, :]
 * with fp32 logits and accumulation, bf16 output.
 *
 * Key source:
 *   block_tables != NULL  (prefix-cache mode): key t of sequence b is slot
 *     block_tables[b*block_table_stride + t/256]*256 + t%256 of k_cache/v_cache
 *     ([num_blocks, 256, 8, 128]). The caller runs pkv_store_kvcache for the
 *     new tokens first, on the same stream, as layers/attention.py does.
 *     Entries past ceil(Lk_b/256) are never read.
 *   block_tables == NULL  (no prefix hit): key t of sequence b is row
 *     cu_seqlens_k[b] + t of k/v ([total_k, 8, 128], rows kv_row_stride
 *     elements apart); k_cache/v_cache are ignored.
 *
 *   q    [total_q, 16, 128] bf16, rows q_row_stride elements apart.
 *   out  [total_q, 16, 128] bf16 contiguous; every row of every sequence written.
 *   total_q, total_k  row counts of q and of contiguous k/v (the tensors'
 *        first dimension; total_k is ignored in prefix-cache mode). Tiles are
 *        fetched by tensor-memory-access copies, which need the exact extent.
 *   cu_seqlens_q/k [num_seqs+1] int32, max_seqlen_q/k their largest lengths;
 *        cu_seqlens_q[num_seqs] <= total_q and, in contiguous mode,
 *        cu_seqlens_k[num_seqs] <= total_k.
 * q, k, v, k_cache, v_cache must be 16-byte aligned and their row strides
 * multiples of 8 elements (tensor-memory-access rules).
 *
 * workspace: NULL, or a tile plan -- workspace_bytes/4 int32 items written by
 *   pkv_prefill_plan for these cu_seqlens and copied to device memory (4-byte
 *   aligned, workspace_bytes a multiple of 4, at most 2^28 items). Without a
 *   plan every (128-row query tile, sequence) pair up to max_seqlen_q is
 *   launched, longest key ranges first, and the tiles past a sequence's end
 *   exit at once; with a plan exactly the plan's items are launched, in its
 *   order. Items past a sequence's end are skipped, items naming a sequence
 *   >= num_seqs are skipped and set PKV_DEVERR_BAD_SEQLEN (a stale plan gives
 *   missing rows, never an out-of-bounds access); results are identical with
 *   and without a plan.
 */
int pkv_prefill_varlen(const void* q, int64_t q_row_stride, int32_t total_q, const void* k, const void* v,
                       int64_t kv_row_stride, int32_t total_k, const void* k_cache, const void* v_cache,
                       int32_t num_blocks,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t max_seqlen_q,
                       int32_t max_seqlen_k, const int32_t* block_tables, int32_t block_table_stride,
                       int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, float softmax_scale, void* out, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream);

/*
 * pkv_prefill_varlen_f16 -- pkv_prefill_varlen with IEEE fp16 q, k, v,
 * caches and output (fp32 logits and accumulation; P is rounded to fp16
 * for the probability-times-value product). Arguments, layouts and errors
 * as for pkv_prefill_varlen.
 */
int pkv_prefill_varlen_f16(const void* q, int64_t q_row_stride, int32_t total_q, const void* k, const void* v,
                           int64_t kv_row_stride, int32_t total_k, const void* k_cache, const void* v_cache,
                           int32_t num_blocks, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t* block_tables,
                           int32_t block_table_stride, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, float softmax_scale, void* out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes pkv_prefill_varlen(_f16) needs for these sizes (0: none;
 * an optional tile plan may be passed in its place). */
size_t pkv_prefill_workspace_bytes(int32_t num_seqs, int32_t max_seqlen_q, int32_t num_heads);

/*
 * pkv_prefill_plan -- host-side tile plan for pkv_prefill_varlen(_f16), built
 * once per engine step from the host copies of the step's cu_seqlens (the
 * pages' prepare_prefill builds them on the host) and reused by every layer.
 *
 * Writes one int32 per (128-row query tile qt, sequence b) pair that holds
 * query rows, encoded (qt << 16) | b, ordered by the number of 128-key tiles
 * the query tile attends to, most first (ties: lower b, then higher qt), so the
 * longest tiles start first. h_cu_seqlens_q / h_cu_seqlens_k: [num_seqs+1]
 * host arrays. h_items: host output with room for `capacity` items; the
 * number needed is sum over b of ceil(Lq_b / 128) <= total_q/128 + num_seqs.
 * Returns the number of items (>= 0), or PKV_ERR_NULL_POINTER, or
 * PKV_ERR_BAD_SIZE (num_seqs outside [0, 65535], lengths not monotone or
 * Lk_b < Lq_b, a sequence of 2^22 or more query rows, or capacity too small).
 */
int32_t pkv_prefill_plan(const int32_t* h_cu_seqlens_q, const int32_t* h_cu_seqlens_k, int32_t num_seqs,
                         int32_t* h_items, int32_t capacity);

/*
 * pkv_decode -- single-query GQA decode attention over the paged cache, the
 * flash_attn_with_kvcache(q.unsqueeze(1), k_cache, v_cache,
 * cache_seqlens=context_lens, block_table=block_tables, causal=True) call of
 * layers/attention.py.
 *
 * For sequence b and query head h, with ctx = context_lens[b] (the length
 * including the token just stored, engine/model_runner.py prepare_decode):
 *   out[b, h, :] = softmax(softmax_scale * q[b, h, :] . K_b[0..ctx-1]^T) V_b[0..ctx-1]
 * where key t of sequence b is slot block_tables[b*block_table_stride + t/256]*256
 * + t%256 of the kv head h/2. Rows with ctx == 0 (graph padding) get zeros.
 * Entries of block_tables past ceil(ctx/256) are never read (they may be -1
 * or stale).
 *
 *   q       [num_seqs, 16, 128] bf16, rows q_row_stride elements apart (>= 2048).
 *   out     [num_seqs, 16, 128] bf16 contiguous.
 *   max_context_len  upper bound on every context_lens[b] (e.g. max_model_len
 *           when the call is captured in a graph and replayed with new lengths);
 *           sizes the split-KV grid. Longer contexts set PKV_DEVERR_BAD_SEQLEN
 *           and give zeros.
 *   workspace  >= pkv_decode_workspace_bytes(num_seqs, num_heads, max_context_len)
 *           bytes of device memory, ZERO-FILLED ONCE before its first use; every
 *           call leaves it ready for the next. Calls that share a workspace
 *           must not overlap in time (same stream, or ordered).
 */
int pkv_decode(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
               int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
               const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
               int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale, void* out,
               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * pkv_store_decode -- store_kvcache fused into the decode step
 * (layers/attention.py runs store_kvcache, then flash_attn_with_kvcache, on
 * the same slot_mapping; "vLLM 学习笔记 02：nano-vllm 源码逐段精读").
 *
 * Same result as pkv_store_kvcache(k, k_row_stride, v, v_row_stride, k_cache,
 * v_cache, slot_mapping, num_seqs, ...) followed by pkv_decode(...), in one
 * launch: the CTA that streams sequence b's last block first writes the new
 * K/V row there. It requires what engine/model_runner.py prepare_decode
 * produces: slot_mapping[b] is -1 (padding, nothing stored) or the slot of
 * position context_lens[b]-1 of sequence b. Any other slot is not stored and
 * sets PKV_DEVERR_BAD_SLOT.
 *   k, v  [num_seqs, 8, 128] bf16, rows k_row_stride / v_row_stride elements
 *         apart, 16-byte aligned, strides multiples of 8 elements.
 * Every other argument is as for pkv_decode.
 */
int pkv_store_decode(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
                     int64_t v_row_stride, const int32_t* slot_mapping, void* k_cache, void* v_cache,
                     int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                     const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale, void* out,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * pkv_decode_f16 / pkv_store_decode_f16 -- pkv_decode and pkv_store_decode
 * with IEEE fp16 q, k, v, caches and output (fp32 arithmetic). Arguments,
 * layouts, workspace and errors as for the bf16 calls; a workspace may be
 * shared between bf16 and fp16 calls under the same ordering rule.
 */
int pkv_decode_f16(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
                   int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                   const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                   int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale, void* out,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);
int pkv_store_decode_f16(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
                         int64_t v_row_stride, const int32_t* slot_mapping, void* k_cache, void* v_cache,
                         int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale,
                         void* out, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes pkv_decode, pkv_store_decode and their _f16 forms need for these sizes. */
size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t max_context_len);

/*
 * pkv_decode_noalloc -- pkv_decode for callers that cannot allocate device
 * memory. The pages have no counterpart to this entry point: it exists for
 * users of this library, not for the method.
 *
 * Who needs it: an engine that sized its KV-cache pool to take all device
 * memory left after start-up, a plug-in whose host process owns the only
 * device allocator, or a latency-critical loop that must not call cudaMalloc
 * because it can synchronise the device. None of them can hand pkv_decode a
 * workspace.
 *
 * Same arguments and result as pkv_decode (bf16 only; there is no fp16 form),
 * without the workspace: the split-KV scratch lives in a fixed array of
 * PKV_DECODE_NOALLOC_SCRATCH_BYTES that is part of the library's device
 * image, reserved on every GPU that loads the library and held until the
 * process exits. The call allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine).
 *   - Limit: sizes with pkv_decode_workspace_bytes(num_seqs, num_heads,
 *     max_context_len) > PKV_DECODE_NOALLOC_SCRATCH_BYTES are rejected with
 *     PKV_ERR_SCRATCH_LIMIT before anything is launched (e.g. 256 sequences
 *     with max_context_len 4096 fit; 512 sequences fit up to 2048). Every
 *     other argument error pkv_decode reports is reported too, also before
 *     anything is queued on the stream.
 *   - The call passes the kernel the array's device address, which it asks
 *     the runtime for (cudaGetSymbolAddress) with the calling thread's device
 *     current, and caches per device and context. The first call on each
 *     device makes that lookup: make it before any stream capture.
 *   - Every call shares the one array and leaves its contents behind; each
 *     call first clears (cudaMemsetAsync on `stream`) the part that must start
 *     at zero. Calls whose execution overlaps on the GPU (different streams
 *     without ordering, or several host threads) race on the array and give
 *     wrong results: order them.
 */
#define PKV_DECODE_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int pkv_decode_noalloc(const void* q, int64_t q_row_stride, const void* k_cache, const void* v_cache,
                       int32_t num_blocks, const int32_t* block_tables, int32_t block_table_stride,
                       const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t max_context_len, float softmax_scale,
                       void* out, cudaStream_t stream);

/*
 * pkv_build_prefill_metadata / pkv_build_decode_metadata -- the per-step index
 * preparation of engine/model_runner.py (prepare_prefill, prepare_decode in
 * "vLLM 学习笔记 02：nano-vllm 源码逐段精读"; worked example in
 * "Nano-vLLM代码手撕笔记", section "请求执行 – 输入序列预处理与context构建"),
 * computed on the GPU from what the scheduler has per sequence, so no
 * per-token host loop and no per-token host-to-device copy is needed.
 * Bit-identical to the host definition. A token whose block-table entry is
 * outside [0, num_blocks) gets slot -1 and sets PKV_DEVERR_BAD_BLOCK.
 *
 * Prefill: sequence b computes positions [num_cached_tokens[b],
 * num_cached_tokens[b] + num_scheduled_tokens[b]).
 *   cu_seqlens_q[num_seqs+1]  prefix sums of num_scheduled_tokens
 *   cu_seqlens_k[num_seqs+1]  prefix sums of num_cached + num_scheduled
 *   max_seqlens[2]            {max_seqlen_q, max_seqlen_k} (device; the
 *                             attention calls accept any upper bounds instead)
 *   slot_mapping[capacity], positions[capacity] (int64)  one entry per new
 *                             token, sequence by sequence; tokens beyond
 *                             `capacity` are not written (PKV_DEVERR_BAD_SEQLEN).
 * Decode: num_tokens[b] = len(seq) including the token being stored;
 *   slot_mapping[b] = slot of position len-1, context_lens[b] = len,
 *   positions[b] = len-1; rows with len 0 are padding (slot -1, context 0).
 * All arrays are int32 device arrays except positions (int64, as the pages'
 * torch.int64 positions). block_tables is [num_seqs, block_table_stride], -1 padded.
 */
int pkv_build_prefill_metadata(const int32_t* num_cached_tokens, const int32_t* num_scheduled_tokens,
                               const int32_t* block_tables, int32_t block_table_stride, int32_t num_blocks,
                               int32_t num_seqs, int32_t capacity, int32_t* cu_seqlens_q, int32_t* cu_seqlens_k,
                               int32_t* max_seqlens, int32_t* slot_mapping, int64_t* positions, cudaStream_t stream);
int pkv_build_decode_metadata(const int32_t* num_tokens, const int32_t* block_tables, int32_t block_table_stride,
                              int32_t num_blocks, int32_t num_seqs, int32_t* slot_mapping, int32_t* context_lens,
                              int64_t* positions, cudaStream_t stream);

/*
 * pkv_device_error -- read (and optionally clear) the current device's
 * error word (PKV_DEVERR_* bits OR-ed by every kernel of this library since
 * the last clear). Synchronises `stream`, so do not call it inside a graph
 * capture. bits may be NULL when only clearing.
 */
int pkv_device_error(uint32_t* bits, int clear, cudaStream_t stream);

/*
 * pkv_selftest_wait_timeout -- failure-detection self test: launches one
 * block that waits on a barrier nothing will ever complete, with the given
 * bound in nanoseconds (clamped to [1000, 100000000]). The wait must give
 * up, set PKV_DEVERR_TIMEOUT and return; the GPU stays usable.
 */
int pkv_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
