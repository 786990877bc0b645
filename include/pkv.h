/*
 * pkv.h - C ABI of libpkv.so, PagedAttention over a flattened, variable-length
 * token batch on one NVIDIA GB300 (sm_103a).
 *
 * Pages cited (by title and section):
 *   [AI Infra]  "AI Infra入门干货总结：大模型是如何高效推理的"
 *   [抢占]      "vLLM 抢占机制源码精读"
 *   [调度实战]  "GPT-5 时代大模型推理调度系统深度实战"
 *   [Chunked]   "Chunked Prefill 与 Preemption"
 *   [显存调度]  "显存与调度" (book chapter 32)
 *
 * Conventions shared by every entry point
 *   - Return value: PKV_OK (0) on success, a negative PKV_E_* code otherwise;
 *     pkv_last_error() returns a message for the calling thread's last error.
 *     No C++ exception crosses this interface and no kernel traps.
 *   - Device entry points take DEVICE pointers owned by the caller and a
 *     cudaStream_t passed as `void* stream` (NULL = the legacy default
 *     stream).  They enqueue work asynchronously, never synchronise the
 *     stream and never allocate or free device memory.
 *   - Validation: with PKV_VALIDATE=1 in the environment, a device entry
 *     point that has an error word (the attention workspace's word 0, or
 *     the error_word argument when it is not NULL) waits for its stream
 *     after launching, reads that word (one device-to-host copy) and returns
 *     PKV_E_INVALID, naming the bits, if any is set.  The word is cumulative,
 *     so once set every later validated call fails until the caller clears
 *     it.  Off by default: no call then synchronises.
 *   - Host entry points (allocator, scheduler, metadata) take HOST pointers;
 *     opaque handles are owned by the library and released by *_destroy.
 *   - Float tensors are all float32 (PKV_F32) or all bfloat16 (PKV_BF16)
 *     within one call.  Index arrays are int32 except slot_mapping (int64).
 *   - Cache layout [AI Infra, section "Paged Attention"]: one layer's key
 *     cache and value cache are each [num_blocks, block_size, num_kv_heads,
 *     head_dim], contiguous, 16-byte aligned.  block_size must be 16;
 *     head_dim 64 or 128; num_heads a multiple of num_kv_heads.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_OK 0
#define PKV_E_INVALID (-1)      /* null pointer, bad size, stride or alignment */
#define PKV_E_UNSUPPORTED (-2)  /* a shape or dtype this build does not handle */
#define PKV_E_WORKSPACE (-3)    /* workspace missing or too small */
#define PKV_E_NO_BLOCKS (-4)    /* allocator: not enough free blocks */
#define PKV_E_STATE (-5)        /* allocator/scheduler call in the wrong state */
#define PKV_E_UNKNOWN_REQ (-6)  /* request id not known */
#define PKV_E_CUDA (-7)         /* a CUDA runtime call or launch failed */
#define PKV_E_CAPACITY (-8)     /* a request would exceed its block-table row */

typedef enum { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Bits the kernels set in a caller-visible device error word instead of
 * faulting; the offending access is skipped (reads yield zeros). */
#define PKV_ERR_BLOCK_ID 1u     /* block_table entry outside [0, num_blocks) */
#define PKV_ERR_SLOT 2u         /* slot_mapping entry >= num_blocks * block_size */
#define PKV_ERR_METADATA 4u     /* seq_len != num_computed + query_len, or a
                                   request longer than its block-table row */
#define PKV_ERR_TIMEOUT 8u      /* a bounded wait inside a kernel gave up */
#define PKV_ERR_POSITION 16u    /* a position outside [0, max_position) */

const char* pkv_last_error(void);
int pkv_version(void);

/* ------------------------------------------------------------------------
 * reshape_and_cache  [AI Infra, section "Paged Attention" (slot_idx rule)
 * and section "Attention Module" (QKV split -> RoPE -> reshape_and_cache
 * scatters the new K/V into the paged cache by slot_mapping)]
 *
 * For every token t < num_tokens with s = slot_mapping[t] >= 0:
 *   key_cache  [s / block_size][s % block_size][:][:] = key  [t][:][:]
 *   value_cache[s / block_size][s % block_size][:][:] = value[t][:][:]
 * A negative slot marks a padding token and is skipped.  A slot >=
 * num_blocks * block_size is skipped and sets PKV_ERR_SLOT in *error_word
 * (if error_word is not NULL).  The copy is bit-exact.
 *
 * key, value: device, [num_tokens, num_kv_heads, head_dim]; token t starts at
 *   element t * key_stride (value_stride); heads and dims are contiguous.
 *   Strides in elements; row bytes and strides must be multiples of 16 bytes.
 * key_cache, value_cache: device, layout above.
 * slot_mapping: device int64 [num_tokens].
 * error_word: device uint32 or NULL (bits are OR-ed in, never cleared).
 * ---------------------------------------------------------------------- */
int pkv_reshape_and_cache(const void* key, const void* value, int64_t key_stride,
                          int64_t value_stride, void* key_cache, void* value_cache,
                          const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                          int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                          int32_t dtype, uint32_t* error_word, void* stream);

/* ------------------------------------------------------------------------
 * reshape_and_cache + paged_attention_varlen in one call  [AI Infra,
 * section "Attention Module": the new K/V go into the paged cache by
 * slot_mapping, then attention reads every request's history, this step's
 * tokens included, through block_table]
 *
 * Same result as pkv_reshape_and_cache(key, value, ..., slot_mapping, error
 * word = workspace word 0) followed by pkv_paged_attention_varlen(...) on the
 * same stream.  key, value: device [num_tokens, num_kv_heads, head_dim] with
 * token strides key_stride / value_stride (elements, 16-byte multiples);
 * slot_mapping: device int64 [num_tokens]; every other argument as for
 * pkv_paged_attention_varlen.
 * When dtype is PKV_BF16 the two run as ONE kernel, so the step costs one
 * launch.  For a decode row (query length 1) the CTA that reads the
 * request's last block writes that token's K and V rows to
 * slot_mapping[token] and uses them in place of the cache's copy (no
 * read-after-write through memory).  For a row of query length > 1 each
 * prefill CTA writes the rows of its own query tiles, and the prefill CTAs
 * meet at a counter in the workspace header before any of them reads K or
 * V.  slot_mapping[token] must be the block table's slot of the token's
 * position (what pkv_build_slot_mapping produces): a token whose slot
 * differs still has its rows written at slot_mapping[token], and
 * PKV_ERR_METADATA is set.  Rows of a request whose metadata fails the
 * attention's checks (PKV_ERR_METADATA) are not written.  For PKV_F32
 * reshape_and_cache runs as its own kernel first.
 * ---------------------------------------------------------------------- */
int pkv_reshape_and_cache_paged_attention(
    const void* key, int64_t key_stride, const void* value, int64_t value_stride,
    const int64_t* slot_mapping, const void* q, int64_t q_stride, void* key_cache,
    void* value_cache, const int32_t* block_table, int32_t block_table_stride,
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* num_computed_tokens,
    float scale, void* out, int64_t out_stride, int64_t num_tokens, int32_t num_reqs,
    int64_t num_blocks, int32_t block_size, int32_t num_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t dtype, int32_t max_query_len, void* workspace,
    size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * rope_reshape_and_cache  [AI Infra, section "Attention Module (以标准GQA +
 * RoPE为例)": Q and K are rotated by RoPE after the QKV split, the rotation
 * being a block-diagonal rotation matrix applied element-wise with the row of
 * a precomputed cos_sin_cache [max_position_embeddings, rotary_dim] picked by
 * each token's position; then reshape_and_cache scatters K/V by slot_mapping]
 *
 * One pass that does both.  For every token t with p = positions[t]:
 *   row c = cos_sin_cache[p][0 : rotary_dim/2], s = [p][rotary_dim/2 : rotary_dim]
 *   pair i of a head is (a, b) = (2i, 2i+1) if is_neox == 0, else
 *   (i, i + rotary_dim/2); (x_a, x_b) -> (x_a c_i - x_b s_i, x_b c_i + x_a s_i);
 *   dimensions >= rotary_dim are unchanged.
 *   query[t][h]  <- rotated, in place, for every query head h;
 *   key_cache[slot] <- rotated key[t];  value_cache[slot] <- value[t]
 *     (slot = slot_mapping[t]; slot < 0 skips the scatter, slot >=
 *     num_blocks * block_size skips it and sets PKV_ERR_SLOT);
 *   key_out[t] <- rotated key[t] if key_out is not NULL (it may equal key).
 * A position outside [0, max_position) sets PKV_ERR_POSITION and the token is
 * left untouched (query not rotated, nothing scattered).  Arithmetic is fp32;
 * bf16 results are rounded to nearest even.
 *
 * positions, slot_mapping: device int64 [num_tokens].
 * query: device [num_tokens, num_heads, head_dim], token stride query_stride.
 * key, value (and key_out): device [num_tokens, num_kv_heads, head_dim], token
 *   strides key_stride / value_stride (key_out uses key_stride).
 * key_cache, value_cache: device [num_blocks, block_size, num_kv_heads,
 *   head_dim].  cos_sin_cache: device float32 [max_position, rotary_dim].
 * dtype (of query, key, value, caches): PKV_BF16 or PKV_F32.  Strides in
 *   elements.  All base pointers and token strides 16-byte aligned; head_dim
 *   * element size a multiple of 16 bytes; 0 < rotary_dim <= head_dim with
 *   rotary_dim / 2 (NeoX) or rotary_dim (interleaved) times the element size
 *   a multiple of 16 bytes; otherwise PKV_E_INVALID / PKV_E_UNSUPPORTED and
 *   nothing is launched.
 * The attention entry points may follow this call directly on the stream:
 *   they read query and the caches only after it has completed.
 * ---------------------------------------------------------------------- */
int pkv_rope_reshape_and_cache(const int64_t* positions, void* query, int64_t query_stride,
                               int32_t num_heads, const void* key, int64_t key_stride,
                               void* key_out, const void* value, int64_t value_stride,
                               void* key_cache, void* value_cache, const int64_t* slot_mapping,
                               const float* cos_sin_cache, int64_t max_position,
                               int32_t rotary_dim, int32_t is_neox, int64_t num_tokens,
                               int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                               int32_t head_dim, int32_t dtype, uint32_t* error_word,
                               void* stream);

/* ------------------------------------------------------------------------
 * copy_blocks  [显存调度, section "共享前缀会改变块的所有权": a shared block still
 * being written is copied first (copy-on-write); 抢占 and [Chunked]: swapping
 * moves a request's KV blocks between GPU and CPU memory]
 *
 * For i < num_pairs, with s = block_pairs[2i] and d = block_pairs[2i+1]:
 *   dst_key_cache[d] = src_key_cache[s];  dst_value_cache[d] = src_value_cache[s]
 * where a block is block_bytes contiguous bytes (block_size * num_kv_heads *
 * head_dim * element size).  Source and destination may be the same pool
 * (copy-on-write) or different ones, either in device memory or in mapped
 * pinned host memory (the GPU reads and writes it over the CPU-GPU link).
 * Destinations must be distinct, and within one pool no destination may
 * also be a source, so the copies are independent.  A pair with s outside
 * [0, src_num_blocks) or d outside [0, dst_num_blocks) is skipped and sets
 * PKV_ERR_BLOCK_ID in *error_word (if not NULL).  The copy is bit-exact.
 *
 * block_pairs: int32 [num_pairs][2], device or mapped host memory.
 * Pointers 16-byte aligned; block_bytes a positive multiple of 16.
 * ---------------------------------------------------------------------- */
int pkv_copy_blocks(const void* src_key_cache, const void* src_value_cache, void* dst_key_cache,
                    void* dst_value_cache, const int32_t* block_pairs, int32_t num_pairs,
                    int64_t src_num_blocks, int64_t dst_num_blocks, int64_t block_bytes,
                    uint32_t* error_word, void* stream);

/* ------------------------------------------------------------------------
 * paged_attention_varlen  [AI Infra, section "Attention Module (以标准GQA +
 * RoPE为例)": attention per request over its whole K/V history read through
 * block_table, requests separated by query_start_loc (cu_seqlens); Flash-
 * Decoding split-KV with log-sum-exp merge; Chunked, section "Chunked
 * Prefill：改变调度粒度，不改变 causal 结果": a chunk [a, b) sees keys j <= i]
 *
 * For request r with query rows t in [query_start_loc[r], query_start_loc[r+1])
 * the row's absolute position is p = num_computed_tokens[r] + (t -
 * query_start_loc[r]); for each query head h, with G = num_heads /
 * num_kv_heads and KV head g = h / G:
 *   out[t][h] = sum_{j <= p} softmax_j(scale * <q[t][h], K_r[j][g]>) V_r[j][g]
 * where K_r[j] is the cache row at slot block_table[r][j / block_size] *
 * block_size + j % block_size.  seq_lens[r] must equal num_computed_tokens[r]
 * + query length (the KV length after this step's reshape_and_cache), so the
 * keys of this step's own tokens must already be in the cache.
 * A bf16 call is one kernel: with only query-length-1 rows the split-KV
 * decode kernel; otherwise one persistent kernel whose CTAs split the SMs on
 * the device between the chunked-prefill tiles of the longer rows and the
 * split-KV decode of the query-length-1 rows.  Query length 0 contributes
 * no rows.
 *
 * q, out: [num_tokens, num_heads, head_dim], token stride q_stride /
 *   out_stride elements, heads and dims contiguous.  q is device memory.
 *   out is device memory, or pinned host memory that the device addresses
 *   at its host pointer (cudaHostAlloc / cudaMallocHost memory under unified
 *   addressing): the kernels only store to out and never read it, so a host
 *   buffer receives the result over the host link with no separate copy.
 *   The call does not check which kind out is.
 * block_table: device int32 [num_reqs, block_table_stride], row-major; only
 *   the first ceil(seq_lens[r] / block_size) entries of row r are read.
 * query_start_loc: device int32 [num_reqs + 1], non-decreasing, [0] = 0,
 *   [num_reqs] = num_tokens.  seq_lens, num_computed_tokens: device int32
 *   [num_reqs].
 * max_query_len: host hint, >= every request's query length, or 0 if
 *   unknown; a value of 1 launches the decode-only kernel (rows longer than
 *   one token are then not computed).
 * workspace: device scratch of at least pkv_attention_workspace_bytes()
 *   bytes for this batch, ZERO-FILLED BEFORE ITS FIRST USE; every call leaves
 *   it ready for the next one, including calls with a different number of
 *   requests (its layout follows the largest batch it can hold).  Word 0 is
 *   the error word (PKV_ERR_* bits, OR-ed in).  A call that reports
 *   PKV_ERR_TIMEOUT may leave its counters set: zero the workspace again
 *   before reusing it.  Two calls that overlap on the GPU must not share a
 *   workspace.
 * Ordering: the kernels are launched as programmatic dependents of the
 * kernel before the call on `stream`, so their set-up overlaps its tail.
 * They read q and the caches and write out and the workspace only after that
 * kernel has completed (reshape_and_cache may come directly before).  The
 * metadata arrays (block_table, query_start_loc, seq_lens,
 * num_computed_tokens) are read earlier: fill them by copies or kernels that
 * come before that kernel, not by the kernel directly before the call.
 * ---------------------------------------------------------------------- */
size_t pkv_attention_workspace_bytes(int32_t num_reqs, int32_t num_heads, int32_t head_dim);

int pkv_paged_attention_varlen(const void* q, int64_t q_stride, const void* key_cache,
                               const void* value_cache, const int32_t* block_table,
                               int32_t block_table_stride, const int32_t* query_start_loc,
                               const int32_t* seq_lens, const int32_t* num_computed_tokens,
                               float scale, void* out, int64_t out_stride, int64_t num_tokens,
                               int32_t num_reqs, int64_t num_blocks, int32_t block_size,
                               int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t dtype, int32_t max_query_len, void* workspace,
                               size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * rope_reshape_and_cache  [AI Infra, section "Attention Module (以标准GQA +
 * RoPE为例)": Q and K are rotated by RoPE after the QKV split, the rotation
 * being a block-diagonal rotation matrix applied element-wise with the row of
 * a precomputed cos_sin_cache [max_position_embeddings, rotary_dim] picked by
 * each token's position; then reshape_and_cache scatters K/V by slot_mapping]
 *
 * One pass that does both.  For every token t with p = positions[t]:
 *   row c = cos_sin_cache[p][0 : rotary_dim/2], s = [p][rotary_dim/2 : rotary_dim]
 *   pair i of a head is (a, b) = (2i, 2i+1) if is_neox == 0, else
 *   (i, i + rotary_dim/2); (x_a, x_b) -> (x_a c_i - x_b s_i, x_b c_i + x_a s_i);
 *   dimensions >= rotary_dim are unchanged.
 *   query[t][h]  <- rotated, in place, for every query head h;
 *   key_cache[slot] <- rotated key[t];  value_cache[slot] <- value[t]
 *     (slot = slot_mapping[t]; slot < 0 skips the scatter, slot >=
 *     num_blocks * block_size skips it and sets PKV_ERR_SLOT);
 *   key_out[t] <- rotated key[t] if key_out is not NULL (it may equal key).
 * A position outside [0, max_position) sets PKV_ERR_POSITION and the token is
 * left untouched (query not rotated, nothing scattered).  Arithmetic is fp32;
 * bf16 results are rounded to nearest even.
 *
 * positions, slot_mapping: device int64 [num_tokens].
 * query: device [num_tokens, num_heads, head_dim], token stride query_stride.
 * key, value (and key_out): device [num_tokens, num_kv_heads, head_dim], token
 *   strides key_stride / value_stride (key_out uses key_stride).
 * key_cache, value_cache: device [num_blocks, block_size, num_kv_heads,
 *   head_dim].  cos_sin_cache: device float32 [max_position, rotary_dim].
 * dtype (of query, key, value, caches): PKV_BF16 or PKV_F32.  Strides in
 *   elements.  All base pointers and token strides 16-byte aligned; head_dim
 *   * element size a multiple of 16 bytes; 0 < rotary_dim <= head_dim with
 *   rotary_dim / 2 (NeoX) or rotary_dim (interleaved) times the element size
 *   a multiple of 16 bytes; otherwise PKV_E_INVALID / PKV_E_UNSUPPORTED and
 *   nothing is launched.
 * The attention entry points may follow this call directly on the stream:
 *   they read query and the caches only after it has completed.
 * ---------------------------------------------------------------------- */
int pkv_rope_reshape_and_cache(const int64_t* positions, void* query, int64_t query_stride,
                               int32_t num_heads, const void* key, int64_t key_stride,
                               void* key_out, const void* value, int64_t value_stride,
                               void* key_cache, void* value_cache, const int64_t* slot_mapping,
                               const float* cos_sin_cache, int64_t max_position,
                               int32_t rotary_dim, int32_t is_neox, int64_t num_tokens,
                               int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                               int32_t head_dim, int32_t dtype, uint32_t* error_word,
                               void* stream);

/* ------------------------------------------------------------------------
 * copy_blocks  [显存调度, section "共享前缀会改变块的所有权": a shared block still
 * being written is copied first (copy-on-write); 抢占 and [Chunked]: swapping
 * moves a request's KV blocks between GPU and CPU memory]
 *
 * For i < num_pairs, with s = block_pairs[2i] and d = block_pairs[2i+1]:
 *   dst_key_cache[d] = src_key_cache[s];  dst_value_cache[d] = src_value_cache[s]
 * where a block is block_bytes contiguous bytes (block_size * num_kv_heads *
 * head_dim * element size).  Source and destination may be the same pool
 * (copy-on-write) or different ones, either in device memory or in mapped
 * pinned host memory (the GPU reads and writes it over the CPU-GPU link).
 * Destinations must be distinct, and within one pool no destination may
 * also be a source, so the copies are independent.  A pair with s outside
 * [0, src_num_blocks) or d outside [0, dst_num_blocks) is skipped and sets
 * PKV_ERR_BLOCK_ID in *error_word (if not NULL).  The copy is bit-exact.
 *
 * block_pairs: int32 [num_pairs][2], device or mapped host memory.
 * Pointers 16-byte aligned; block_bytes a positive multiple of 16.
 * ---------------------------------------------------------------------- */
int pkv_copy_blocks(const void* src_key_cache, const void* src_value_cache, void* dst_key_cache,
                    void* dst_value_cache, const int32_t* block_pairs, int32_t num_pairs,
                    int64_t src_num_blocks, int64_t dst_num_blocks, int64_t block_bytes,
                    uint32_t* error_word, void* stream);

/* ------------------------------------------------------------------------
 * paged_attention_varlen without a workspace.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory
 * where they run attention - an engine plugin whose enqueue step must not
 * allocate, a server that gave all free HBM to the KV block pool up front, or
 * a latency-critical loop that must avoid what cudaMalloc/cudaFree can cost.
 *
 * Same arguments and result as pkv_paged_attention_varlen, minus the
 * workspace.  The split-KV scratch lives in a 16 MiB array compiled into the
 * library (held by every GPU that loads it until the process exits); a batch
 * whose scratch (pkv_attention_workspace_bytes) exceeds 16 MiB is rejected
 * with PKV_E_WORKSPACE.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current): make that
 * first call before any stream capture begins.  Every call clears the
 * scratch's error word and split counters on `stream` before its kernels and
 * calls no allocating routine.  All calls share the array, so calls whose
 * work overlaps on the GPU race: serialise them.  error_word (device uint32,
 * or NULL) receives this call's PKV_ERR_* bits.
 * ---------------------------------------------------------------------- */
int pkv_paged_attention_varlen_noalloc(const void* q, int64_t q_stride, const void* key_cache,
                                       const void* value_cache, const int32_t* block_table,
                                       int32_t block_table_stride, const int32_t* query_start_loc,
                                       const int32_t* seq_lens, const int32_t* num_computed_tokens,
                                       float scale, void* out, int64_t out_stride,
                                       int64_t num_tokens, int32_t num_reqs, int64_t num_blocks,
                                       int32_t block_size, int32_t num_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                                       int32_t max_query_len, uint32_t* error_word, void* stream);

/* ------------------------------------------------------------------------
 * Step metadata (host)  [AI Infra, section "Paged Attention": slot_idx =
 * block_table[r][pos // block_size] * block_size + pos % block_size]
 *
 * slot_mapping[t] for every token of the flattened batch, requests in order:
 * request r's tokens sit at positions num_computed_tokens[r] + k, k <
 * query_start_loc[r+1] - query_start_loc[r].  All pointers are host memory;
 * block_table is [num_reqs, block_table_stride].  Returns PKV_E_INVALID if a
 * position's logical block is outside the row or num_tokens disagrees with
 * query_start_loc[num_reqs].
 * ---------------------------------------------------------------------- */
int pkv_build_slot_mapping(const int32_t* block_table, int32_t block_table_stride,
                           const int32_t* query_start_loc, const int32_t* num_computed_tokens,
                           int32_t num_reqs, int32_t block_size, int64_t* slot_mapping,
                           int64_t num_tokens);

/* ------------------------------------------------------------------------
 * Block allocator (host)  [显存调度, section "分配是词元计划的一部分" and
 * Fig. 32.2: reserve all new blocks of a plan atomically, execute, then
 * commit; failure or cancellation rolls the reservation back;
 * q_free + q_reserved + q_committed = q_capacity after every transition;
 * delta_q_i = ceil((T_i + s_i) / B) - ceil(T_i / B); section "从保留词元到物理块":
 * q_i = ceil(T_i / B), w_i = q_i B - T_i.  调度实战, section 5.3: the free list
 * is drained from its front and refilled at its back.]
 *
 * Blocks are ids 0..num_blocks-1; the free list starts in that order.
 * reserve() takes n (request id, new token count) pairs, computes each
 * request's delta_q_i from its committed token count T_i and either takes all
 * blocks (from the front of the free list, in pair order) or none
 * (PKV_E_NO_BLOCKS, state unchanged).  commit() makes the reservation part of
 * each request's table and adds s_i to T_i; rollback() returns the reserved
 * blocks to the front of the free list so it is exactly as before.
 * free_request() releases a request's committed blocks (block-table order),
 * then any of its reserved ones, to the back of the free list (with prefix
 * sharing, only blocks no other request holds; indexed ones become cached).
 * ---------------------------------------------------------------------- */
typedef struct pkv_alloc pkv_alloc;

typedef struct {
  int64_t capacity;        /* q_capacity */
  int64_t free;            /* q_free */
  int64_t reserved;        /* q_reserved (open plan) */
  int64_t committed;       /* q_committed = q_live, the union of the block sets */
  int64_t num_requests;    /* requests holding committed blocks */
  int64_t tail_waste;      /* sum of w_i over committed requests, in token slots */
  int64_t alloc_failures;  /* reserve() calls refused for lack of blocks */
  int64_t peak_used;       /* highest reserved + committed seen */
} pkv_alloc_stats;

pkv_alloc* pkv_alloc_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_req);
void pkv_alloc_destroy(pkv_alloc* a);
int pkv_alloc_reserve(pkv_alloc* a, int32_t n, const int32_t* req_ids, const int32_t* new_tokens);
int pkv_alloc_commit(pkv_alloc* a);
int pkv_alloc_rollback(pkv_alloc* a);
/* returns the number of blocks released (>= 0) or an error */
int pkv_alloc_free_request(pkv_alloc* a, int32_t req_id);
int pkv_alloc_get_stats(const pkv_alloc* a, pkv_alloc_stats* out);
/* committed + reserved blocks of req_id into out[0..capacity); returns the
 * count (0 for an unknown request) or an error if capacity is too small */
int pkv_alloc_table(const pkv_alloc* a, int32_t req_id, int32_t* out, int32_t capacity);
/* T_i: committed token count of req_id (0 if unknown) */
int64_t pkv_alloc_held_tokens(const pkv_alloc* a, int32_t req_id);
/* the free list, front first; returns its length or an error */
int pkv_alloc_free_list(const pkv_alloc* a, int32_t* out, int32_t capacity);
/* verifies conservation, q_i = ceil(T_i / B), that every block id is in
 * exactly one place, holder counts, and the prefix index's tree; PKV_OK or
 * PKV_E_STATE */
int pkv_alloc_check(const pkv_alloc* a);

/* ------------------------------------------------------------------------
 * Prefix sharing  [显存调度, section "共享前缀会改变块的所有权": identical KV
 * prefixes share physical blocks; q_live = |union of the requests' block
 * sets| <= q_capacity; r_p counts the active requests and the retaining cache
 * owner of block p, which is recycled only at r_p = 0; a prefix index finds
 * the longest reusable prefix and evicts reusable leaf entries under memory
 * pressure; full shared blocks are immutable, a shared block still being
 * written is copied first (copy-on-write).  Section "同时验证分配器与调度器":
 * shared blocks are recycled only after the last reference; an incompatible
 * namespace never hits.]
 *
 * The cache identity of a block is (namespace, the block it extends, its
 * block_size token ids): the namespace stands for model version, adapter,
 * position handling, cache format, modality and tenant.  Only full blocks
 * wholly inside a prompt registered with match_prefix are indexed, at the
 * commit that completes them.  A block held by no request but retained by the
 * index is "cached": q_free + q_reserved + q_live + q_cached = q_capacity,
 * where pkv_alloc_stats.committed is q_live.  reserve() evicts the oldest
 * cached blocks that no indexed block extends (to the back of the free list)
 * when a plan fits in q_free + q_cached but not in q_free; evictions stand
 * after a rollback.  A plan entry that writes into a partial last block held
 * by another request too gets one extra block: its table shows the copy, and
 * pkv_alloc_pending_copies lists (source, destination) for the device copy
 * (pkv_copy_blocks) that must run before the step writes; in plan order, the
 * last writer of such a block keeps the original.  free_request() returns
 * how many of the request's blocks no request holds any more.
 * ---------------------------------------------------------------------- */
typedef struct {
  int64_t lookups;         /* match_prefix calls */
  int64_t hits;            /* calls that matched at least one block */
  int64_t matched_tokens;  /* prefix tokens served from the index */
  int64_t evictions;       /* blocks evicted from the index */
  int64_t cow_copies;      /* copy-on-write copies committed */
  int64_t indexed;         /* blocks in the index */
  int64_t shared;          /* live blocks held by two or more requests */
  int64_t cached;          /* q_cached */
} pkv_prefix_stats;

/* Registers req_id's prompt (tokens[0..n)) for indexing and gives it the
 * longest indexed prefix of at most n - 1 tokens in namespace ns: its table
 * starts with those blocks and T_i = the matched token count, which is
 * returned.  req_id must hold nothing and no reservation may be open
 * (PKV_E_STATE). */
int pkv_alloc_match_prefix(pkv_alloc* a, int32_t req_id, uint64_t ns, const int32_t* tokens,
                           int32_t n);
/* The matched token count match_prefix would return, with no side effects;
 * *cached_blocks (if not NULL) receives how many of those blocks are cached
 * now (they leave q_cached when matched). */
int pkv_alloc_peek_prefix(const pkv_alloc* a, uint64_t ns, const int32_t* tokens, int32_t n,
                          int32_t* cached_blocks);
/* child_id starts with parent_id's committed blocks and token count (no
 * prompt registration); e.g. parallel samples of one prompt. */
int pkv_alloc_fork(pkv_alloc* a, int32_t parent_id, int32_t child_id);
/* (source, destination) block pairs of the open plan's copy-on-writes into
 * pairs[2 * capacity]; returns the count. */
int pkv_alloc_pending_copies(const pkv_alloc* a, int32_t* pairs, int32_t capacity);
int pkv_alloc_get_prefix_stats(const pkv_alloc* a, pkv_prefix_stats* out);
/* r_p of a block: requests holding it plus one if the index retains it */
int pkv_alloc_ref_count(const pkv_alloc* a, int32_t block);
/* the cached blocks, oldest release first; returns the count */
int pkv_alloc_cached_list(const pkv_alloc* a, int32_t* out, int32_t capacity);
/* q_free + q_cached: the blocks a plan may take */
int64_t pkv_alloc_available(const pkv_alloc* a);

/* ------------------------------------------------------------------------
 * Swapping  [抢占, sections "Swap 模式" (can_swap_out, swap_out returning
 * the GPU -> CPU block mapping, RUNNING -> SWAPPED) and "Swap-in 恢复流程"
 * (can_swap_in: ok / later / never; swap_in returning the CPU -> GPU mapping)]
 *
 * The allocator keeps a pool of num_cpu_blocks host block ids, a FIFO free
 * list like the GPU one.  swap_out(req) needs a free CPU block for each of
 * req's GPU blocks (else PKV_E_NO_BLOCKS, nothing changes), writes the
 * (GPU, CPU) pairs in table order, and releases the GPU blocks as
 * free_request() would (*released = how many no request holds any more).
 * swap_in_status: 0 ok, 1 later (not enough q_free + q_cached), 2 never
 * (more blocks than the GPU pool).  swap_in takes fresh GPU blocks from the
 * front of the free list (evicting cached blocks as reserve() does), writes
 * the (CPU, GPU) pairs and releases the CPU blocks.  Neither may be called
 * while a reservation is open.  The data itself moves with pkv_copy_blocks.
 * ---------------------------------------------------------------------- */
pkv_alloc* pkv_alloc_create_with_cpu_pool(int32_t num_blocks, int32_t block_size,
                                          int32_t max_blocks_per_req, int32_t num_cpu_blocks);
/* returns the pair count or an error */
int pkv_alloc_swap_out(pkv_alloc* a, int32_t req_id, int32_t* pairs, int32_t capacity,
                       int32_t* released);
int pkv_alloc_swap_in_status(const pkv_alloc* a, int32_t req_id);
int pkv_alloc_swap_in(pkv_alloc* a, int32_t req_id, int32_t* pairs, int32_t capacity);
/* CPU blocks of a swapped request (0 if it is not swapped); *tokens = its T_i */
int pkv_alloc_swapped_blocks(const pkv_alloc* a, int32_t req_id, int32_t* out, int32_t capacity,
                             int64_t* tokens);
int pkv_alloc_cpu_free_list(const pkv_alloc* a, int32_t* out, int32_t capacity);

/* ------------------------------------------------------------------------
 * Continuous-batching scheduler (host)  [AI Infra, sections "连续批处理" and
 * "附4：vLLM调度详细流程"; 抢占, sections "抢占的触发条件", "_schedule_running 中
 * 的抢占循环", "reset_state_for_recompute 的巧妙设计", "人工抢占测试"; 显存调度,
 * sections "分配是词元计划的一部分" and "分块预填充共享每轮预算"]
 *
 * One step: RUNNING requests head first get s_i = min(num_tokens -
 * num_computed, chunk_size, remaining budget); when a request's new blocks do
 * not fit, the tail of RUNNING is preempted by recompute (blocks freed,
 * num_computed = 0, moved to the front of WAITING) until it fits, or the
 * request preempts itself when it is the tail and the scan stops.  Only in a
 * step without preemption are WAITING requests admitted, head first, while
 * RUNNING < max_num_seqs, budget remains and their first chunk fits.  All new
 * blocks are then reserved at once (plan order).  finish_step(1) commits:
 * num_computed += s_i; a request that caught up samples one token and
 * either finishes (blocks freed) or grows num_tokens by one.
 * finish_step(0) rolls the reservation back.
 *
 * Swap preemption (preemption_mode = PKV_PREEMPT_SWAP)  [抢占, sections
 * "Swap 模式", "CPU swap 空间不足时的处理", "Swap-in 恢复流程"; 调度实战,
 * section 4.3]: a victim's blocks are swapped out to a pool of
 * num_cpu_blocks host blocks (it keeps num_computed and joins the back of
 * the SWAPPED queue); if the CPU pool is too small it is preempted by
 * recompute instead.  In a step without preemption the SWAPPED queue is
 * served head first before any admission: a request with more blocks than
 * the GPU pool finishes as ignored; one whose blocks plus its first chunk's
 * new blocks do not fit (or with no budget or seat left) stops the loop;
 * otherwise it is swapped in and scheduled at the back of RUNNING.  WAITING
 * requests are admitted only when nothing is left swapped.  The step's
 * block moves (pkv_sched_swaps) must be done with pkv_copy_blocks before
 * the step's kernels run: first GPU -> CPU, then CPU -> GPU.
 * ---------------------------------------------------------------------- */
typedef struct pkv_sched pkv_sched;

#define PKV_PREEMPT_RECOMPUTE 0
#define PKV_PREEMPT_SWAP 1

typedef struct {
  int32_t max_num_seqs;
  int32_t max_num_batched_tokens;   /* token budget K per step */
  int32_t chunk_size;               /* largest s_i per request per step */
  int32_t max_model_len;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_req;
  int32_t artificial_preempt_max;   /* test hook: at most this many forced failures */
  double artificial_preempt_prob;   /* test hook: 0 disables it */
  uint64_t artificial_seed;         /* splitmix64 seed of the test hook */
  int32_t preemption_mode;          /* PKV_PREEMPT_RECOMPUTE (0) or PKV_PREEMPT_SWAP */
  int32_t num_cpu_blocks;           /* host blocks for swapping (swap mode) */
} pkv_sched_config;

typedef struct {
  int32_t num_reqs;       /* requests in the plan */
  int32_t num_preempted;
  int32_t num_admitted;
  int32_t max_blocks;     /* longest block-table row among planned requests */
  int64_t num_tokens;     /* sum of s_i */
  int32_t max_query_len;  /* largest s_i */
  int32_t pad_;
} pkv_step_info;

typedef struct {
  int32_t status;         /* 0 waiting, 1 running, 2 finished, 3 swapped,
                             4 finished as ignored, -1 unknown */
  int32_t prompt_len;
  int32_t max_output;
  int32_t outputs;
  int64_t num_tokens;
  int64_t num_computed;
  int32_t preemptions;
  int32_t pad_;
} pkv_request_state;

pkv_sched* pkv_sched_create(const pkv_sched_config* cfg);
void pkv_sched_destroy(pkv_sched* s);
/* 1 accepted, 0 rejected (duplicate id, prompt >= max_model_len, or a
 * footprint that can never fit); the output target is clamped to
 * max_model_len - prompt_len */
int pkv_sched_add_request(pkv_sched* s, int32_t req_id, int32_t prompt_len, int32_t max_output);
/* As pkv_sched_add_request, with the prompt's token ids tokens[0..prompt_len)
 * in namespace ns: on admission the request is matched against the prefix
 * index (pkv_alloc_match_prefix) and starts at the matched token count; its
 * full prompt blocks are indexed as they are committed.  Returns 1 if
 * queued, 0 if rejected. */
int pkv_sched_add_request_tokens(pkv_sched* s, int32_t req_id, int32_t prompt_len,
                                 int32_t max_output, uint64_t ns, const int32_t* tokens);
int pkv_sched_step(pkv_sched* s, pkv_step_info* info);
/* plan entries, in batch order */
int pkv_sched_plan(const pkv_sched* s, int32_t* req_ids, int32_t* num_new_tokens,
                   int32_t* num_computed_before, int32_t capacity);
int pkv_sched_preempted(const pkv_sched* s, int32_t* out, int32_t capacity);
/* The open step's block moves: (GPU block, CPU block) pairs of its swap-outs
 * into out_pairs[2 * out_capacity], (CPU block, GPU block) pairs of its
 * swap-ins into in_pairs[2 * in_capacity]; *num_out / *num_in receive the
 * counts.  Either array may be NULL with capacity 0 to query the counts. */
int pkv_sched_swaps(const pkv_sched* s, int32_t* out_pairs, int32_t out_capacity,
                    int32_t* num_out, int32_t* in_pairs, int32_t in_capacity, int32_t* num_in);
/* Requests swapped out, swapped in and finished as ignored in the open step. */
int pkv_sched_swap_events(const pkv_sched* s, int32_t* swapped_out, int32_t* num_swapped_out,
                          int32_t* swapped_in, int32_t* num_swapped_in, int32_t* ignored,
                          int32_t* num_ignored, int32_t capacity);
int pkv_sched_admitted(const pkv_sched* s, int32_t* out, int32_t capacity);
/* the open step's kernel inputs, requests in plan order: block_table rows
 * (committed + reserved blocks, unused entries -1), query_start_loc [R+1],
 * seq_lens [R], num_computed_tokens [R], slot_mapping [num_tokens]; host
 * buffers, block_table_stride >= info.max_blocks */
int pkv_sched_build_metadata(const pkv_sched* s, int32_t* block_table, int32_t block_table_stride,
                             int32_t* query_start_loc, int32_t* seq_lens,
                             int32_t* num_computed_tokens, int64_t* slot_mapping);
/* commit (executed_ok != 0) or roll back; finished request ids go to
 * finished[0..capacity); returns how many finished */
int pkv_sched_finish_step(pkv_sched* s, int32_t executed_ok, int32_t* finished, int32_t capacity);
int pkv_sched_request(const pkv_sched* s, int32_t req_id, pkv_request_state* out);
int pkv_sched_queues(const pkv_sched* s, int32_t* running, int32_t* num_running, int32_t* waiting,
                     int32_t* num_waiting, int32_t capacity);
/* The SWAPPED queue (swap preemption), head first: *num ids go to
 * out[0..capacity); PKV_E_INVALID if capacity is smaller than the queue. */
int pkv_sched_swapped_queue(const pkv_sched* s, int32_t* out, int32_t* num, int32_t capacity);
/* counters: [0] total preemptions, [1] recomputed tokens, [2] finished requests,
 * [3] remaining artificial failures */
int pkv_sched_counters(const pkv_sched* s, int64_t* out4);
const pkv_alloc* pkv_sched_allocator(const pkv_sched* s);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H_ */
