/*
 * kvpaged.h - C ABI of the GB300 paged KV-cache attention library (libkvpaged.so).
 *
 * The three calls are the data-parallel hot path of one attention layer of a
 * nano-vLLM-style serving engine, as the engine's ModelRunner feeds it:
 *
 *   kv_store             scatter the step's new K/V rows into the paged cache
 *   attn_prefill_varlen  varlen causal prefill over packed sequences, with a
 *                        prefix cache (only the uncached suffix is queried)
 *   attn_decode_paged    one query token per sequence over its paged history
 *   attn_decode_paged_append  kv_store of the new rows + attn_decode_paged, fused
 *   attn_prefill_varlen_append  kv_store of the new rows + attn_prefill_varlen, fused
 *   attn_mixed_step      a step of prefill chunks and decode rows, the two side by side
 *
 * Sources: "nano-vLLM-1" (Senjl's Digital Garden), ModelRunner sections
 * "3. KV cache 分配", "4. prefill 输入打包", "5. deocde 输入打包" and BlockManager
 * section "3. 核心方法一：分配 (allocate)"; "Nano vLLM 解读（5）：解析 ModelRunner",
 * sections on the KV cache tensor and "FlashAttention Kernel 函参准备";
 * "【nano-vllm 学习】04 - 自顶向下的引擎调度层源码学习2", section
 * "KV-Cache … 是什么？" (softmax(QK^T/sqrt(d_k))V with a causal mask).
 *
 * Conventions shared by every call
 * --------------------------------
 * - bf16 tensors are passed as pointers to their raw 16-bit patterns
 *   (kvp_bf16).  Every pointer is a DEVICE pointer owned by the caller; the
 *   library keeps no pointer after a call returns and allocates no memory
 *   (scratch space, where a call needs it, is passed in as `workspace`).
 * - Strides are in elements.  A "row" is one token: [heads, head_dim] contiguous.
 * - One layer's caches: k_cache and v_cache are the views kv_cache[0, layer]
 *   and kv_cache[1, layer] of the engine's [2, layers, num_blocks, block_size,
 *   num_kv_heads, head_dim] tensor, i.e. each is [num_blocks, block_size,
 *   num_kv_heads, head_dim] and contiguous.  Token slot s lives at block
 *   s / block_size, offset s % block_size.
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *   default stream) and runs on the current CUDA device.
 * - Return value: KVP_OK, or a negative KVP_ERR_* code when the call was
 *   rejected before launch (nothing was enqueued) or the launch failed.
 *   kvp_last_error() describes the last failure of the calling thread.
 * - Contents of device-side metadata (slot values, block ids, context
 *   lengths) are range-checked inside the kernels: an out-of-range value is
 *   never dereferenced; the kernel records KVP_ERR_DEVICE_DATA in a device
 *   status word that kvp_device_status() reads back.  Waits inside the kernels
 *   are bounded; a wait that times out records KVP_ERR_DEVICE_TIMEOUT.
 * - Head mapping (GQA): query head h reads kv head h / (num_heads /
 *   num_kv_heads).
 * - Arithmetic: bf16 inputs, fp32 accumulation, softmax in fp32 (base-2
 *   exponentials with log2(e) folded into the scale), bf16 outputs.
 */
#ifndef KVPAGED_H
#define KVPAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvp_bf16;               /* raw bf16 bit pattern */
typedef struct CUstream_st *kvp_stream_t; /* same type as cudaStream_t */

enum {
  KVP_OK = 0,
  KVP_ERR_INVALID_ARG = -1,    /* null/misaligned pointer, bad size or stride */
  KVP_ERR_UNSUPPORTED = -2,    /* shape outside what the kernels implement */
  KVP_ERR_WORKSPACE = -3,      /* workspace missing or too small */
  KVP_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed */
  KVP_ERR_DEVICE_TIMEOUT = -5, /* (device status) a bounded in-kernel wait expired */
  KVP_ERR_DEVICE_DATA = -6     /* (device status) out-of-range slot / block id / length */
};

/* Message for the calling thread's last failed call ("" if none). */
const char *kvp_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int kvp_version(void);

/* Reads and clears the device status word of the current device (a blocking
 * device-to-host read; it synchronizes with the device).  Returns KVP_OK,
 * KVP_ERR_DEVICE_TIMEOUT, KVP_ERR_DEVICE_DATA, or KVP_ERR_CUDA if the read
 * itself failed. */
int kvp_device_status(void);

/* Self-test of the bounded-wait failure path (no fault, no hang): launches one
 * thread on `stream` that waits on a shared-memory mbarrier through the wait
 * every kernel uses, with a 2 ms limit instead of the kernels' 2 s.
 *   arrive = 0  nothing arrives: the wait expires, KVP_ERR_DEVICE_TIMEOUT is
 *               recorded in the device status word, the kernel returns.
 *   arrive != 0 the thread arrives first: the wait succeeds, nothing recorded.
 * Returns KVP_OK once launched, or KVP_ERR_CUDA.  Read the outcome with
 * kvp_device_status() after the stream has finished. */
int kvp_selftest_wait(int arrive, kvp_stream_t stream);

/*
 * kv_store - slot-mapped scatter of the step's new K/V rows.
 *
 * For every t < num_tokens with s = slot_mapping[t] >= 0:
 *     k_cache[s / block_size][s % block_size][:][:] = k[t][:][:]
 *     v_cache[s / block_size][s % block_size][:][:] = v[t][:][:]
 * bit-exactly.  A slot of -1 (the engine's padding for CUDA-graph batches)
 * writes nothing.  Source: "nano-vLLM-1" ModelRunner "4. prefill 输入打包" /
 * "5. deocde 输入打包" (slot_mapping); "Nano vLLM 解读（5）" prepare_prefill.
 *
 *   k, v            [num_tokens, num_kv_heads, head_dim] bf16, row strides
 *                   k_stride_tok / v_stride_tok (>= num_kv_heads*head_dim)
 *   slot_mapping    [num_tokens] int32; values in [-1, num_blocks*block_size)
 *   k_cache,v_cache [num_blocks, block_size, num_kv_heads, head_dim] bf16
 * num_tokens == 0 is a no-op.  Slots must be distinct within one call (the
 * engine never repeats one); a slot >= num_blocks*block_size or < -1 is
 * skipped and flagged as KVP_ERR_DEVICE_DATA.
 */
int kv_store(const kvp_bf16 *k, const kvp_bf16 *v, int64_t k_stride_tok, int64_t v_stride_tok,
             const int32_t *slot_mapping, int64_t num_tokens, kvp_bf16 *k_cache,
             kvp_bf16 *v_cache, int64_t num_blocks, int block_size, int num_kv_heads,
             int head_dim, kvp_stream_t stream);

/*
 * kv_copy_blocks - copy-on-write copies of whole cache blocks.
 *
 * For every pair i < num_pairs with src = block_mapping[2i] and
 * dst = block_mapping[2i+1], and every plane p < num_planes:
 *     cache[p * plane_stride + dst * block_elems + e] =
 *         cache[p * plane_stride + src * block_elems + e],   e < block_elems
 * bit-exactly.  A plane is one layer's K or one layer's V cache: the engine's
 * [2, layers, num_blocks, block_size, num_kv_heads, head_dim] tensor is
 * num_planes = 2 * layers planes with plane_stride = num_blocks * block_elems
 * and block_elems = block_size * num_kv_heads * head_dim.
 * Source: "【nano-vllm 学习】04 - 自顶向下的引擎调度层源码学习2", section
 * "场景优化1：Parallel Memory Shared": when a sequence must append into a
 * block it shares with others (reference count > 1), the engine gives it a
 * new physical block holding a copy of the shared one (copy on write).
 *
 *   cache          bf16 base of plane 0 (device)
 *   num_planes     >= 1
 *   plane_stride   elements from one plane to the next (>= num_blocks*block_elems)
 *   num_blocks     blocks per plane
 *   block_elems    elements per block
 *   block_mapping  [num_pairs, 2] int32 (src, dst), device
 * Destinations must be distinct, and no destination may be the source of
 * another pair (the engine copies into freshly allocated blocks); otherwise
 * the result is undefined.  num_pairs == 0 is a no-op.  A src or dst outside
 * [0, num_blocks) skips that pair and sets KVP_ERR_DEVICE_DATA.  The 16-byte
 * path is taken when cache, plane_stride and block_elems are 16-byte / 8-element
 * aligned; other layouts are copied element by element.
 */
int kv_copy_blocks(kvp_bf16 *cache, int64_t num_planes, int64_t plane_stride, int64_t num_blocks,
                   int64_t block_elems, const int32_t *block_mapping, int64_t num_pairs,
                   kvp_stream_t stream);

/*
 * attn_prefill_varlen - causal attention over sequences packed back to back.
 *
 * Sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and has
 * k_len_b = cu_seqlens_k[b+1] - cu_seqlens_k[b] keys; its first
 * c_b = k_len_b - q_len_b tokens are a cached prefix, so query row i is the
 * token at absolute position c_b + i and attends to keys 0 .. c_b + i:
 *     out[row, h] = sum_j softmax_j(q[row, h] . k_j * softmax_scale) v_j
 * Source: "Nano vLLM 解读（5）" prepare_prefill (cu_seqlens_q/k, max_seqlen_q/k,
 * block_tables only on a prefix hit); "nano-vLLM-1" "4. prefill 输入打包";
 * "【nano-vllm 学习】04 …" causal mask.
 *
 *   q               [total_q, num_heads, head_dim] bf16, row stride q_stride_tok;
 *                   total_q (= cu_seqlens_q[num_seqs]) bounds every read of q
 *   block_tables    NULL: keys/values are the packed rows k, v
 *                   [total_k, num_kv_heads, head_dim] (row stride
 *                   kv_stride_tok; total_k = cu_seqlens_k[num_seqs]) and
 *                   every q_len must equal its k_len;
 *                   else [num_seqs, max_blocks_per_seq] int32 (right-padded
 *                   with -1): keys/values are read from k_cache / v_cache
 *                   through the block table (the step's own rows must already
 *                   have been written there by kv_store)
 *   cu_seqlens_q/k  [num_seqs + 1] int32 prefix sums, cu[0] = 0
 *   max_seqlen_q/k  upper bounds of q_len / k_len over the batch
 *   positions       optional [total_q] int64 (may be NULL); not read by the
 *                   kernels (the causal offset is c_b + i)
 *   out             [total_q, num_heads, head_dim] bf16, row stride out_stride_tok
 * Supported: head_dim in {64, 128}; num_heads / num_kv_heads in {1, 2, 4, 8};
 * block_size 16 * 2^k (16..4096).  q_len = 0 for a sequence is allowed (no
 * rows).  No workspace: the CTAs share their work through a counter in one
 * of 64 library-owned slots per device (one slot per call, in turn), so at
 * most 64 attn_prefill_varlen calls may be in flight on a device at the same
 * time (calls on one stream follow each other and are always fine; CUDA-graph
 * replays of a captured call are fine too).
 */
int attn_prefill_varlen(const kvp_bf16 *q, int64_t q_stride_tok, int64_t total_q,
                        const kvp_bf16 *k, const kvp_bf16 *v, int64_t kv_stride_tok,
                        int64_t total_k, const kvp_bf16 *k_cache,
                        const kvp_bf16 *v_cache, int64_t num_blocks, int block_size,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                        int max_seqlen_q, int max_seqlen_k, int num_seqs,
                        const int64_t *positions, int num_heads, int num_kv_heads, int head_dim,
                        float softmax_scale, kvp_bf16 *out, int64_t out_stride_tok,
                        kvp_stream_t stream);

/*
 * attn_prefill_varlen_append - the prefill step of one layer in one launch:
 * kv_store(k, v, slot_mapping) followed by attn_prefill_varlen.
 *
 * Source: "nano-vLLM-1" "4. prefill 输入打包" (slot_mapping lists the slots of
 * the uncached tokens, one per query row; the keys of a prefix hit are read
 * through block_tables) and "Nano vLLM 解读（5）" (the store into the KV cache
 * comes before the attention of the same layer).
 *
 *   k, v            [total_q, num_kv_heads, head_dim] bf16, row stride
 *                   kv_stride_tok (a multiple of 8 elements, 16-byte aligned):
 *                   the new key / value of query row t
 *   slot_mapping    [total_q] int32: cache slot of row t, -1 = no store
 *   k_cache/v_cache written at the slots of slot_mapping; in paged mode also
 *                   read through block_tables
 *   block_tables    NULL: packed mode, keys/values are the rows k, v
 *                   themselves (every k_len must equal its q_len; a sequence
 *                   that breaks this records KVP_ERR_DEVICE_DATA and gets no
 *                   output); else paged mode as in attn_prefill_varlen
 *   other arguments as attn_prefill_varlen (total_k is total_q)
 * The result is that of the two calls, for any metadata.  The call enqueues
 * a store grid on at most half of the SMs and the prefill as its
 * programmatic dependent: the prefill starts on the other SMs at once, takes
 * each sequence's uncached key tiles first (read from k / v, which hold
 * them) and waits for the store grid before its first read of the cache, so
 * a sequence may read, as cached prefix, rows another sequence of the same
 * call stores.  A slot >= num_blocks * block_size stores nothing and records
 * KVP_ERR_DEVICE_DATA.  The limit of 64 calls in flight per device is shared
 * with attn_prefill_varlen.
 */
int attn_prefill_varlen_append(const kvp_bf16 *q, int64_t q_stride_tok, int64_t total_q,
                               const kvp_bf16 *k, const kvp_bf16 *v, int64_t kv_stride_tok,
                               const int32_t *slot_mapping, kvp_bf16 *k_cache, kvp_bf16 *v_cache,
                               int64_t num_blocks, int block_size, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *cu_seqlens_q,
                               const int32_t *cu_seqlens_k, int max_seqlen_q, int max_seqlen_k,
                               int num_seqs, const int64_t *positions, int num_heads,
                               int num_kv_heads, int head_dim, float softmax_scale, kvp_bf16 *out,
                               int64_t out_stride_tok, kvp_stream_t stream);

/*
 * attn_mixed_step - one engine step that mixes chunked prefill and decode:
 * kv_store of every new row, then attn_prefill_varlen (paged) over all
 * sequences, where the last num_decode_seqs sequences are decode rows (one
 * query row each, q_len 1; their query rows are the last num_decode_seqs rows).
 *
 * Source: the mixed step is the chunked-prefill extension that "nano-vLLM-1"
 * names (the pages' engine runs prefill-only or decode-only steps); its
 * decode rows follow "5. deocde 输入打包" (one token per sequence at position
 * len - 1) and its chunks "4. prefill 输入打包" (a suffix whose cached prefix
 * may end inside a block).
 *
 * Arguments as attn_prefill_varlen_append (block_tables required), plus:
 *   num_decode_seqs  0 .. num_seqs: the trailing decode rows.  Each must have
 *                    q_len 1 (otherwise KVP_ERR_DEVICE_DATA is recorded) and
 *                    its slot_mapping entry must be the slot of its position
 *                    k_len - 1 (as attn_decode_paged_append requires)
 *   decode_sms       SMs given to the decode rows while the chunks run on the
 *                    others (0, or a value not below the device's SM count:
 *                    5/8 of the SMs, 95 of 152); all SMs when no chunk has
 *                    query rows
 *   workspace        as attn_decode_paged, for the decode rows: at least
 *                    attn_decode_workspace_size(num_decode_seqs, num_heads,
 *                    head_dim, max_seqlen_k, block_size) bytes
 * Everything is enqueued on the caller's stream as one chain of programmatic
 * dependent launches: the store of the chunks' rows and the prefill of
 * attn_prefill_varlen_append on device SMs - decode_sms SMs, then the decode
 * (store fused) of attn_decode_paged_append on the other decode_sms SMs,
 * which starts as soon as the prefill grid is resident and completes after
 * it, then the decode's merge.  The chunks and the decode rows thus run side
 * by side, and work enqueued on the stream after the call sees both done.
 * The two halves read and write disjoint slots (a decode row writes its own
 * last block; a chunk writes its own uncached blocks).  The call holds no
 * stream or event of its own and may be captured in a CUDA graph.
 */
int attn_mixed_step(const kvp_bf16 *q, int64_t q_stride_tok, int64_t total_q, const kvp_bf16 *k,
                    const kvp_bf16 *v, int64_t kv_stride_tok, const int32_t *slot_mapping,
                    kvp_bf16 *k_cache, kvp_bf16 *v_cache, int64_t num_blocks, int block_size,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int max_seqlen_q,
                    int max_seqlen_k, int num_seqs, int num_decode_seqs, int decode_sms,
                    int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                    void *workspace, size_t workspace_bytes, kvp_bf16 *out,
                    int64_t out_stride_tok, kvp_stream_t stream);

/*
 * Bytes of device workspace attn_decode_paged needs for this shape on the
 * current device (0 on error; see kvp_last_error).
 */
size_t attn_decode_workspace_size(int num_seqs, int num_heads, int head_dim,
                                  int max_context_len, int block_size);

/*
 * attn_decode_paged - one query token per sequence over its paged history.
 *
 * Sequence b attends to its context_lens[b] tokens (the count includes the
 * token being decoded, which kv_store has just written), token p being read at
 * k_cache/v_cache[block_tables[b][p / block_size]][p % block_size]:
 *     out[b, h] = sum_{p < context_lens[b]} softmax_p(q[b, h] . k_p * scale) v_p
 * A sequence with context_lens[b] == 0 (the engine's padding rows) reads
 * nothing and gets an all-zero output row.
 * Source: "Nano vLLM 解读（5）" prepare_decode (context_lens, block_tables);
 * "nano-vLLM-1" "5. deocde 输入打包".
 *
 *   q               [num_seqs, num_heads, head_dim] bf16, row stride q_stride_tok
 *   block_tables    [num_seqs, max_blocks_per_seq] int32
 *   context_lens    [num_seqs] int32, each <= max_context_len and
 *                   <= max_blocks_per_seq * block_size
 *   workspace       device scratch of at least attn_decode_workspace_size()
 *                   bytes, 16-byte aligned; its contents need no
 *                   initialisation and are garbage afterwards.  Two calls that
 *                   run at the same time must not share a workspace.
 *   out             [num_seqs, num_heads, head_dim] bf16, row stride out_stride_tok
 * Supported: head_dim in {64, 128}; num_kv_heads in {1, 2, 4, 8};
 * num_heads / num_kv_heads in {1, 2, 4, 8}; any block_size >= 1.
 */
int attn_decode_paged(const kvp_bf16 *q, int64_t q_stride_tok, const kvp_bf16 *k_cache,
                      const kvp_bf16 *v_cache, int64_t num_blocks, int block_size,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int num_seqs, int max_context_len,
                      int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                      void *workspace, size_t workspace_bytes, kvp_bf16 *out,
                      int64_t out_stride_tok, kvp_stream_t stream);

/*
 * attn_decode_paged_append - kv_store of the step's new rows and
 * attn_decode_paged in one launch.
 *
 * A decode step stores one new token per sequence (its K and V rows, at the
 * slot of its last position) and then attends over the sequence's history
 * including that token ("nano-vLLM-1" ModelRunner "5. deocde 输入打包":
 * slot_mapping holds, per sequence, the slot of the token at position
 * len - 1; context_lens counts that token).  This call computes exactly what
 * kv_store(k, v, slot_mapping) followed by attn_decode_paged does, in one
 * kernel launch (plus the merge launch): the new rows are written to the
 * caches, and the sequence's last token is read from k / v instead of from
 * the cache slot being written.
 *
 *   k, v            [num_seqs, num_kv_heads, head_dim] bf16, row strides
 *                   k_stride_tok / v_stride_tok (multiples of 8 elements,
 *                   16-byte aligned): the new row of sequence b is row b
 *   slot_mapping    [num_seqs] int32: cache slot of sequence b's new row,
 *                   -1 = no store (padding rows, context_lens 0)
 *   k_cache/v_cache written at the slots of slot_mapping, read elsewhere
 *   other arguments as attn_decode_paged
 * Requirements beyond attn_decode_paged: for every b with context_lens[b]
 * > 0 and slot_mapping[b] >= 0, slot_mapping[b] is the slot of position
 * context_lens[b] - 1 through block_tables[b] (otherwise KVP_ERR_DEVICE_DATA
 * is recorded in the device status; the row is still stored and the
 * attention uses k / v for that position); no sequence of the batch reads
 * another sequence's new-row slot (true for the engine, whose last blocks
 * are private).  A slot >= num_blocks * block_size stores nothing and
 * records KVP_ERR_DEVICE_DATA.
 */
int attn_decode_paged_append(const kvp_bf16 *q, int64_t q_stride_tok, const kvp_bf16 *k,
                             const kvp_bf16 *v, int64_t k_stride_tok, int64_t v_stride_tok,
                             const int32_t *slot_mapping, kvp_bf16 *k_cache, kvp_bf16 *v_cache,
                             int64_t num_blocks, int block_size, const int32_t *block_tables,
                             int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                             int max_context_len, int num_heads, int num_kv_heads, int head_dim,
                             float softmax_scale, void *workspace, size_t workspace_bytes,
                             kvp_bf16 *out, int64_t out_stride_tok, kvp_stream_t stream);

/*
 * attn_decode_paged_noalloc - attn_decode_paged for callers that cannot
 * allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for integration.
 * Some callers have no way to obtain device memory on the call path: a
 * plugin inside a host runtime that owns every allocation and hands out no
 * allocator, a real-time serving loop that forbids cudaMalloc after start-up
 * (it can block and synchronize the device), or code that must not add an
 * allocation failure mode.  This entry point needs no workspace argument:
 * the split partials go into a scratch array compiled into the library
 * (a file-scope device variable of 8 MiB).  It calls no cudaMalloc, cudaFree
 * or other allocating routine.
 *
 * Arguments, results and errors are those of attn_decode_paged without
 * `workspace` / `workspace_bytes`, and checked in the same order (messages
 * name this entry point).  In addition:
 * - after those checks, a call whose scratch need (what
 *   attn_decode_workspace_size returns for it: CTAs x 2 x num_heads x
 *   (head_dim + 4) x 4 bytes plus 4 bytes per CTA, with one CTA per 64
 *   tokens of num_seqs x max_context_len, at most one per SM) exceeds 8 MiB
 *   is rejected with KVP_ERR_WORKSPACE and a message naming both sizes.
 *   Not every supported shape fits: on a 152-SM GB300, 64 query heads at
 *   head_dim 128 (8 kv heads x 8) need up to 9.8 MiB and are rejected once
 *   num_seqs x max_context_len exceeds 124 x 64 tokens; every other shape
 *   attn_decode_paged supports (at most 32 query heads at head_dim 128, or
 *   64 at head_dim 64) fits on GPUs of up to 240 SMs;
 * - every GPU that loads the library reserves the 8 MiB until the process
 *   exits;
 * - the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) and caches it; make that first call before any
 *   stream capture on that device;
 * - all calls share the one array and each call overwrites it (nothing in
 *   it needs to start at zero): calls that can overlap on the GPU (different
 *   streams, or different host threads without ordering) race and must not be
 *   issued; calls in order on one stream are safe.
 */
int attn_decode_paged_noalloc(const kvp_bf16 *q, int64_t q_stride_tok, const kvp_bf16 *k_cache,
                              const kvp_bf16 *v_cache, int64_t num_blocks, int block_size,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int num_seqs, int max_context_len,
                              int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                              kvp_bf16 *out, int64_t out_stride_tok, kvp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVPAGED_H */
