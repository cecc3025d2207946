/*
 * kvpaged_sched.h - host-side block manager and scheduler of a nano-vLLM-style
 * engine, in C++ behind a C ABI (part of libkvpaged.so; no GPU work).
 *
 * It turns requests into engine steps and builds, for each step, the metadata
 * the attention calls of kvpaged.h take.  Policy and data structures follow
 * "nano-vLLM-1" (Senjl's Digital Garden):
 *   - BlockManager ("1. Block", "2. BlockManager 初始化与链式哈希",
 *     "3. 核心方法一：分配 (allocate)", "4. 核心方法二：追加 (may_append)",
 *     "5. 核心方法三：回收块（deallocate）"): FIFO free list; a full block's
 *     chained hash (previous block's hash, then the token ids) registers it for
 *     prefix caching, and a hit is confirmed by comparing token ids; freed
 *     blocks keep their hash; a hit on a block that is in use takes one more
 *     reference.
 *   - Scheduler ("1. 队列与状态机", "2. prefill 的 schedule", "3. decode 的
 *     schedule", "4. 后处理：postprocess()"): prefill first, FCFS from the head
 *     of `waiting`, stopping at the first sequence that does not fit the token
 *     budget (its full length) or the free blocks; the budget is charged
 *     length - cached tokens; otherwise a decode step over `running`, preempting
 *     from the tail of `running` when a sequence cannot append (the sequence
 *     itself when it is alone); preempted sequences go to the head of `waiting`;
 *     a sequence finishes after max_tokens generated tokens (no EOS).
 *   - ModelRunner "4. prefill 输入打包" / "5. deocde 输入打包": the metadata.
 * The 64-bit chained hash is FNV-1a over (previous hash, token ids); any 64-bit
 * hash gives the same schedule because a hit also compares the token ids.
 *
 * All buffers are host memory owned by the caller.  Functions return 0 or a
 * negative KVP_ERR_* code (kvpaged.h); the message is in kvp_last_error().
 */
#ifndef KVPAGED_SCHED_H_
#define KVPAGED_SCHED_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvp_scheduler kvp_scheduler; /* opaque */

/* New scheduler over a pool of num_blocks blocks of block_size tokens.
 * Returns NULL (and sets the last error) on bad arguments. */
kvp_scheduler *kvp_sched_create(int num_blocks, int block_size, int max_num_seqs,
                                int max_num_batched_tokens);
void kvp_sched_destroy(kvp_scheduler *s);

/* Queues a request at the tail of `waiting`: prompt token ids (copied) and the
 * number of tokens to generate (>= 1).  seq_id must be unique. */
int kvp_sched_add(kvp_scheduler *s, int64_t seq_id, const int64_t *token_ids, int num_tokens,
                  int max_tokens);

/* 1 when no request is waiting or running. */
int kvp_sched_is_finished(const kvp_scheduler *s);

/* Schedules the next step.  Writes the ids of the scheduled sequences, in
 * step order, to seq_ids (capacity max_num_seqs) and *is_prefill; returns how
 * many were scheduled (>= 1), or a negative code (KVP_ERR_INVALID_ARG when
 * nothing is queued, KVP_ERR_UNSUPPORTED when the pool cannot hold a single
 * sequence). */
int kvp_sched_schedule(kvp_scheduler *s, int64_t *seq_ids, int *is_prefill);

/* Sizes of the scheduled step's metadata: rows stored and queried this step
 * (prefill: sum of uncached lengths; decode: one per sequence) and the widest
 * block table. */
int kvp_sched_step_sizes(const kvp_scheduler *s, int64_t *num_new_tokens, int *max_blocks);

/* Metadata of the scheduled step (the pages' prepare_prefill / prepare_decode),
 * for n scheduled sequences and T = num_new_tokens:
 *   prefill: cu_seqlens_q/k [n+1], positions [T], slot_mapping [T],
 *            *max_seqlen_q / *max_seqlen_k, and *has_prefix = 1 when some
 *            sequence has cached tokens (then block_tables [n, stride] is
 *            filled, -1 padded; the kernels read keys from the cache);
 *   decode:  positions [n], context_lens [n], slot_mapping [n],
 *            block_tables [n, stride] (-1 padded); cu_seqlens and the maxima
 *            are not touched.
 * Pointers the step kind does not use may be NULL; stride >= max_blocks. */
int kvp_sched_prepare(const kvp_scheduler *s, int32_t *cu_seqlens_q, int32_t *cu_seqlens_k,
                      int64_t *positions, int32_t *slot_mapping, int32_t *context_lens,
                      int32_t *block_tables, int block_tables_stride, int *max_seqlen_q,
                      int *max_seqlen_k, int *has_prefix);

/* Appends one generated token to every scheduled sequence (token_ids[i] for
 * the i-th one, n = the count kvp_sched_schedule returned); finished
 * sequences release their blocks. */
int kvp_sched_postprocess(kvp_scheduler *s, const int64_t *token_ids, int n);

/* Inspection: preemptions so far, free blocks, and one sequence's state
 * (block table copied to table[0 .. cap), its length in *num_table_entries;
 * status 0 waiting / 1 running / 2 finished). */
int64_t kvp_sched_num_preemptions(const kvp_scheduler *s);
int kvp_sched_num_free_blocks(const kvp_scheduler *s);
int kvp_sched_seq_state(const kvp_scheduler *s, int64_t seq_id, int *num_tokens,
                        int *num_cached_tokens, int *status, int32_t *table, int cap,
                        int *num_table_entries);

#ifdef __cplusplus
}
#endif

#endif /* KVPAGED_SCHED_H_ */
