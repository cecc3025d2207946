/*
 * Reference oracle for paged KV-cache attention: plain, slow, scalar C in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only the
 * test-suite, the smoke check and the CPU-baseline leg of the benchmark load it.
 * It shares no code, header or helper with the CUDA library; it reads the same
 * seeded inputs and nothing else.
 *
 * Sources (web pages on nano-vLLM):
 *   [P1] "nano-vLLM-1" (Senjl's Digital Garden): ModelRunner "3. KV cache 分配",
 *        "4. prefill 输入打包", "5. deocde 输入打包"; BlockManager
 *        "3. 核心方法一：分配 (allocate)" (slot = block_table[p // bs] * bs + p % bs).
 *   [P2] "Nano vLLM 解读（5）：解析 ModelRunner": cache layout
 *        [key/value, layer, block_id, token_offset_in_block, kv_head, head_dim];
 *        "prepare_prefill" / "prepare_decode" (meaning of cu_seqlens_q/k,
 *        block_tables, context_lens, slot_mapping).
 *   [P3] "【nano-vllm 学习】04 - 自顶向下的引擎调度层源码学习2", section
 *        "KV-Cache … 是什么？": Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V with
 *        a causal mask (masked scores -> -inf -> weight 0), and S_i = { j <= i };
 *        section "场景优化1：Parallel Memory Shared": copy on write of a shared
 *        block into a freshly allocated one.
 *
 * Readings where the pages leave a step open (each is also listed in the design
 * notes):
 *   - the visible set is inclusive (a token sees itself): S_i = { j <= i };
 *   - with a cached prefix of c tokens, query row i sits at absolute position c+i
 *     (the positions the pages build start at num_cached_tokens), so it sees keys
 *     0 .. c+i ("bottom-right" alignment);
 *   - GQA: query head h reads kv head h / (Hq / Hkv) (contiguous groups);
 *   - a decode row with context_len 0 reads nothing and its output is 0;
 *   - a slot of -1 (CUDA-graph padding in the pages) writes nothing.
 *
 * Arithmetic: every bf16 input is decoded exactly to double; scores, softmax and
 * the weighted sum are fp64; outputs are fp64 (the caller rounds if it wants).
 * The softmax subtracts the row maximum before exponentiating, which leaves
 * softmax(x) unchanged mathematically.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_SLOT (-1)
#define ORACLE_BAD_BLOCK (-2)
#define ORACLE_BAD_ARG (-3)
#define ORACLE_NOMEM (-4)

/* bf16 bit pattern -> double, exactly (bf16 is the top half of an IEEE float). */
static double bf16_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * Slot scatter [P1 "4. prefill 输入打包" / "5. deocde 输入打包"; P2 prepare_prefill]:
 * for each new token t with s = slot_mapping[t] >= 0, copy the bf16 bits of
 * k[t] (Hkv*d values) to k_cache[s / bs][s % bs] and likewise v.
 * k and v rows are [num_tokens, Hkv, d] with a row stride in elements.
 * Caches are one layer's [num_blocks, bs, Hkv, d], contiguous.
 */
int oracle_kv_store(const uint16_t *k, const uint16_t *v, int64_t k_stride_tok,
                    int64_t v_stride_tok, const int32_t *slot_mapping,
                    int64_t num_tokens, uint16_t *k_cache, uint16_t *v_cache,
                    int64_t num_blocks, int block_size, int num_kv_heads,
                    int head_dim) {
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue; /* padding: nothing written */
    int64_t blk = s / block_size, off = s % block_size;
    if (blk >= num_blocks) return ORACLE_BAD_SLOT;
    for (int h = 0; h < num_kv_heads; ++h) {
      for (int e = 0; e < head_dim; ++e) {
        int64_t dst = ((blk * block_size + off) * num_kv_heads + h) * head_dim + e;
        k_cache[dst] = k[t * k_stride_tok + (int64_t)h * head_dim + e];
        v_cache[dst] = v[t * v_stride_tok + (int64_t)h * head_dim + e];
      }
    }
  }
  return ORACLE_OK;
}

/*
 * Block-table gather [P1 BlockManager "3. 核心方法一：分配 (allocate)": logical token p
 * of a sequence lives in physical block block_table[p // bs] at offset p % bs;
 * P3 "代码分析": logical block i -> physical block block_table[i]].
 * Copies tokens 0..num_tokens-1 of one sequence into out [num_tokens, Hkv, d].
 */
int oracle_gather(const uint16_t *cache, int64_t num_blocks, int block_size,
                  int num_kv_heads, int head_dim, const int32_t *block_table_row,
                  int num_table_entries, int64_t num_tokens, uint16_t *out) {
  for (int64_t p = 0; p < num_tokens; ++p) {
    int64_t li = p / block_size;
    if (li >= num_table_entries) return ORACLE_BAD_BLOCK;
    int64_t blk = block_table_row[li];
    if (blk < 0 || blk >= num_blocks) return ORACLE_BAD_BLOCK;
    int64_t off = p % block_size;
    for (int h = 0; h < num_kv_heads; ++h)
      for (int e = 0; e < head_dim; ++e)
        out[(p * num_kv_heads + h) * head_dim + e] =
            cache[((blk * block_size + off) * num_kv_heads + h) * head_dim + e];
  }
  return ORACLE_OK;
}

/*
 * Copy on write [P3 "场景优化1：Parallel Memory Shared": a sequence that must
 * append into a block shared with others gets a new physical block holding a
 * copy of the shared one].  For every pair i (src = mapping[2i],
 * dst = mapping[2i+1]) and every plane p (one layer's K or V cache), copy the
 * block_elems bf16 bits of block src to block dst.  Pairs are applied in order.
 */
int oracle_copy_blocks(uint16_t *cache, int64_t num_planes, int64_t plane_stride,
                       int64_t num_blocks, int64_t block_elems, const int32_t *mapping,
                       int64_t num_pairs) {
  for (int64_t i = 0; i < num_pairs; ++i) {
    int64_t src = mapping[2 * i], dst = mapping[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return ORACLE_BAD_BLOCK;
    for (int64_t p = 0; p < num_planes; ++p)
      for (int64_t e = 0; e < block_elems; ++e)
        cache[p * plane_stride + dst * block_elems + e] =
            cache[p * plane_stride + src * block_elems + e];
  }
  return ORACLE_OK;
}

/* Address of key/value element (token p of sequence b, kv head g, dim e).
 * Paged: through the block table [P1 allocate; P2 block_tables].
 * Packed: row cu_k[b] + p of the step's own k/v [P2 prepare_prefill: without a
 * prefix hit the kernel uses the K/V computed in this step]. */
typedef struct {
  const uint16_t *k, *v; /* packed rows, or caches */
  int64_t kv_stride;     /* packed row stride (elements) */
  const int32_t *bt;     /* NULL -> packed */
  int max_blocks;
  int64_t num_blocks;
  int block_size;
  int num_kv_heads;
  int head_dim;
} kv_source;

static int kv_row_index(const kv_source *src, int b, int64_t kv_start, int64_t p,
                        int64_t *row_out) {
  if (src->bt == NULL) {
    *row_out = (kv_start + p) * src->kv_stride;
    return ORACLE_OK;
  }
  int64_t li = p / src->block_size;
  if (li >= src->max_blocks) return ORACLE_BAD_BLOCK;
  int64_t blk = src->bt[(int64_t)b * src->max_blocks + li];
  if (blk < 0 || blk >= src->num_blocks) return ORACLE_BAD_BLOCK;
  *row_out = (blk * src->block_size + p % src->block_size) *
             (int64_t)src->num_kv_heads * src->head_dim;
  return ORACLE_OK;
}

/*
 * One attention row: o = sum_{j < n_visible} softmax_j(q . k_j * scale) v_j
 * [P3 "KV-Cache … 是什么？": softmax(QK^T / sqrt(d_k)) V, masked entries get
 * weight 0].  q is one query head's row (d values); keys 0..n_visible-1 of
 * sequence b from kv head g.  Result written to out[0..d-1] in fp64.
 */
static int attend_row(const uint16_t *q, const kv_source *src, int b,
                      int64_t kv_start, int g, int64_t n_visible, double scale,
                      double *scores, double *out) {
  int d = src->head_dim;
  for (int e = 0; e < d; ++e) out[e] = 0.0;
  if (n_visible <= 0) return ORACLE_OK; /* empty context: output 0 */
  double qd[512];
  for (int e = 0; e < d; ++e) qd[e] = bf16_to_double(q[e]);
  double mx = -INFINITY;
  for (int64_t j = 0; j < n_visible; ++j) {
    int64_t row;
    int rc = kv_row_index(src, b, kv_start, j, &row);
    if (rc) return rc;
    const uint16_t *kr = src->k + row + (int64_t)g * d;
    double s = 0.0;
    for (int e = 0; e < d; ++e) s += qd[e] * bf16_to_double(kr[e]);
    s *= scale;
    scores[j] = s;
    if (s > mx) mx = s;
  }
  double denom = 0.0;
  for (int64_t j = 0; j < n_visible; ++j) {
    scores[j] = exp(scores[j] - mx);
    denom += scores[j];
  }
  for (int64_t j = 0; j < n_visible; ++j) {
    int64_t row;
    kv_row_index(src, b, kv_start, j, &row);
    const uint16_t *vr = src->v + row + (int64_t)g * d;
    double w = scores[j] / denom;
    for (int e = 0; e < d; ++e) out[e] += w * bf16_to_double(vr[e]);
  }
  return ORACLE_OK;
}

/*
 * Varlen causal prefill [P2 prepare_prefill; P1 "4. prefill 输入打包"]:
 * sequences packed by cu_seqlens_q / cu_seqlens_k (prefix sums of
 * q_len = len - num_cached_tokens and k_len = len).  Query row i of sequence b
 * is at absolute position c_b + i, c_b = k_len - q_len, and sees keys
 * 0 .. c_b + i.  Keys come from the caches through block_tables when
 * block_tables != NULL (prefix-cache hit), otherwise from the packed k / v rows
 * of this step (then k_len must equal q_len).
 *
 * q: [sum q, Hq, d] (row stride q_stride_tok); out: [sum q, Hq, d] fp64 dense.
 * rows / num_rows: optional list of packed query-token indices to compute
 * (NULL = all); rows not listed are left untouched.
 */
int oracle_prefill(const uint16_t *q, int64_t q_stride_tok, const uint16_t *k,
                   const uint16_t *v, int64_t kv_stride_tok,
                   const uint16_t *k_cache, const uint16_t *v_cache,
                   int64_t num_blocks, int block_size,
                   const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                   int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                   double scale, const int64_t *rows, int64_t num_rows,
                   double *out) {
  if (num_heads % num_kv_heads != 0 || head_dim > 512) return ORACLE_BAD_ARG;
  int group = num_heads / num_kv_heads;
  kv_source src;
  src.bt = block_tables;
  src.k = block_tables ? k_cache : k;
  src.v = block_tables ? v_cache : v;
  src.kv_stride = kv_stride_tok;
  src.max_blocks = max_blocks_per_seq;
  src.num_blocks = num_blocks;
  src.block_size = block_size;
  src.num_kv_heads = num_kv_heads;
  src.head_dim = head_dim;
  int64_t total_q = cu_seqlens_q[num_seqs];
  int64_t n_work = rows ? num_rows : total_q;
  int64_t max_k = 0;
  for (int b = 0; b < num_seqs; ++b) {
    int64_t kl = cu_seqlens_k[b + 1] - cu_seqlens_k[b];
    int64_t ql = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    if (ql > kl || ql < 0) return ORACLE_BAD_ARG;
    if (!block_tables && ql != kl) return ORACLE_BAD_ARG;
    if (kl > max_k) max_k = kl;
  }
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)(max_k > 0 ? max_k : 1));
    if (!scores) {
#pragma omp atomic write
      err = ORACLE_NOMEM;
    }
#pragma omp for schedule(dynamic, 1) collapse(2)
    for (int64_t w = 0; w < n_work; ++w) {
      for (int h = 0; h < num_heads; ++h) {
        if (!scores) continue;
        int64_t t = rows ? rows[w] : w;
        if (t < 0 || t >= total_q) {
#pragma omp atomic write
          err = ORACLE_BAD_ARG;
          continue;
        }
        int b = 0; /* sequence owning packed row t */
        while (b + 1 < num_seqs && cu_seqlens_q[b + 1] <= t) ++b;
        int64_t i = t - cu_seqlens_q[b];
        int64_t kl = cu_seqlens_k[b + 1] - cu_seqlens_k[b];
        int64_t ql = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        int64_t cached = kl - ql;
        int64_t n_visible = cached + i + 1; /* keys 0 .. cached+i */
        int rc = attend_row(q + t * q_stride_tok + (int64_t)h * head_dim, &src, b,
                            cu_seqlens_k[b], h / group, n_visible, scale, scores,
                            out + (t * num_heads + h) * (int64_t)head_dim);
        if (rc) {
#pragma omp atomic write
          err = rc;
        }
      }
    }
    free(scores);
  }
  return err;
}

/*
 * Paged decode [P2 prepare_decode; P1 "5. deocde 输入打包"]: one query token per
 * sequence; sequence b attends to its context_lens[b] cached tokens (the count
 * includes the token being decoded, whose K/V the step has just stored),
 * reached through block_tables[b].
 *
 * q: [B, Hq, d] (row stride q_stride_tok); out: [B, Hq, d] fp64 dense.
 * seqs / num_sel: optional subset of sequences to compute (NULL = all).
 */
int oracle_decode(const uint16_t *q, int64_t q_stride_tok, const uint16_t *k_cache,
                  const uint16_t *v_cache, int64_t num_blocks, int block_size,
                  const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *context_lens, int num_seqs, int num_heads,
                  int num_kv_heads, int head_dim, double scale,
                  const int32_t *seqs, int num_sel, double *out) {
  if (num_heads % num_kv_heads != 0 || head_dim > 512) return ORACLE_BAD_ARG;
  int group = num_heads / num_kv_heads;
  kv_source src;
  src.bt = block_tables;
  src.k = k_cache;
  src.v = v_cache;
  src.kv_stride = 0;
  src.max_blocks = max_blocks_per_seq;
  src.num_blocks = num_blocks;
  src.block_size = block_size;
  src.num_kv_heads = num_kv_heads;
  src.head_dim = head_dim;
  int n_work = seqs ? num_sel : num_seqs;
  int64_t max_ctx = 1;
  for (int b = 0; b < num_seqs; ++b)
    if (context_lens[b] > max_ctx) max_ctx = context_lens[b];
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)max_ctx);
#pragma omp for schedule(dynamic, 1) collapse(2)
    for (int w = 0; w < n_work; ++w) {
      for (int h = 0; h < num_heads; ++h) {
        int b = seqs ? seqs[w] : w;
        if (!scores || b < 0 || b >= num_seqs) {
#pragma omp atomic write
          err = scores ? ORACLE_BAD_ARG : ORACLE_NOMEM;
          continue;
        }
        int rc = attend_row(q + (int64_t)b * q_stride_tok + (int64_t)h * head_dim, &src,
                            b, 0, h / group, context_lens[b], scale, scores,
                            out + ((int64_t)b * num_heads + h) * head_dim);
        if (rc) {
#pragma omp atomic write
          err = rc;
        }
      }
    }
    free(scores);
  }
  return err;
}

/* Number of OpenMP threads the oracle runs with (for the CPU-baseline report). */
int oracle_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      n = omp_get_num_threads();
#endif
    }
  }
  return n;
}
