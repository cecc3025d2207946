// C ABI of libkvpaged: argument validation, error reporting, dispatch.
// The declarations and the contract of every entry point are in kvpaged.h.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "kvp_internal.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(KVP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// One status word per device; kernels record their first in-kernel error
// here (out-of-range metadata, expired wait).
__device__ int g_kvp_status;

constexpr int kMaxDevices = 64;
std::atomic<int*> g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];
std::mutex g_device_mu;

// Per-device set-up: device address of the status word and the SM count.
// Done once per device under a lock (first calls may come from several host
// threads); later calls read the published pointer without locking.
int device_info(int* dev_out, int** status, int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(KVP_ERR_UNSUPPORTED, "device %d", dev);
  int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_device_mu);
    p = g_status_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_kvp_status);
      if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(status)");
      int sms = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
      g_num_sms[dev] = sms;
      p = static_cast<int*>(addr);
      g_status_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *dev_out = dev;
  *status = p;
  *num_sms = g_num_sms[dev];
  return KVP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_block_size_pow2(int bs) {
  if (bs < 16 || bs > 4096 || bs % 16) return false;
  int m = bs / 16;
  return (m & (m - 1)) == 0;
}

}  // namespace

namespace kvp {

int set_last_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

// The argument checks of attn_decode_paged, in its order, with `fn` naming
// the entry point in the message.  num_seqs == 0 passes before the pointer
// checks (the call is then a no-op).
int check_decode_args(const char* fn, const kvp_bf16* q, int64_t q_stride_tok,
                      const kvp_bf16* k_cache, const kvp_bf16* v_cache, int64_t num_blocks,
                      int block_size, const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int num_seqs, int max_context_len,
                      int num_heads, int num_kv_heads, int head_dim, const kvp_bf16* out,
                      int64_t out_stride_tok) {
  if (num_seqs < 0 || max_context_len < 0 || num_blocks <= 0 || block_size <= 0 ||
      max_blocks_per_seq < 0)
    return fail(KVP_ERR_INVALID_ARG, "%s: bad sizes", fn);
  if (!decode_supported(num_heads, num_kv_heads, head_dim))
    return fail(KVP_ERR_UNSUPPORTED, "%s: unsupported heads %d/%d or head_dim %d", fn, num_heads,
                num_kv_heads, head_dim);
  if (q_stride_tok < (int64_t)num_heads * head_dim || out_stride_tok < (int64_t)num_heads * head_dim)
    return fail(KVP_ERR_INVALID_ARG, "%s: row stride too small", fn);
  if ((int64_t)max_blocks_per_seq * block_size > (int64_t)1 << 30)
    return fail(KVP_ERR_UNSUPPORTED, "%s: context capacity too large", fn);
  if (num_seqs == 0) return KVP_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return fail(KVP_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      q_stride_tok % 8 || out_stride_tok % 8)
    return fail(KVP_ERR_INVALID_ARG,
                "%s: q, caches and out need 16-byte alignment and row strides that are multiples "
                "of 8 elements",
                fn);
  return KVP_OK;
}

int device_sm_count(int* num_sms) {
  int dev, *status;
  return device_info(&dev, &status, num_sms);
}

}  // namespace kvp

extern "C" {

const char* kvp_last_error(void) { return g_last_error; }

int kvp_version(void) { return 100; }  // 0.1.0

int kvp_device_status(void) {
  int dev, *status, sms;
  int rc = device_info(&dev, &status, &sms);
  if (rc) return rc;
  int value = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&value, g_kvp_status, sizeof(int));
  if (e != cudaSuccess) return fail_cuda(e, "read device status");
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_kvp_status, &zero, sizeof(int));
  if (e != cudaSuccess) return fail_cuda(e, "clear device status");
  return value;
}

int kvp_selftest_wait(int arrive, kvp_stream_t stream) {
  int dev, *status, sms;
  int rc = device_info(&dev, &status, &sms);
  if (rc) return rc;
  cudaError_t e = kvp::launch_selftest_wait(arrive, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "kvp_selftest_wait launch");
  return KVP_OK;
}

int kv_store(const kvp_bf16* k, const kvp_bf16* v, int64_t k_stride_tok, int64_t v_stride_tok,
             const int32_t* slot_mapping, int64_t num_tokens, kvp_bf16* k_cache,
             kvp_bf16* v_cache, int64_t num_blocks, int block_size, int num_kv_heads,
             int head_dim, kvp_stream_t stream) {
  if (num_tokens < 0) return fail(KVP_ERR_INVALID_ARG, "kv_store: num_tokens < 0");
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return fail(KVP_ERR_INVALID_ARG, "kv_store: non-positive shape");
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (row > (1 << 20)) return fail(KVP_ERR_UNSUPPORTED, "kv_store: row too long");
  if (k_stride_tok < row || v_stride_tok < row)
    return fail(KVP_ERR_INVALID_ARG, "kv_store: row stride smaller than num_kv_heads*head_dim");
  if (num_tokens == 0) return KVP_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(KVP_ERR_INVALID_ARG, "kv_store: null pointer");
  int dev, *status, sms;
  int rc = device_info(&dev, &status, &sms);
  if (rc) return rc;
  const bool vec16 = aligned16(k) && aligned16(v) && aligned16(k_cache) && aligned16(v_cache) &&
                     row % 8 == 0 && k_stride_tok % 8 == 0 && v_stride_tok % 8 == 0;
  cudaError_t e = kvp::launch_kv_store(k, v, k_stride_tok, v_stride_tok, slot_mapping, num_tokens,
                                       k_cache, v_cache, num_blocks * (int64_t)block_size,
                                       (int)row, vec16, sms, status, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, "kv_store launch");
  return KVP_OK;
}

int kv_copy_blocks(kvp_bf16* cache, int64_t num_planes, int64_t plane_stride, int64_t num_blocks,
                   int64_t block_elems, const int32_t* block_mapping, int64_t num_pairs,
                   kvp_stream_t stream) {
  if (num_pairs < 0) return fail(KVP_ERR_INVALID_ARG, "kv_copy_blocks: num_pairs < 0");
  if (num_planes <= 0 || num_blocks <= 0 || block_elems <= 0)
    return fail(KVP_ERR_INVALID_ARG, "kv_copy_blocks: non-positive shape");
  if (plane_stride < num_blocks * block_elems)
    return fail(KVP_ERR_INVALID_ARG, "kv_copy_blocks: plane_stride < num_blocks * block_elems");
  if (num_pairs == 0) return KVP_OK;
  if (!cache || !block_mapping) return fail(KVP_ERR_INVALID_ARG, "kv_copy_blocks: null pointer");
  int dev, *status, sms;
  int rc = device_info(&dev, &status, &sms);
  if (rc) return rc;
  const bool vec16 = aligned16(cache) && plane_stride % 8 == 0 && block_elems % 8 == 0;
  cudaError_t e = kvp::launch_copy_blocks(cache, num_planes, plane_stride, num_blocks, block_elems,
                                          block_mapping, num_pairs, vec16, sms, status,
                                          (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, "kv_copy_blocks launch");
  return KVP_OK;
}

size_t attn_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                  int block_size) {
  (void)block_size;
  if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0) {
    fail(KVP_ERR_INVALID_ARG, "attn_decode_workspace_size: bad shape");
    return 0;
  }
  int dev, *status, sms;
  if (device_info(&dev, &status, &sms)) return 0;
  return kvp::plan_decode(num_seqs, num_heads, head_dim, max_context_len, sms).total_bytes;
}

int attn_decode_paged(const kvp_bf16* q, int64_t q_stride_tok, const kvp_bf16* k_cache,
                      const kvp_bf16* v_cache, int64_t num_blocks, int block_size,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int num_seqs, int max_context_len,
                      int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                      void* workspace, size_t workspace_bytes, kvp_bf16* out,
                      int64_t out_stride_tok, kvp_stream_t stream) {
  int rc = kvp::check_decode_args("attn_decode_paged", q, q_stride_tok, k_cache, v_cache,
                                  num_blocks, block_size, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, max_context_len, num_heads, num_kv_heads,
                                  head_dim, out, out_stride_tok);
  if (rc) return rc;
  if (num_seqs == 0) return KVP_OK;
  int dev, *status, sms;
  rc = device_info(&dev, &status, &sms);
  if (rc) return rc;
  const kvp::DecodePlan plan = kvp::plan_decode(num_seqs, num_heads, head_dim, max_context_len, sms);
  if (!workspace || workspace_bytes < plan.total_bytes || !aligned16(workspace))
    return fail(KVP_ERR_WORKSPACE, "attn_decode_paged: workspace needs %zu bytes (got %zu)",
                plan.total_bytes, workspace_bytes);
  cudaError_t e = kvp::launch_decode(q, q_stride_tok, k_cache, v_cache, num_blocks, block_size,
                                     block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                     num_heads, num_kv_heads, head_dim, softmax_scale, plan,
                                     workspace, out, out_stride_tok, status, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, "attn_decode_paged launch");
  return KVP_OK;
}

int attn_decode_paged_append(const kvp_bf16* q, int64_t q_stride_tok, const kvp_bf16* k,
                             const kvp_bf16* v, int64_t k_stride_tok, int64_t v_stride_tok,
                             const int32_t* slot_mapping, kvp_bf16* k_cache, kvp_bf16* v_cache,
                             int64_t num_blocks, int block_size, const int32_t* block_tables,
                             int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                             int max_context_len, int num_heads, int num_kv_heads, int head_dim,
                             float softmax_scale, void* workspace, size_t workspace_bytes,
                             kvp_bf16* out, int64_t out_stride_tok, kvp_stream_t stream) {
  if (num_seqs < 0 || max_context_len < 0 || num_blocks <= 0 || block_size <= 0 ||
      max_blocks_per_seq < 0)
    return fail(KVP_ERR_INVALID_ARG, "attn_decode_paged_append: bad sizes");
  if (!kvp::decode_supported(num_heads, num_kv_heads, head_dim))
    return fail(KVP_ERR_UNSUPPORTED,
                "attn_decode_paged_append: unsupported heads %d/%d or head_dim %d", num_heads,
                num_kv_heads, head_dim);
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (q_stride_tok < (int64_t)num_heads * head_dim || out_stride_tok < (int64_t)num_heads * head_dim ||
      k_stride_tok < row || v_stride_tok < row)
    return fail(KVP_ERR_INVALID_ARG, "attn_decode_paged_append: row stride too small");
  if ((int64_t)max_blocks_per_seq * block_size > (int64_t)1 << 30)
    return fail(KVP_ERR_UNSUPPORTED, "attn_decode_paged_append: context capacity too large");
  if (num_blocks * (int64_t)block_size >= ((int64_t)1 << 31))
    return fail(KVP_ERR_UNSUPPORTED, "attn_decode_paged_append: pool has 2^31 or more slots");
  if (num_seqs == 0) return KVP_OK;
  if (!q || !k || !v || !slot_mapping || !k_cache || !v_cache || !block_tables || !context_lens ||
      !out)
    return fail(KVP_ERR_INVALID_ARG, "attn_decode_paged_append: null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || q_stride_tok % 8 || out_stride_tok % 8 ||
      k_stride_tok % 8 || v_stride_tok % 8)
    return fail(KVP_ERR_INVALID_ARG,
                "attn_decode_paged_append: q, k, v, caches and out need 16-byte alignment and "
                "row strides that are multiples of 8 elements");
  int dev, *status, sms;
  int rc = device_info(&dev, &status, &sms);
  if (rc) return rc;
  const kvp::DecodePlan plan = kvp::plan_decode(num_seqs, num_heads, head_dim, max_context_len, sms);
  if (!workspace || workspace_bytes < plan.total_bytes || !aligned16(workspace))
    return fail(KVP_ERR_WORKSPACE, "attn_decode_paged_append: workspace needs %zu bytes (got %zu)",
                plan.total_bytes, workspace_bytes);
  const kvp::DecodeAppend app{k, v, k_stride_tok, v_stride_tok, slot_mapping, k_cache, v_cache};
  cudaError_t e = kvp::launch_decode(q, q_stride_tok, k_cache, v_cache, num_blocks, block_size,
                                     block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                     num_heads, num_kv_heads, head_dim, softmax_scale, plan,
                                     workspace, out, out_stride_tok, status, (cudaStream_t)stream,
                                     &app);
  if (e != cudaSuccess) return fail_cuda(e, "attn_decode_paged_append launch");
  return KVP_OK;
}

int attn_prefill_varlen(const kvp_bf16* q, int64_t q_stride_tok, int64_t total_q,
                        const kvp_bf16* k, const kvp_bf16* v, int64_t kv_stride_tok,
                        int64_t total_k, const kvp_bf16* k_cache,
                        const kvp_bf16* v_cache, int64_t num_blocks, int block_size,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                        int max_seqlen_q, int max_seqlen_k, int num_seqs,
                        const int64_t* positions, int num_heads, int num_kv_heads, int head_dim,
                        float softmax_scale, kvp_bf16* out, int64_t out_stride_tok,
                        kvp_stream_t stream) {
  (void)positions;
  if (num_seqs < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return fail(KVP_ERR_INVALID_ARG, "attn_prefill_varlen: bad sizes");
  if (!kvp::prefill_supported(num_heads, num_kv_heads, head_dim, block_size))
    return fail(KVP_ERR_UNSUPPORTED,
                "attn_prefill_varlen: unsupported heads %d/%d, head_dim %d or block_size %d",
                num_heads, num_kv_heads, head_dim, block_size);
  if (q_stride_tok < (int64_t)num_heads * head_dim || out_stride_tok < (int64_t)num_heads * head_dim)
    return fail(KVP_ERR_INVALID_ARG, "attn_prefill_varlen: row stride too small");
  if (num_seqs == 0 || max_seqlen_q == 0 || total_q == 0) return KVP_OK;
  if (total_q < 0 || total_q >= ((int64_t)1 << 31) || total_k < 0 || total_k >= ((int64_t)1 << 31))
    return fail(KVP_ERR_INVALID_ARG, "attn_prefill_varlen: total_q / total_k out of range");
  if (!q || !cu_seqlens_q || !cu_seqlens_k || !out)
    return fail(KVP_ERR_INVALID_ARG, "attn_prefill_varlen: null pointer");
  if (block_tables) {
    if (!k_cache || !v_cache || num_blocks <= 0 || max_blocks_per_seq <= 0)
      return fail(KVP_ERR_INVALID_ARG, "attn_prefill_varlen: paged mode needs the caches");
    if (num_blocks * (int64_t)block_size >= ((int64_t)1 << 31))
      return fail(KVP_ERR_UNSUPPORTED, "attn_prefill_varlen: pool has 2^31 or more slots");
    if (!aligned16(k_cache) || !aligned16(v_cache))
      return fail(KVP_ERR_INVALID_ARG, "attn_prefill_varlen: caches need 16-byte alignment");
  } else {
    if (!k || !v || total_k <= 0)
      return fail(KVP_ERR_INVALID_ARG, "attn_prefill_varlen: packed mode needs k, v, total_k");
    if (kv_stride_tok < (int64_t)num_kv_heads * head_dim || kv_stride_tok % 8 || !aligned16(k) ||
        !aligned16(v))
      return fail(KVP_ERR_INVALID_ARG, "attn_prefill_varlen: packed k/v alignment or stride");
  }
  if (!aligned16(q) || !aligned16(out) || q_stride_tok % 8 || out_stride_tok % 8)
    return fail(KVP_ERR_INVALID_ARG,
                "attn_prefill_varlen: q/out need 16-byte alignment and strides multiple of 8");
  int dev, *status, sms;
  int rc = device_info(&dev, &status, &sms);
  if (rc) return rc;
  const char* why = nullptr;
  rc = kvp::launch_prefill(q, q_stride_tok, total_q, k, v, kv_stride_tok, total_k, k_cache,
                           v_cache, num_blocks,
                           block_size, block_tables, max_blocks_per_seq, cu_seqlens_q,
                           cu_seqlens_k, max_seqlen_q, max_seqlen_k, num_seqs, num_heads,
                           num_kv_heads, head_dim, softmax_scale, out, out_stride_tok, sms, status,
                           (cudaStream_t)stream, &why);
  if (rc) return fail(rc, "attn_prefill_varlen: %s", why ? why : "launch failed");
  return KVP_OK;
}

int attn_prefill_varlen_append(const kvp_bf16* q, int64_t q_stride_tok, int64_t total_q,
                               const kvp_bf16* k, const kvp_bf16* v, int64_t kv_stride_tok,
                               const int32_t* slot_mapping, kvp_bf16* k_cache, kvp_bf16* v_cache,
                               int64_t num_blocks, int block_size, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* cu_seqlens_q,
                               const int32_t* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k,
                               int num_seqs, const int64_t* positions, int num_heads,
                               int num_kv_heads, int head_dim, float softmax_scale, kvp_bf16* out,
                               int64_t out_stride_tok, kvp_stream_t stream) {
  (void)positions;
  const char* fn = "attn_prefill_varlen_append";
  if (num_seqs < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return fail(KVP_ERR_INVALID_ARG, "%s: bad sizes", fn);
  if (!kvp::prefill_supported(num_heads, num_kv_heads, head_dim, block_size))
    return fail(KVP_ERR_UNSUPPORTED, "%s: unsupported heads %d/%d, head_dim %d or block_size %d",
                fn, num_heads, num_kv_heads, head_dim, block_size);
  if (q_stride_tok < (int64_t)num_heads * head_dim || out_stride_tok < (int64_t)num_heads * head_dim ||
      kv_stride_tok < (int64_t)num_kv_heads * head_dim)
    return fail(KVP_ERR_INVALID_ARG, "%s: row stride too small", fn);
  if (num_blocks <= 0) return fail(KVP_ERR_INVALID_ARG, "%s: num_blocks <= 0", fn);
  if (num_blocks * (int64_t)block_size >= ((int64_t)1 << 31))
    return fail(KVP_ERR_UNSUPPORTED, "%s: pool has 2^31 or more slots", fn);
  if (num_seqs == 0 || max_seqlen_q == 0 || total_q == 0) return KVP_OK;
  if (total_q < 0 || total_q >= ((int64_t)1 << 31))
    return fail(KVP_ERR_INVALID_ARG, "%s: total_q out of range", fn);
  if (!q || !k || !v || !slot_mapping || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k ||
      !out)
    return fail(KVP_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (block_tables && max_blocks_per_seq <= 0)
    return fail(KVP_ERR_INVALID_ARG, "%s: paged mode needs max_blocks_per_seq > 0", fn);
  if (!aligned16(q) || !aligned16(out) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) ||
      !aligned16(v_cache) || q_stride_tok % 8 || out_stride_tok % 8 || kv_stride_tok % 8)
    return fail(KVP_ERR_INVALID_ARG,
                "%s: q, k, v, caches and out need 16-byte alignment and row strides that are "
                "multiples of 8 elements",
                fn);
  int dev, *status, sms;
  int rc = device_info(&dev, &status, &sms);
  if (rc) return rc;
  cudaError_t e = kvp::launch_kv_store_narrow(k, v, kv_stride_tok, slot_mapping, total_q, k_cache,
                                              v_cache, num_blocks * (int64_t)block_size,
                                              num_kv_heads * head_dim, sms, status,
                                              (cudaStream_t)stream, true);
  if (e != cudaSuccess) return fail_cuda(e, "attn_prefill_varlen_append store launch");
  const kvp::PrefillAppend app{k, v, kv_stride_tok};
  const char* why = nullptr;
  rc = kvp::launch_prefill(q, q_stride_tok, total_q, k, v, kv_stride_tok, total_q, k_cache,
                           v_cache, num_blocks, block_size, block_tables, max_blocks_per_seq,
                           cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, num_seqs,
                           num_heads, num_kv_heads, head_dim, softmax_scale, out, out_stride_tok,
                           sms, status, (cudaStream_t)stream, &why, &app);
  if (rc) return fail(rc, "%s: %s", fn, why ? why : "launch failed");
  return KVP_OK;
}

int attn_mixed_step(const kvp_bf16* q, int64_t q_stride_tok, int64_t total_q, const kvp_bf16* k,
                    const kvp_bf16* v, int64_t kv_stride_tok, const int32_t* slot_mapping,
                    kvp_bf16* k_cache, kvp_bf16* v_cache, int64_t num_blocks, int block_size,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int max_seqlen_q,
                    int max_seqlen_k, int num_seqs, int num_decode_seqs, int decode_sms,
                    int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                    void* workspace, size_t workspace_bytes, kvp_bf16* out,
                    int64_t out_stride_tok, kvp_stream_t stream) {
  const char* fn = "attn_mixed_step";
  if (num_seqs < 0 || num_decode_seqs < 0 || num_decode_seqs > num_seqs || decode_sms < 0 ||
      max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_q >= ((int64_t)1 << 31) ||
      num_decode_seqs > total_q)
    return fail(KVP_ERR_INVALID_ARG, "%s: bad sizes", fn);
  if (!kvp::prefill_supported(num_heads, num_kv_heads, head_dim, block_size) ||
      !kvp::decode_supported(num_heads, num_kv_heads, head_dim))
    return fail(KVP_ERR_UNSUPPORTED, "%s: unsupported heads %d/%d, head_dim %d or block_size %d",
                fn, num_heads, num_kv_heads, head_dim, block_size);
  if (q_stride_tok < (int64_t)num_heads * head_dim || out_stride_tok < (int64_t)num_heads * head_dim ||
      kv_stride_tok < (int64_t)num_kv_heads * head_dim)
    return fail(KVP_ERR_INVALID_ARG, "%s: row stride too small", fn);
  if (num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(KVP_ERR_INVALID_ARG, "%s: num_blocks and max_blocks_per_seq must be positive", fn);
  if (num_blocks * (int64_t)block_size >= ((int64_t)1 << 31))
    return fail(KVP_ERR_UNSUPPORTED, "%s: pool has 2^31 or more slots", fn);
  if ((int64_t)max_blocks_per_seq * block_size > (int64_t)1 << 30)
    return fail(KVP_ERR_UNSUPPORTED, "%s: context capacity too large", fn);
  if (num_seqs == 0 || total_q == 0) return KVP_OK;
  if (!q || !k || !v || !slot_mapping || !k_cache || !v_cache || !block_tables || !cu_seqlens_q ||
      !cu_seqlens_k || !out)
    return fail(KVP_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(q) || !aligned16(out) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) ||
      !aligned16(v_cache) || q_stride_tok % 8 || out_stride_tok % 8 || kv_stride_tok % 8)
    return fail(KVP_ERR_INVALID_ARG,
                "%s: q, k, v, caches and out need 16-byte alignment and row strides that are "
                "multiples of 8 elements",
                fn);
  int dev, *status, sms;
  int rc = device_info(&dev, &status, &sms);
  if (rc) return rc;
  const int nd = num_decode_seqs, np = num_seqs - nd;
  const int64_t tq_p = total_q - nd;  // query rows of the prefill sequences
  // Default share of the decode rows: 5/8 of the SMs (95 of 152), near the
  // best split measured on a step of 4 chunks (3772 rows) and 128 decode rows
  // (past ~97 of 152 the chunks become the longer half).
  const bool chunks = np > 0 && tq_p > 0;  // prefill rows to run beside the decode rows
  const int dec_sms =
      nd == 0 ? 0 : (!chunks ? sms : (decode_sms > 0 && decode_sms < sms ? decode_sms : sms * 5 / 8));
  // The decode rows: the last nd sequences, one query row each, the store of
  // their new rows fused into the decode.
  kvp::DecodePlan plan{};
  if (nd > 0) {
    plan = kvp::plan_decode(nd, num_heads, head_dim, max_seqlen_k, dec_sms);
    if (!workspace || workspace_bytes < plan.total_bytes || !aligned16(workspace))
      return fail(KVP_ERR_WORKSPACE, "%s: workspace needs %zu bytes (got %zu)", fn,
                  plan.total_bytes, workspace_bytes);
  }
  // One stream, chained by programmatic dependent launches: the store of the
  // prefill rows, the prefill on sms - dec_sms SMs (a dependent of the store;
  // it lets its own dependents start at once), then the decode rows' split
  // kernel on the remaining SMs (a dependent of the prefill that completes
  // after it) and its merge.  The two halves touch disjoint rows, slots and
  // outputs, and a kernel that follows the call on the stream sees them both
  // complete.
  const cudaStream_t st = (cudaStream_t)stream;
  if (chunks) {
    cudaError_t e = kvp::launch_kv_store_narrow(k, v, kv_stride_tok, slot_mapping, tq_p, k_cache,
                                                v_cache, num_blocks * (int64_t)block_size,
                                                num_kv_heads * head_dim, sms - dec_sms, status, st,
                                                true);
    if (e != cudaSuccess) return fail_cuda(e, "attn_mixed_step: store launch");
    const kvp::PrefillAppend app{k, v, kv_stride_tok};
    const char* why = nullptr;
    rc = kvp::launch_prefill(q, q_stride_tok, tq_p, k, v, kv_stride_tok, tq_p, k_cache, v_cache,
                             num_blocks, block_size, block_tables, max_blocks_per_seq, cu_seqlens_q,
                             cu_seqlens_k, max_seqlen_q, max_seqlen_k, np, num_heads, num_kv_heads,
                             head_dim, softmax_scale, out, out_stride_tok, sms - dec_sms, status, st,
                             &why, &app);
    if (rc) return fail(rc, "%s: %s", fn, why ? why : "prefill launch failed");
  }
  if (nd > 0) {
    const int64_t r0 = tq_p;
    const kvp::DecodeAppend app{k + r0 * kv_stride_tok, v + r0 * kv_stride_tok, kv_stride_tok,
                                kv_stride_tok, slot_mapping + r0, k_cache, v_cache};
    const kvp::DecodeRowsOf rows{cu_seqlens_q, cu_seqlens_k, np};
    cudaError_t e = kvp::launch_decode(q + r0 * q_stride_tok, q_stride_tok, k_cache, v_cache,
                                       num_blocks, block_size,
                                       block_tables + (int64_t)np * max_blocks_per_seq,
                                       max_blocks_per_seq, nullptr, nd, num_heads, num_kv_heads,
                                       head_dim, softmax_scale, plan, workspace,
                                       out + r0 * out_stride_tok, out_stride_tok, status, st, &app,
                                       &rows, chunks);
    if (e != cudaSuccess) return fail_cuda(e, "attn_mixed_step: decode launch");
  }
  return KVP_OK;
}

}  // extern "C"
