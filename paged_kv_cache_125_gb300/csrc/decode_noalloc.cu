// attn_decode_paged_noalloc: paged decode for callers that cannot allocate
// device memory.  Same contract as attn_decode_paged, except that the split
// partials go into a scratch array that lives in this file as a static device
// variable instead of a caller-provided workspace.
//
// The array is part of the library's device image: every GPU on which the
// library is loaded reserves kNoAllocScratchBytes for it until the process
// exits.  Host code may not hand the array's name to a kernel (on the host
// that name is only a stand-in for the device variable); the device address
// is fetched once per device with cudaGetSymbolAddress and cached.
#include <mutex>

#include "kvp_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;  // 8 MiB

__device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (set up on the
// first call for that device).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvp::set_last_error(KVP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return kvp::set_last_error(KVP_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr)
      return kvp::set_last_error(KVP_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s",
                                 cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KVP_OK;
}

}  // namespace

extern "C" int attn_decode_paged_noalloc(const kvp_bf16* q, int64_t q_stride_tok,
                                         const kvp_bf16* k_cache, const kvp_bf16* v_cache,
                                         int64_t num_blocks, int block_size,
                                         const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* context_lens, int num_seqs,
                                         int max_context_len, int num_heads, int num_kv_heads,
                                         int head_dim, float softmax_scale, kvp_bf16* out,
                                         int64_t out_stride_tok, kvp_stream_t stream) {
  // attn_decode_paged's own checks first, so a bad argument is reported as it
  // would be there; the scratch size after them.
  int rc = kvp::check_decode_args("attn_decode_paged_noalloc", q, q_stride_tok, k_cache, v_cache,
                                  num_blocks, block_size, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, max_context_len, num_heads, num_kv_heads,
                                  head_dim, out, out_stride_tok);
  if (rc != KVP_OK) return rc;
  if (num_seqs == 0) return KVP_OK;
  int sms = 0;
  rc = kvp::device_sm_count(&sms);
  if (rc != KVP_OK) return rc;
  const size_t need =
      kvp::plan_decode(num_seqs, num_heads, head_dim, max_context_len, sms).total_bytes;
  if (need > kNoAllocScratchBytes)
    return kvp::set_last_error(
        KVP_ERR_WORKSPACE,
        "attn_decode_paged_noalloc: this shape needs %zu bytes of scratch, more than the %zu "
        "bytes the built-in scratch holds; use attn_decode_paged with a caller workspace",
        need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != KVP_OK) return rc;
  // The split kernel writes every partial and boundary record the merge reads
  // within the same call, so nothing in the scratch has to start at zero.
  return attn_decode_paged(q, q_stride_tok, k_cache, v_cache, num_blocks, block_size, block_tables,
                           max_blocks_per_seq, context_lens, num_seqs, max_context_len, num_heads,
                           num_kv_heads, head_dim, softmax_scale, scratch, kNoAllocScratchBytes, out,
                           out_stride_tok, stream);
}
