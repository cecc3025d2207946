// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units of libkvpaged.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvpaged.h"

namespace kvp {

// api.cu: records the calling thread's message for kvp_last_error(); returns code.
int set_last_error(int code, const char* fmt, ...);
// api.cu: attn_decode_paged's argument checks (message names `fn`); the
// current device's SM count (set-up on first use per device).
int check_decode_args(const char* fn, const kvp_bf16* q, int64_t q_stride_tok,
                      const kvp_bf16* k_cache, const kvp_bf16* v_cache, int64_t num_blocks,
                      int block_size, const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int num_seqs, int max_context_len,
                      int num_heads, int num_kv_heads, int head_dim, const kvp_bf16* out,
                      int64_t out_stride_tok);
int device_sm_count(int* num_sms);

// selftest.cu: one thread waits on a barrier (arrive: after arriving on it
// itself; else nothing arrives and the 2 ms wait expires).
cudaError_t launch_selftest_wait(int arrive, int* status, cudaStream_t stream);

// kv_store.cu
cudaError_t launch_kv_store(const uint16_t* k, const uint16_t* v, int64_t k_stride,
                            int64_t v_stride, const int32_t* slots, int64_t n, uint16_t* k_cache,
                            uint16_t* v_cache, int64_t total_slots, int row_elems, bool vec16,
                            int num_sms, int* status, cudaStream_t stream);
// The store of attn_prefill_varlen_append (16-byte aligned rows; k and v
// share a row stride): at most num_sms / 2 CTAs of 1024 threads, which let
// the prefill launched as their programmatic dependent start on the others.
// pdl: launched itself as a programmatic dependent of the stream's previous
// kernel (it waits for that kernel before touching memory).
cudaError_t launch_kv_store_narrow(const uint16_t* k, const uint16_t* v, int64_t stride,
                                   const int32_t* slots, int64_t n, uint16_t* k_cache,
                                   uint16_t* v_cache, int64_t total_slots, int row_elems,
                                   int num_sms, int* status, cudaStream_t stream, bool pdl);

// copy_blocks.cu
cudaError_t launch_copy_blocks(uint16_t* cache, int64_t num_planes, int64_t plane_stride,
                               int64_t num_blocks, int64_t block_elems, const int32_t* mapping,
                               int64_t num_pairs, bool vec16, int num_sms, int* status,
                               cudaStream_t stream);

// decode.cu
struct DecodePlan {
  int ctas;            // persistent CTAs of the split kernel (one per SM at most)
  size_t part_bytes;   // partial results: ctas * 2 * Hq * (D + 4) floats
  size_t split_bytes;  // one int per CTA
  size_t total_bytes;  // workspace needed
};
DecodePlan plan_decode(int num_seqs, int num_heads, int head_dim, int max_context_len,
                       int num_sms);
bool decode_supported(int num_heads, int num_kv_heads, int head_dim);
// New rows of a fused store (attn_decode_paged_append).
struct DecodeAppend {
  const uint16_t* k;
  const uint16_t* v;
  int64_t k_stride, v_stride;
  const int32_t* slot_mapping;
  uint16_t* k_cache;
  uint16_t* v_cache;
};
// The decode rows of a mixed step: sequence b of the call is sequence
// offset + b of a varlen batch; its context length is cu_k[offset + b + 1] -
// cu_k[offset + b] (context_lens unused) and its q_len (cu_q) must be 1.
// pdl: the split kernel is launched as a programmatic dependent of the
// stream's previous kernel (it starts beside it and completes after it).
struct DecodeRowsOf {
  const int32_t* cu_q;
  const int32_t* cu_k;
  int offset;
};
cudaError_t launch_decode(const uint16_t* q, int64_t q_stride, const uint16_t* k_cache,
                          const uint16_t* v_cache, int64_t num_blocks, int block_size,
                          const int32_t* block_tables, int max_blocks, const int32_t* ctx,
                          int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                          float softmax_scale, const DecodePlan& plan, void* workspace,
                          uint16_t* out, int64_t out_stride, int* status, cudaStream_t stream,
                          const DecodeAppend* app = nullptr, const DecodeRowsOf* rows_of = nullptr,
                          bool pdl = false);

// prefill.cu: cuTensorMapEncodeTiled (a PFN_cuTensorMapEncodeTiled_v12000), or
// null if the driver does not provide it.
void* tensor_map_encoder();
bool prefill_supported(int num_heads, int num_kv_heads, int head_dim, int block_size);
// New rows of attn_prefill_varlen_append, stored by a kv_store launch just
// before the prefill: row t of k / v (row stride `stride`) is the key /
// value of query row t.  The prefill is launched as a programmatic dependent
// of the store and reads uncached keys from these rows.
struct PrefillAppend {
  const uint16_t* k;
  const uint16_t* v;
  int64_t stride;
};
int launch_prefill(const uint16_t* q, int64_t q_stride, int64_t total_q, const uint16_t* k,
                   const uint16_t* v, int64_t kv_stride, int64_t total_k,
                   const uint16_t* k_cache, const uint16_t* v_cache,
                   int64_t num_blocks, int block_size, const int32_t* block_tables,
                   int max_blocks, const int32_t* cu_q, const int32_t* cu_k, int max_seqlen_q,
                   int max_seqlen_k, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                   float softmax_scale, uint16_t* out, int64_t out_stride, int num_sms,
                   int* status, cudaStream_t stream, const char** why,
                   const PrefillAppend* app = nullptr);

}  // namespace kvp
