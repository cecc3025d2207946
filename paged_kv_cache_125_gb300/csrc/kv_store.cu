// kv_store: slot-mapped scatter of a step's new K/V rows into the paged cache.
//
// Source: "nano-vLLM-1", ModelRunner "4. prefill 输入打包" / "5. deocde 输入打包"
// (slot_mapping: linear slot block_id * block_size + offset of every new token;
// -1 marks CUDA-graph padding) and "Nano vLLM 解读（5）：解析 ModelRunner" (the
// [k/v, layer, block, offset, kv_head, head_dim] cache).
//
// One warp copies one (token, K-or-V) row of num_kv_heads * head_dim bf16
// values.  With the 16-byte path every lane moves whole 16-byte vectors: the
// row is read once (streaming, no L1 allocation) and written once.  HBM
// traffic is the algorithmic minimum: 2 * N * row bytes read + the same written.
#include "kvp_device.cuh"

namespace kvp {
namespace {

constexpr int kStoreThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <bool kVec16>
__global__ void __launch_bounds__(kStoreThreads) kv_store_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t k_stride,
    int64_t v_stride, const int32_t* __restrict__ slots, int64_t n, uint16_t* __restrict__ k_cache,
    uint16_t* __restrict__ v_cache, int64_t total_slots, int row_elems, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kStoreThreads / 32);
  for (int64_t r = (int64_t)blockIdx.x * (kStoreThreads / 32) + (threadIdx.x >> 5); r < 2 * n;
       r += warps) {
    const int64_t t = r >> 1;
    const bool is_v = r & 1;
    const int64_t s = slots[t];
    const uint16_t* src = is_v ? v + t * v_stride : k + t * k_stride;
    if constexpr (kVec16) {
      // The first four vectors per lane are loaded before the slot is known,
      // so the data loads do not wait for the slot load.
      const int nvec = row_elems >> 3;
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4 x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (lane + 32 * j < nvec) x[j] = ld_stream(s4 + lane + 32 * j);
      if (s < 0) continue;  // padding slot: nothing to write
      if (s >= total_slots) {
        if (lane == 0) record_error(status, KVP_ERR_DEVICE_DATA);
        continue;
      }
      uint4* d4 = reinterpret_cast<uint4*>((is_v ? v_cache : k_cache) + s * (int64_t)row_elems);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (lane + 32 * j < nvec) d4[lane + 32 * j] = x[j];
      for (int i = lane + 128; i < nvec; i += 128) {  // rows longer than 1024 elements
        uint4 a = ld_stream(s4 + i), b, c, d;
        if (i + 32 < nvec) b = ld_stream(s4 + i + 32);
        if (i + 64 < nvec) c = ld_stream(s4 + i + 64);
        if (i + 96 < nvec) d = ld_stream(s4 + i + 96);
        d4[i] = a;
        if (i + 32 < nvec) d4[i + 32] = b;
        if (i + 64 < nvec) d4[i + 64] = c;
        if (i + 96 < nvec) d4[i + 96] = d;
      }
    } else {
      if (s < 0) continue;  // padding slot: nothing to write
      if (s >= total_slots) {
        if (lane == 0) record_error(status, KVP_ERR_DEVICE_DATA);
        continue;
      }
      uint16_t* dst = (is_v ? v_cache : k_cache) + s * (int64_t)row_elems;
      for (int i = lane; i < row_elems; i += 32) dst[i] = src[i];
    }
  }
}

// The store of attn_prefill_varlen_append: few CTAs of 1024 threads (one per
// SM, on half of the SMs at most), so that the prefill launched as its
// programmatic dependent starts at once on the other SMs.  A warp copies two
// rows at a time with all their 16-byte loads in flight before the stores;
// the loads do not wait for the slots.
constexpr int kNarrowThreads = 1024;

__global__ void __launch_bounds__(kNarrowThreads, 1) kv_store_narrow_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t stride,
    const int32_t* __restrict__ slots, int64_t n, uint16_t* __restrict__ k_cache,
    uint16_t* __restrict__ v_cache, int64_t total_slots, int row_elems, int* status) {
  // Launched as a programmatic dependent of the previous grid on the stream
  // (which may have written k / v or still read the cache): wait for it to
  // complete before touching memory; only the launch latency is overlapped.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int nvec = row_elems >> 3;
  const int64_t warps = (int64_t)gridDim.x * (kNarrowThreads / 32);
  // Row pairs: pair p is token p (K row and V row).
  for (int64_t t = (int64_t)blockIdx.x * (kNarrowThreads / 32) + (threadIdx.x >> 5); t < n;
       t += warps) {
    const int64_t s = slots[t];
    const uint4* ks = reinterpret_cast<const uint4*>(k + t * stride);
    const uint4* vs = reinterpret_cast<const uint4*>(v + t * stride);
    for (int j0 = 0; j0 < nvec; j0 += 128) {
      uint4 xk[4], xv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = j0 + 32 * j + lane;
        if (i < nvec) {
          xk[j] = ld_stream(ks + i);
          xv[j] = ld_stream(vs + i);
        }
      }
      if (s < 0) break;  // padding slot: nothing to write
      if (s >= total_slots) {
        if (lane == 0) record_error(status, KVP_ERR_DEVICE_DATA);
        break;
      }
      uint4* kd = reinterpret_cast<uint4*>(k_cache + s * (int64_t)row_elems);
      uint4* vd = reinterpret_cast<uint4*>(v_cache + s * (int64_t)row_elems);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = j0 + 32 * j + lane;
        if (i < nvec) {
          kd[i] = xk[j];
          vd[i] = xv[j];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_store_narrow(const uint16_t* k, const uint16_t* v, int64_t stride,
                                   const int32_t* slots, int64_t n, uint16_t* k_cache,
                                   uint16_t* v_cache, int64_t total_slots, int row_elems,
                                   int num_sms, int* status, cudaStream_t stream, bool pdl) {
  if (n == 0) return cudaSuccess;
  int64_t grid = (n + kNarrowThreads / 32 - 1) / (kNarrowThreads / 32);
  const int64_t cap = num_sms / 2 > 0 ? num_sms / 2 : 1;
  if (grid > cap) grid = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kNarrowThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kv_store_narrow_kernel, k, v, stride, slots, n, k_cache, v_cache,
                            total_slots, row_elems, status);
}

cudaError_t launch_kv_store(const uint16_t* k, const uint16_t* v, int64_t k_stride,
                            int64_t v_stride, const int32_t* slots, int64_t n, uint16_t* k_cache,
                            uint16_t* v_cache, int64_t total_slots, int row_elems, bool vec16,
                            int num_sms, int* status, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t rows_per_cta = kStoreThreads / 32;
  int64_t grid = (2 * n + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = (int64_t)num_sms * 16;
  if (grid > cap) grid = cap;
  if (vec16)
    kv_store_kernel<true><<<(unsigned)grid, kStoreThreads, 0, stream>>>(
        k, v, k_stride, v_stride, slots, n, k_cache, v_cache, total_slots, row_elems, status);
  else
    kv_store_kernel<false><<<(unsigned)grid, kStoreThreads, 0, stream>>>(
        k, v, k_stride, v_stride, slots, n, k_cache, v_cache, total_slots, row_elems, status);
  return cudaGetLastError();
}

}  // namespace kvp
