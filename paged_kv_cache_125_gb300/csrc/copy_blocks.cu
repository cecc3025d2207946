// kv_copy_blocks: copy-on-write copies of whole cache blocks.
//
// Source: "【nano-vllm 学习】04 - 自顶向下的引擎调度层源码学习2", section
// "场景优化1：Parallel Memory Shared": sequences sampled from one prompt map
// their prompt blocks to the same physical blocks (reference counted); when
// one of them must append into a shared block that is not full, the engine
// gives it a fresh physical block holding a copy of the shared one (copy on
// write) and drops one reference from the old block.
//
// The cache is num_planes planes (one layer's K or V each, the pages'
// [k/v, layer, block, offset, kv_head, head_dim] tensor), every plane
// num_blocks blocks of block_elems bf16.  A work item is one 32 KiB chunk of
// one (pair, plane) block copy; each thread keeps eight 16-byte loads in
// flight.  HBM traffic is the algorithmic minimum: every source byte read
// once, every destination byte written once.
#include "kvp_device.cuh"

namespace kvp {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kVecPerThread = 8;
constexpr int64_t kChunkVecs = (int64_t)kCopyThreads * kVecPerThread;  // 32 KiB

__device__ __forceinline__ uint4 ld_once(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_once(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// 16-byte path: block_elems, plane_stride and the base are multiples of 8
// elements / 16 bytes.
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_vec_kernel(
    uint16_t* __restrict__ cache, int64_t num_planes, int64_t plane_stride, int64_t num_blocks,
    int64_t block_elems, const int32_t* __restrict__ mapping, int64_t num_pairs,
    int64_t chunks_per_block, int* status) {
  const int64_t block_vecs = block_elems >> 3;
  const int64_t items = num_pairs * num_planes * chunks_per_block;
  for (int64_t w = blockIdx.x; w < items; w += gridDim.x) {
    const int64_t chunk = w % chunks_per_block;
    const int64_t pp = w / chunks_per_block;  // pair * num_planes + plane
    const int64_t plane = pp % num_planes;
    const int64_t pair = pp / num_planes;
    const int32_t src = mapping[2 * pair], dst = mapping[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (threadIdx.x == 0 && plane == 0 && chunk == 0) record_error(status, KVP_ERR_DEVICE_DATA);
      continue;
    }
    const uint4* s4 = reinterpret_cast<const uint4*>(cache + plane * plane_stride +
                                                     (int64_t)src * block_elems);
    uint4* d4 = reinterpret_cast<uint4*>(cache + plane * plane_stride + (int64_t)dst * block_elems);
    const int64_t v0 = chunk * kChunkVecs;
    const int64_t v1 = min(v0 + kChunkVecs, block_vecs);
    if (v1 - v0 == kChunkVecs) {
      uint4 r[kVecPerThread];
#pragma unroll
      for (int i = 0; i < kVecPerThread; ++i) r[i] = ld_once(s4 + v0 + i * kCopyThreads + threadIdx.x);
#pragma unroll
      for (int i = 0; i < kVecPerThread; ++i) st_once(d4 + v0 + i * kCopyThreads + threadIdx.x, r[i]);
    } else {
      for (int64_t v = v0 + threadIdx.x; v < v1; v += kCopyThreads) st_once(d4 + v, ld_once(s4 + v));
    }
  }
}

// Any alignment: 2-byte elements, grid-stride over (pair, plane, element).
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_scalar_kernel(
    uint16_t* __restrict__ cache, int64_t num_planes, int64_t plane_stride, int64_t num_blocks,
    int64_t block_elems, const int32_t* __restrict__ mapping, int64_t num_pairs, int* status) {
  const int64_t units = num_pairs * num_planes;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t plane = u % num_planes, pair = u / num_planes;
    const int32_t src = mapping[2 * pair], dst = mapping[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (threadIdx.x == 0 && plane == 0) record_error(status, KVP_ERR_DEVICE_DATA);
      continue;
    }
    const uint16_t* s = cache + plane * plane_stride + (int64_t)src * block_elems;
    uint16_t* d = cache + plane * plane_stride + (int64_t)dst * block_elems;
    for (int64_t e = threadIdx.x; e < block_elems; e += kCopyThreads) d[e] = s[e];
  }
}

}  // namespace

cudaError_t launch_copy_blocks(uint16_t* cache, int64_t num_planes, int64_t plane_stride,
                               int64_t num_blocks, int64_t block_elems, const int32_t* mapping,
                               int64_t num_pairs, bool vec16, int num_sms, int* status,
                               cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t cap = (int64_t)num_sms * 8;
  if (vec16) {
    const int64_t chunks = ((block_elems >> 3) + kChunkVecs - 1) / kChunkVecs;
    const int64_t items = num_pairs * num_planes * chunks;
    const int64_t grid = items < cap ? items : cap;
    copy_blocks_vec_kernel<<<(unsigned)grid, kCopyThreads, 0, stream>>>(
        cache, num_planes, plane_stride, num_blocks, block_elems, mapping, num_pairs, chunks, status);
  } else {
    const int64_t units = num_pairs * num_planes;
    const int64_t grid = units < cap ? units : cap;
    copy_blocks_scalar_kernel<<<(unsigned)grid, kCopyThreads, 0, stream>>>(
        cache, num_planes, plane_stride, num_blocks, block_elems, mapping, num_pairs, status);
  }
  return cudaGetLastError();
}

}  // namespace kvp
