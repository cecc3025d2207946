// attn_decode_paged: one query token per sequence over its paged KV history.
//
// Source: "Nano vLLM 解读（5）：解析 ModelRunner", prepare_decode (context_lens
// counts the token being decoded; block_tables map logical to physical
// blocks); "nano-vLLM-1" "5. deocde 输入打包"; attention itself is
// softmax(q K^T * scale) V ("【nano-vllm 学习】04 …", "KV-Cache … 是什么？").
//
// Design (memory bound: every K/V byte of the batch is read exactly once).
//
// * Flat split over the whole batch.  The tokens of all sequences, laid end
//   to end (T = sum context_lens), are cut into one contiguous chunk per CTA
//   (ceil(T / CTAs)), and the grid is one persistent CTA per SM.  Every SM
//   streams the same number of bytes whatever the length mix; a sequence cut
//   by a chunk boundary leaves partial results (running max m, sum l, and the
//   un-normalised accumulator) that a small merge kernel combines by
//   log-sum-exp.  A sequence inside one chunk is finished in place.
// * Each CTA reads all kv heads of a token at once: a token's K row for all
//   heads is num_kv_heads * head_dim contiguous bf16 (2 KiB for 8 x 128), so
//   a stage of up to 64 / num_kv_heads tokens of one physical block is one
//   contiguous 1-D bulk copy for K and one for V (16 KiB each at 8 x 128).  A
//   producer warp streams stages into a 6-deep shared-memory ring
//   (cp.async.bulk + mbarrier transaction counts); it reads the block table as
//   it goes, so the gather costs nothing beyond the copy addresses.
// * Eight consumer warps; warp w serves kv head w % Hkv (and, when
//   Hkv < 8, tokens (w / Hkv) * 8 .. + 7 of each stage, or the token subset
//   w / Hkv).  Two kinds of consumers:
//   - one or two query heads per kv head (CUDA cores): a lane owns 1/8 of
//     head_dim (two 16-byte chunks at head_dim 128) of one token; 4 tokens
//     per pass.  q . k is an fp32 dot product over the lane's slice reduced
//     over 8 lanes by shuffles, with q pre-scaled by softmax_scale * log2(e)
//     so the softmax uses exp2.  The running max is warp-uniform and updated
//     once per stage.  These stream at the HBM rate.
//   - four or eight query heads per kv head (tensor cores, mma.sync): the
//     stage is copied by one 4-D tensor copy per half into a swizzled
//     [head][panel][token][64] layout; S = q K^T and O^T = V^T P^T are
//     m16n8k16 / m16n8k8 MMAs over the warp's 8 tokens (see the section
//     "tensor-core consumers" below).  The CUDA-core form needs 2 FMAs per
//     K/V byte at G = 4 and is issue-bound there.
// * Optional store of the step's new rows (attn_decode_paged_append): the
//   kv_store of one new token per sequence is folded into the same launch.
//   After the producer has issued every stage, its warp writes the rows of
//   sequences i, i + P, ... (CTA i) into the cache slots slot_mapping[b];
//   the stage that ends at a sequence's last context token
//   takes that token's K and V row straight from the new rows (one more bulk
//   copy; on the tensor-core path the consumer writes that row into the
//   swizzled stage) instead of from the cache, so no CTA reads a slot written
//   in the same launch.
#include <cudaTypedefs.h>

#include <cfloat>

#include "kvp_device.cuh"

namespace kvp {
namespace {

constexpr int kBaseWarps = 8;  // consumer warps
constexpr int kStages = 6;  // ring depth (one less where a tensor-core CTA would not fit)
constexpr size_t kSmemPerCta = 227 * 1024;

constexpr int kTokensAllHeads = 64;  // tokens * kv heads per stage

// Row of one split partial in the workspace: accumulator[D], m, l, and two pad
// floats so that every row starts on a 16-byte boundary (float4 stores).
template <int D>
__host__ __device__ constexpr int part_stride() {
  return D + 4;
}

// F_TAIL (tensor-core path with the fused store): the stage ends at the
// sequence's last context token, whose K / V row the consumer takes from the
// new rows instead of the cache.
enum : int { F_NEW = 1, F_LAST = 2, F_ENTERED = 4, F_EXITS = 8, F_DONE = 16, F_TAIL = 32 };

struct StageMeta {
  int b;
  int n;
  int flags;
  int pad;
};

struct DecodeArgs {
  const uint16_t* q;
  int64_t q_stride;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  int64_t num_blocks;
  int block_size;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* ctx;  // context_lens, or null: from cu_k (the decode rows of a mixed step)
  const int32_t* cu_q;  // mixed step: cu_seqlens_q / cu_seqlens_k of the whole batch, whose
  const int32_t* cu_k;  //   sequences cu_off .. cu_off + num_seqs - 1 are this call's rows
  int cu_off;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  float scale_log2;
  float* part;     // [ctas][2][Hq][D + 4]: accumulator[D], m, l, pad
  int* split_seq;  // [ctas]: sequence continuing into the next CTA, or -1
  uint16_t* out;
  int64_t out_stride;
  int* status;
  int tma_per_head;  // tensor-core path: one box per (kv head, panel) instead of one per stage
};

// Fused store of the new rows (null k_new: plain decode).  A kernel parameter
// of its own: the consumer warps never touch it, and keeping it out of
// DecodeArgs keeps their register allocation as it is without it.
struct AppendArgs {
  const uint16_t* k_new;  // [num_seqs, Hkv, D], row stride k_new_stride
  const uint16_t* v_new;
  int64_t k_new_stride, v_new_stride;
  const int32_t* slot_mapping;  // [num_seqs]; -1 = no store
  uint16_t* k_cache_w;          // the caches, written by the store
  uint16_t* v_cache_w;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int clamp_len(int c, int cap) { return c < 0 ? 0 : (c > cap ? cap : c); }

// Context length of sequence b: context_lens[b], or, for the decode rows of a
// mixed step, the key count of batch sequence cu_off + b (its one query row
// is the token at position context - 1).
__device__ __forceinline__ int seq_ctx(const DecodeArgs& a, int b) {
  if (a.ctx) return a.ctx[b];
  return a.cu_k[a.cu_off + b + 1] - a.cu_k[a.cu_off + b];
}

template <int D>
__host__ __device__ constexpr size_t stage_half_bytes() {
  return (size_t)kTokensAllHeads * D * sizeof(uint16_t);
}

// CUDA-core path (one or two query heads per kv head): the ring, the stage
// records, the ring and hand-off barriers and each warp's partial staging.
// With 9 warps per CTA one SM sub-partition runs 3 of them, so a thread can
// hold at most 168 registers: a lane's query slice (G * D / 8 floats) and
// accumulators fit.
template <int D, int G>
__host__ __device__ constexpr size_t decode_smem_bytes(int ns) {
  return 2 * ns * stage_half_bytes<D>() + ns * sizeof(StageMeta) +
         (2 * ns + 2 * kBaseWarps) * sizeof(uint64_t) + (size_t)kBaseWarps * G * (D + 2) * sizeof(float);
}
static_assert(decode_smem_bytes<128, 2>(kStages) <= kSmemPerCta, "decode CTA smem");

// ---------------------------------------------------------------- producer

// Stage loop of the producer (one thread): copies the CTA's token range
// [start, end), first sequence b0 starting at token cum0 of the batch, into
// the ring, then posts the end marker.
template <int D, int RS, bool kTma>
__device__ void stream_stages(const DecodeArgs& a, const AppendArgs& app, const CUtensorMap* tmK,
                              const CUtensorMap* tmV, uint8_t* ringK, uint8_t* ringV,
                              StageMeta* meta, uint64_t* full, uint64_t* empty,
                              long long start, long long end, int b0, long long cum0, int cap) {
  const int Hkv = a.num_kv_heads;
  a.split_seq[blockIdx.x] = -1;
  const int T = kTokensAllHeads / Hkv;
  const int64_t row_elems = (int64_t)Hkv * D;
  int s = 0;
  uint32_t ph = 0;
  uint32_t issued = 0, issued_ph = 0;  // per stage: ever issued / parity of the last issue
  bool ok = true;

  long long pos = start, cum = cum0;
  int b = b0;
  while (ok && pos < end && b < a.num_seqs) {
    const int L = clamp_len(seq_ctx(a, b), cap);
    if (L == 0) {
      ++b;
      continue;
    }
    const long long seq_end = cum + L;
    const long long seg_end = end < seq_end ? end : seq_end;
    int t = (int)(pos - cum);
    const int t1 = (int)(seg_end - cum);
    const int seg_flags = (pos > cum ? F_ENTERED : 0) | (seg_end < seq_end ? F_EXITS : 0);
    bool first = true;
    int cur_bi = -1, phys = 0;
    while (t < t1) {
      const int bi = t / a.block_size, off = t - bi * a.block_size;
      int n = a.block_size - off;
      if (n > T) n = T;
      if (n > t1 - t) n = t1 - t;
      if (bi != cur_bi) {
        cur_bi = bi;
        phys = a.block_tables[(int64_t)b * a.max_blocks + bi];
        if (phys < 0 || phys >= a.num_blocks) {
          record_error(a.status, KVP_ERR_DEVICE_DATA);
          phys = 0;  // never dereference an out-of-range block
        }
      }
      if (!mbar_wait(&empty[s], ph ^ 1u, a.status)) {
        ok = false;
        break;
      }
      // With the fused store, the sequence's last token comes from the new rows.
      const bool tail = app.k_new != nullptr && t + n == L;
      meta[s].b = b;
      meta[s].n = n;
      meta[s].flags = (first ? F_NEW : 0) | (t + n == t1 ? F_LAST : 0) | seg_flags |
                      (kTma && tail ? F_TAIL : 0);
      uint8_t* dk = ringK + (size_t)s * stage_half_bytes<D>();
      uint8_t* dv = ringV + (size_t)s * stage_half_bytes<D>();
      if constexpr (kTma) {
        // One box of T rows x all heads x head_dim from the stage's first
        // token on (rows past n are masked by the consumers); the tail row is
        // patched in shared memory by the consumer that reads it.
        mbar_arrive_expect_tx(&full[s], 2 * (uint32_t)stage_half_bytes<D>());
        const int row = (int)((int64_t)phys * a.block_size + off);
        if (!a.tma_per_head) {
          tma_load_4d(dk, tmK, 0, row, 0, 0, &full[s]);
          tma_load_4d(dv, tmV, 0, row, 0, 0, &full[s]);
        } else {  // the same layout, one box {64, 1, T} per (kv head, panel)
          const uint32_t region = (uint32_t)T * 128;
          for (int h = 0; h < Hkv; ++h)
            for (int p = 0; p < D / 64; ++p) {
              const uint32_t off_b = (uint32_t)(h * (D / 64) + p) * region;
              tma_load_3d(dk + off_b, tmK, p * 64, h, row, &full[s]);
              tma_load_3d(dv + off_b, tmV, p * 64, h, row, &full[s]);
            }
        }
      } else {
        const uint32_t bytes = (uint32_t)(n * row_elems * sizeof(uint16_t));
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        const int64_t row0 = ((int64_t)phys * a.block_size + off) * row_elems;
        const uint32_t row_bytes = (uint32_t)(row_elems * sizeof(uint16_t));
        const uint32_t cbytes = tail ? bytes - row_bytes : bytes;
        if (cbytes) {
          bulk_g2s(dk, a.k_cache + row0, cbytes, &full[s]);
          bulk_g2s(dv, a.v_cache + row0, cbytes, &full[s]);
        }
        if (tail) {
          bulk_g2s(dk + cbytes, app.k_new + (int64_t)b * app.k_new_stride, row_bytes, &full[s]);
          bulk_g2s(dv + cbytes, app.v_new + (int64_t)b * app.v_new_stride, row_bytes, &full[s]);
        }
      }
      issued |= 1u << s;
      issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
      first = false;
      t += n;
      if (++s == RS) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (seg_flags & F_EXITS) a.split_seq[blockIdx.x] = b;
    pos = seg_end;
    cum = seq_end;
    ++b;
  }
  if (ok && mbar_wait(&empty[s], ph ^ 1u, a.status)) {
    meta[s].flags = F_DONE;
    mbar_arrive(&full[s]);
    return;
  }
  // A wait expired: let every copy this CTA issued land before the CTA exits.
  for (int i = 0; i < RS; ++i)
    if (issued >> i & 1u) mbar_wait(&full[i], issued_ph >> i & 1u, a.status);
}

// Store of the step's new rows (attn_decode_paged_append), one warp: this CTA
// writes the rows of sequences blockIdx.x + k * gridDim.x.  The slot must be
// that of the sequence's last context token (the engine's decode step);
// otherwise the step would not equal store-then-attend, and the mismatch is
// reported.
template <int D>
__device__ void fused_store(const DecodeArgs& a, const AppendArgs& app, int lane, int cap) {
  const int64_t row_elems = (int64_t)a.num_kv_heads * D;
  const int64_t pool_slots = a.num_blocks * a.block_size;
  for (int b = blockIdx.x; b < a.num_seqs; b += gridDim.x) {
    const int slot = app.slot_mapping[b];
    if (slot < 0) continue;
    if (slot >= pool_slots) {
      if (lane == 0) record_error(a.status, KVP_ERR_DEVICE_DATA);
      continue;
    }
    const int L = clamp_len(seq_ctx(a, b), cap);
    if (L > 0 && lane == 0) {
      const int lb = (L - 1) / a.block_size;
      const int phys = a.block_tables[(int64_t)b * a.max_blocks + lb];
      if ((int64_t)phys * a.block_size + (L - 1 - lb * a.block_size) != slot)
        record_error(a.status, KVP_ERR_DEVICE_DATA);
    }
    const uint4* ks = reinterpret_cast<const uint4*>(app.k_new + (int64_t)b * app.k_new_stride);
    const uint4* vs = reinterpret_cast<const uint4*>(app.v_new + (int64_t)b * app.v_new_stride);
    uint4* kd = reinterpret_cast<uint4*>(app.k_cache_w + (int64_t)slot * row_elems);
    uint4* vd = reinterpret_cast<uint4*>(app.v_cache_w + (int64_t)slot * row_elems);
    for (int i = lane; i < row_elems / 8; i += 32) {
      kd[i] = ks[i];
      vd[i] = vs[i];
    }
  }
}

template <int D, int RS, bool kTma>
__device__ void decode_producer(const DecodeArgs& a, const AppendArgs& app, const CUtensorMap* tmK,
                                const CUtensorMap* tmV, uint8_t* ringK, uint8_t* ringV,
                                StageMeta* meta, uint64_t* full, uint64_t* empty) {
  const int lane = threadIdx.x & 31;
  const int cap = a.max_blocks * a.block_size;
  const int P = gridDim.x;

  // Total tokens of the batch (every CTA computes the same value).
  long long tot = 0;
  for (int i = lane; i < a.num_seqs; i += 32) {
    const int c = seq_ctx(a, i);
    if (!a.ctx && a.cu_q[a.cu_off + i + 1] - a.cu_q[a.cu_off + i] != 1)
      record_error(a.status, KVP_ERR_DEVICE_DATA);  // a decode row queries one token
    if (c < 0 || c > cap) record_error(a.status, KVP_ERR_DEVICE_DATA);
    tot += clamp_len(c, cap);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const long long chunk = (tot + P - 1) / P;
  const long long start = (long long)blockIdx.x * chunk;
  const long long end = start + chunk < tot ? start + chunk : tot;

  // Rows of sequences with no context are zero (they read nothing).
  for (int b = blockIdx.x; b < a.num_seqs; b += P) {
    if (clamp_len(seq_ctx(a, b), cap) != 0) continue;
    uint4* o = reinterpret_cast<uint4*>(a.out + (int64_t)b * a.out_stride);
    for (int i = lane; i < a.num_heads * D / 8; i += 32) o[i] = make_uint4(0, 0, 0, 0);
  }

  // First sequence overlapping [start, end): warp scan over context_lens.
  int b0 = 0;
  long long cum0 = 0;
  if (start < end) {
    long long run = 0;
    for (int base = 0; base < a.num_seqs; base += 32) {
      const int i = base + lane;
      const long long c = i < a.num_seqs ? clamp_len(seq_ctx(a, i), cap) : 0;
      long long incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, i < a.num_seqs && run + incl > start);
      if (hit) {
        const int L = __ffs(hit) - 1;
        b0 = base + L;
        cum0 = run + __shfl_sync(0xffffffffu, incl - c, L);
        break;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (lane == 0) {
    if constexpr (kTma) {
      prefetch_tensormap(tmK);
      prefetch_tensormap(tmV);
    }
    stream_stages<D, RS, kTma>(a, app, tmK, tmV, ringK, ringV, meta, full, empty, start, end, b0,
                               cum0, cap);
  }
  // The fused store, by the whole warp once every stage is issued: it overlaps
  // the consumers' last stages instead of delaying the first copies.
  __syncwarp();
  if (app.k_new != nullptr) fused_store<D>(a, app, lane, cap);
}

// ---------------------------------------------------------------- consumers

// The CUDA-core consumers (G = 1 or 2 query heads per kv head).
template <int D, int G, int RS>
__device__ void decode_consumer(const DecodeArgs& a, const uint8_t* ringK, const uint8_t* ringV,
                                const StageMeta* meta, uint64_t* full, uint64_t* empty,
                                uint64_t* xfull, uint64_t* xfree, float* xw) {
  constexpr int NCH = D / 64;  // 16-byte chunks of one row per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = a.num_kv_heads;
  const int NS = kBaseWarps / Hkv;
  const int g = warp % Hkv, sub = warp / Hkv;
  const int head0 = g * G;  // first query head of this warp
  const int li = lane & 7, tg = lane >> 3;
  const int row_elems = Hkv * D;

  float qf[G][NCH][8];  // scaled query
  float acc[G][NCH][8];
  float m[G], l[G];
  int b = 0;
  int s = 0;
  uint32_t ph = 0;
  int seg = 0;  // segments finished so far (same count in every warp)

  while (true) {
    if (!mbar_wait(&full[s], ph, a.status)) return;
    const StageMeta md = meta[s];
    if (md.flags & F_DONE) break;

    if (md.flags & F_NEW) {
      b = md.b;
      const uint16_t* qrow = a.q + (int64_t)b * a.q_stride + (int64_t)head0 * D;
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const uint4 u = *reinterpret_cast<const uint4*>(qrow + h * D + (c * 8 + li) * 8);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qf[h][c][2 * e] = bf16lo(w[e]) * a.scale_log2;
            qf[h][c][2 * e + 1] = bf16hi(w[e]) * a.scale_log2;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][c][e] = 0.f;
        }
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
    }

    const uint16_t* Ks = reinterpret_cast<const uint16_t*>(ringK + (size_t)s * stage_half_bytes<D>());
    const uint16_t* Vs = reinterpret_cast<const uint16_t*>(ringV + (size_t)s * stage_half_bytes<D>());

    // Scores of this warp's 2 x 4 tokens for its G query heads.
    float sc[2][G];
    bool valid[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int tl = (p * NS + sub) * 4 + tg;
      valid[p] = tl < md.n;
      const uint4* kr = reinterpret_cast<const uint4*>(Ks + (size_t)tl * row_elems + g * D);
      uint4 kv[NCH];
#pragma unroll
      for (int c = 0; c < NCH; ++c) kv[c] = kr[c * 8 + li];
      float xs[G];  // this lane's partial dot products
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const uint32_t w[4] = {kv[c].x, kv[c].y, kv[c].z, kv[c].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {  // packed fp32x2 FMA: elements 2e, 2e+1
            const float2 r = __ffma2_rn(make_float2(qf[h][c][2 * e], qf[h][c][2 * e + 1]),
                                        make_float2(bf16lo(w[e]), bf16hi(w[e])),
                                        make_float2(acc0, acc1));
            acc0 = r.x;
            acc1 = r.y;
          }
        }
        xs[h] = acc0 + acc1;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float x = xs[h];
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        sc[p][h] = valid[p] ? x : -INFINITY;
      }
    }

    // Online softmax: one max update per stage (warp-uniform per head).
    float pr[2][G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = fmaxf(sc[0][h], sc[1][h]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (mx > m[h]) {
          const float alpha = fast_exp2(m[h] - mx);  // exp2(-inf) = 0 on the first stage
          m[h] = mx;
          l[h] *= alpha;
#pragma unroll
          for (int c = 0; c < NCH; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][c][e] *= alpha;
        }
        const float mu = m[h] == -INFINITY ? 0.f : m[h];
        pr[0][h] = fast_exp2(sc[0][h] - mu);
        pr[1][h] = fast_exp2(sc[1][h] - mu);
        l[h] += pr[0][h] + pr[1][h];
    }

    // acc += p * v
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int tl = (p * NS + sub) * 4 + tg;
      const uint4* vr = reinterpret_cast<const uint4*>(Vs + (size_t)tl * row_elems + g * D);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        uint4 u = vr[c * 8 + li];
        if (!valid[p]) u = make_uint4(0, 0, 0, 0);  // stale smem may hold NaN patterns
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 r = __ffma2_rn(make_float2(pr[p][h], pr[p][h]),
                                        make_float2(bf16lo(w[e]), bf16hi(w[e])),
                                        make_float2(acc[h][c][2 * e], acc[h][c][2 * e + 1]));
            acc[h][c][2 * e] = r.x;
            acc[h][c][2 * e + 1] = r.y;
          }
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == RS) {
      s = 0;
      ph ^= 1u;
    }

    if (!(md.flags & F_LAST)) continue;

    // ---- end of this CTA's segment of sequence b: reduce over the 4 token groups
#pragma unroll
    for (int h = 0; h < G; ++h) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 8);
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 16);
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc[h][c][e] += __shfl_xor_sync(0xffffffffu, acc[h][c][e], 8);
          acc[h][c][e] += __shfl_xor_sync(0xffffffffu, acc[h][c][e], 16);
        }
    }
    bool writer = true;
    if (NS > 1) {
      // Several warps share kv head g.  Hand-off through shared memory with
      // bounded mbarrier waits: warps sub > 0 publish (acc, m, l) and arrive
      // on xfull[g]; warp sub 0 waits, combines by log-sum-exp and releases
      // the buffer through xfree[g] before the next segment's hand-off.
      writer = sub == 0;
      if (!writer) {
        if (seg > 0 && !mbar_wait(&xfree[g], (uint32_t)((seg - 1) & 1), a.status)) return;
        float* mine = xw + (size_t)warp * G * (D + 2);
        if (tg == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int c = 0; c < NCH; ++c)
#pragma unroll
              for (int e = 0; e < 8; ++e) mine[h * (D + 2) + (c * 8 + li) * 8 + e] = acc[h][c][e];
            if (li == 0) {
              mine[h * (D + 2) + D] = m[h];
              mine[h * (D + 2) + D + 1] = l[h];
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&xfull[g]);
      } else {
        if (!mbar_wait(&xfull[g], (uint32_t)(seg & 1), a.status)) return;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float M = m[h];
          for (int k = 1; k < NS; ++k)
            M = fmaxf(M, xw[(size_t)(g + k * Hkv) * G * (D + 2) + h * (D + 2) + D]);
          const float Mu = M == -INFINITY ? 0.f : M;
          const float w0 = fast_exp2(m[h] - Mu);
          float ls = w0 * l[h];
#pragma unroll
          for (int c = 0; c < NCH; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][c][e] *= w0;
          for (int k = 1; k < NS; ++k) {
            const float* o = xw + (size_t)(g + k * Hkv) * G * (D + 2) + h * (D + 2);
            const float w = fast_exp2(o[D] - Mu);
            ls += w * o[D + 1];
#pragma unroll
            for (int c = 0; c < NCH; ++c)
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[h][c][e] += w * o[(c * 8 + li) * 8 + e];
          }
          m[h] = M;
          l[h] = ls;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&xfree[g]);
      }
    }
    ++seg;
    if (!writer || tg != 0) continue;
    if (!(md.flags & (F_ENTERED | F_EXITS))) {
      // whole sequence inside this CTA: normalise and write bf16
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float inv = 1.f / l[h];
        uint16_t* orow = a.out + (int64_t)b * a.out_stride + (int64_t)(head0 + h) * D;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          uint4 u;
          u.x = pack_bf16x2(acc[h][c][0] * inv, acc[h][c][1] * inv);
          u.y = pack_bf16x2(acc[h][c][2] * inv, acc[h][c][3] * inv);
          u.z = pack_bf16x2(acc[h][c][4] * inv, acc[h][c][5] * inv);
          u.w = pack_bf16x2(acc[h][c][6] * inv, acc[h][c][7] * inv);
          *reinterpret_cast<uint4*>(orow + (c * 8 + li) * 8) = u;
        }
      }
    } else {
      const int slot = (md.flags & F_ENTERED) ? 0 : 1;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float* dst =
            a.part + (((size_t)blockIdx.x * 2 + slot) * a.num_heads + head0 + h) * part_stride<D>();
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float4* d4 = reinterpret_cast<float4*>(dst + (c * 8 + li) * 8);
          d4[0] = make_float4(acc[h][c][0], acc[h][c][1], acc[h][c][2], acc[h][c][3]);
          d4[1] = make_float4(acc[h][c][4], acc[h][c][5], acc[h][c][6], acc[h][c][7]);
        }
        if (li == 0) {
          dst[D] = m[h];
          dst[D + 1] = l[h];
        }
      }
    }
  }
}

// The CUDA-core split kernel: 8 consumer warps + 1 producer warp.
template <int D, int G>
__global__ void __launch_bounds__((kBaseWarps + 1) * 32, 1)
    decode_split_kernel(const DecodeArgs a, const AppendArgs app) {
  static_assert(G <= 2, "groups of 4 and 8 query heads take the tensor-core kernel");
  constexpr int RS = kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ringK = smem;
  uint8_t* ringV = smem + RS * stage_half_bytes<D>();
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + 2 * RS * stage_half_bytes<D>());
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + RS);
  uint64_t* empty = full + RS;
  uint64_t* xfull = empty + RS;
  uint64_t* xfree = xfull + kBaseWarps;
  float* xw = reinterpret_cast<float*>(xfree + kBaseWarps);

  if (threadIdx.x == 0) {
    // The merge kernel may be scheduled now; it waits for this grid to finish.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = 0; i < RS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kBaseWarps);
    }
    const int ns = kBaseWarps / a.num_kv_heads;
    for (int i = 0; i < kBaseWarps; ++i) {
      mbar_init(&xfull[i], ns > 1 ? ns - 1 : 1);
      mbar_init(&xfree[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if (warp == kBaseWarps)
    decode_producer<D, RS, false>(a, app, nullptr, nullptr, ringK, ringV, meta, full, empty);
  else
    decode_consumer<D, G, RS>(a, ringK, ringV, meta, full, empty, xfull, xfree, xw);
  // Launched as a programmatic dependent (the decode rows of a mixed step,
  // beside the prefill): do not complete before the prerequisite grid.
  // Otherwise a no-op.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- tensor-core consumers
//
// Stage layout of the tensor-core path: the producer's 4-D tensor copy lands
// a stage half (K or V) as [kv head][64-column panel][T tokens][128 bytes]
// with the 128-byte swizzle (16-byte chunk c of a token's 128-byte panel row
// sits at chunk c ^ (token & 7)), so the eight token rows an ldmatrix reads
// fall in eight different bank groups.  Every region of T rows is 1 KiB
// aligned (T >= 8).
//
// A warp serves kv head g and the 8 tokens sub*8 .. sub*8+7 of every stage:
//   S = q K^T:    mma m16n8k16, M = the G query heads of kv head g (rows G..15
//                 zero), N = the 8 tokens, K = head_dim (D / 16 steps); the q
//                 fragments stay in registers for the whole sequence;
//   O^T += V^T P^T: mma m16n8k8, M = 16 columns of head_dim (D / 16 tiles),
//                 N = 8 query heads, K = the 8 tokens.  The S accumulator of
//                 thread (r = lane / 4, c = lane % 4) holds head r's scores
//                 of tokens 2c, 2c + 1, which is exactly that thread's B
//                 fragment of P^T, so P never leaves the thread; V^T comes from
//                 transposing shared-memory loads.
// Thread (r, c) keeps head r's running max m and row sum l (shared by the
// quad), and O[head 2c + x][16 i + r + 8 y] in ot[i][2 y + x].  O and l are
// rescaled only when a head's max grows by more than 2^8 (exact: O and l keep
// the same stale reference, and P <= 2^8 fits bf16).

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// d += a b: m16n8k16, bf16 inputs, fp32 accumulate (rows 8..15 of a are zero).
__device__ __forceinline__ void mma_k16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// d += a b: m16n8k8, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// Byte offset of 16-byte chunk q of token row `row` in a stage half.
__device__ __forceinline__ uint32_t chunk_off(uint32_t region, int T, int row, int q) {
  return region + (uint32_t)(((q >> 3) * T + row) * 128 + (((q & 7) ^ (row & 7)) << 4));
}

template <int D, int G, int RS>
__device__ void decode_consumer_mma(const DecodeArgs& a, const AppendArgs& app,
                                    const uint8_t* ringK, const uint8_t* ringV,
                                    const StageMeta* meta, uint64_t* full, uint64_t* empty,
                                    uint64_t* xfull, uint64_t* xfree, float* xw) {
  constexpr int P = D / 64;   // 128-byte panels of a row
  constexpr int NQ = D / 8;   // 16-byte chunks of a row
  constexpr int KS = D / 16;  // k-steps of S; tiles of O^T
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = a.num_kv_heads;
  const int NS = kBaseWarps / Hkv;
  const int g = warp % Hkv, sub = warp / Hkv;
  const int T = kTokensAllHeads / Hkv;
  const int head0 = g * G;
  const int r = lane >> 2, c = lane & 3;
  const bool srow = r < G;                    // this thread's S row is a real head
  const bool ocol0 = 2 * c < G, ocol1 = 2 * c + 1 < G;  // its O columns are real heads
  const uint32_t region = (uint32_t)(g * P * T * 128);
  const int mrow = sub * 8 + (lane & 7);  // ldmatrix: lane L gives row L % 8 of matrix L / 8
  const int msel = lane >> 3;
  const uint32_t kbase = smem_u32(ringK), vbase = smem_u32(ringV);

  uint32_t qa[KS][2];
  float ot[KS][4];
  float m = -INFINITY, l = 0.f;
  int b = 0;
  int s = 0;
  uint32_t ph = 0;
  int seg = 0;

  while (true) {
    if (!mbar_wait(&full[s], ph, a.status)) return;
    const StageMeta md = meta[s];
    if (md.flags & F_DONE) break;
    if (md.flags & F_NEW) {
      b = md.b;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(a.q + (int64_t)b * a.q_stride +
                                                               (int64_t)(head0 + r) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = srow ? qrow[ks * 8 + c] : 0u;
        qa[ks][1] = srow ? qrow[ks * 8 + 4 + c] : 0u;
      }
#pragma unroll
      for (int i = 0; i < KS; ++i) ot[i][0] = ot[i][1] = ot[i][2] = ot[i][3] = 0.f;
      m = -INFINITY;
      l = 0.f;
    }
    const uint32_t kst = kbase + (uint32_t)(s * stage_half_bytes<D>());
    const uint32_t vst = vbase + (uint32_t)(s * stage_half_bytes<D>());
    const int nt = md.n - sub * 8;  // this warp's tokens in the stage (<= 0: none)
    bool patched = false;
    if (nt > 0) {
      if ((md.flags & F_TAIL) && (md.n - 1) >> 3 == sub) {
        // The sequence's last token: its row comes from the new rows (the
        // cache slot is written in this launch).  Lanes 0..15 patch K, 16..31 V.
        const int row = md.n - 1, q = lane & 15;
        if (q < NQ) {
          const uint16_t* src = (lane < 16 ? app.k_new + (int64_t)b * app.k_new_stride
                                           : app.v_new + (int64_t)b * app.v_new_stride) +
                                (int64_t)g * D + q * 8;
          const uint4 u = *reinterpret_cast<const uint4*>(src);
          const uint32_t dst = (lane < 16 ? kst : vst) + chunk_off(region, T, row, q);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(u.x), "r"(u.y),
                       "r"(u.z), "r"(u.w)
                       : "memory");
        }
        __syncwarp();
        patched = true;
      }
      // S = q K^T for the warp's 8 tokens; two accumulators halve the chain.
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NQ / 4; ++j) {
        uint32_t k0, k1, k2, k3;
        ldsm_x4(kst + chunk_off(region, T, mrow, 4 * j + msel), k0, k1, k2, k3);
        mma_k16(sa, qa[2 * j][0], qa[2 * j][1], k0, k1);
        mma_k16(sb, qa[2 * j + 1][0], qa[2 * j + 1][1], k2, k3);
      }
      float x0 = (sa[0] + sb[0]) * a.scale_log2, x1 = (sa[1] + sb[1]) * a.scale_log2;
      if (2 * c >= nt) x0 = -INFINITY;
      if (2 * c + 1 >= nt) x1 = -INFINITY;
      float mx = fmaxf(x0, x1);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      // Also the first stage of a sequence (m = -inf, alpha = 0, O still zero).
      const bool grow = mx > m + 8.0f;
      if (__any_sync(0xffffffffu, grow)) {
        const float alpha = grow ? fast_exp2(m - mx) : 1.f;
        if (grow) {
          m = mx;
          l *= alpha;
        }
        const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * c);
        const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * c + 4);
#pragma unroll
        for (int i = 0; i < KS; ++i) {
          ot[i][0] *= a0;
          ot[i][1] *= a1;
          ot[i][2] *= a0;
          ot[i][3] *= a1;
        }
      }
      const float p0 = fast_exp2(x0 - m), p1 = fast_exp2(x1 - m);
      l += p0 + p1;
      const uint32_t pb = pack_bf16x2(p0, p1);
      // O^T += V^T P^T.  V rows past the warp's tokens may hold anything: zero them.
      const uint32_t keep = 2 * c >= nt ? 0u : (2 * c + 1 >= nt ? 0x0000ffffu : 0xffffffffu);
#pragma unroll
      for (int j = 0; j < NQ / 4; ++j) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vst + chunk_off(region, T, mrow, 4 * j + msel), v0, v1, v2, v3);
        mma_k8(ot[2 * j], v0 & keep, v1 & keep, pb);
        mma_k8(ot[2 * j + 1], v2 & keep, v3 & keep, pb);
      }
    }
    if (patched) fence_proxy_async_smem();  // generic writes before the next tensor copy
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == RS) {
      s = 0;
      ph ^= 1u;
    }
    if (!(md.flags & F_LAST)) continue;

    // ---- end of this CTA's segment of sequence b: heads 2c, 2c + 1 of each thread
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    float mh[2] = {__shfl_sync(0xffffffffu, m, 8 * c), __shfl_sync(0xffffffffu, m, 8 * c + 4)};
    float lh[2] = {__shfl_sync(0xffffffffu, l, 8 * c), __shfl_sync(0xffffffffu, l, 8 * c + 4)};
    const bool oc[2] = {ocol0, ocol1};
    bool writer = true;
    if (NS > 1) {
      // Warps sub > 0 of kv head g publish (O, m, l) of their heads; warp
      // sub 0 combines them by log-sum-exp (bounded mbarrier hand-off).
      writer = sub == 0;
      if (!writer) {
        if (seg > 0 && !mbar_wait(&xfree[g], (uint32_t)((seg - 1) & 1), a.status)) return;
        float* mine = xw + (size_t)warp * G * (D + 2);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!oc[x]) continue;
          float* row = mine + (2 * c + x) * (D + 2);
#pragma unroll
          for (int i = 0; i < KS; ++i) {
            row[16 * i + r] = ot[i][x];
            row[16 * i + r + 8] = ot[i][2 + x];
          }
          if (r == 0) {
            row[D] = mh[x];
            row[D + 1] = lh[x];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&xfull[g]);
      } else {
        if (!mbar_wait(&xfull[g], (uint32_t)(seg & 1), a.status)) return;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!oc[x]) continue;
          float M = mh[x];
          for (int k = 1; k < NS; ++k)
            M = fmaxf(M, xw[(size_t)(g + k * Hkv) * G * (D + 2) + (2 * c + x) * (D + 2) + D]);
          const float Mu = M == -INFINITY ? 0.f : M;
          const float w0 = fast_exp2(mh[x] - Mu);
          float ls = w0 * lh[x];
#pragma unroll
          for (int i = 0; i < KS; ++i) {
            ot[i][x] *= w0;
            ot[i][2 + x] *= w0;
          }
          for (int k = 1; k < NS; ++k) {
            const float* row = xw + (size_t)(g + k * Hkv) * G * (D + 2) + (2 * c + x) * (D + 2);
            const float w = fast_exp2(row[D] - Mu);
            ls += w * row[D + 1];
#pragma unroll
            for (int i = 0; i < KS; ++i) {
              ot[i][x] += w * row[16 * i + r];
              ot[i][2 + x] += w * row[16 * i + r + 8];
            }
          }
          mh[x] = M;
          lh[x] = ls;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&xfree[g]);
      }
    }
    ++seg;
    if (!writer) continue;
    if (!(md.flags & (F_ENTERED | F_EXITS))) {
      // whole sequence inside this CTA: normalise and write bf16
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (!oc[x]) continue;
        const float inv = 1.f / lh[x];
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(
            a.out + (int64_t)b * a.out_stride + (int64_t)(head0 + 2 * c + x) * D);
#pragma unroll
        for (int i = 0; i < KS; ++i) {
          orow[16 * i + r] = __float2bfloat16_rn(ot[i][x] * inv);
          orow[16 * i + r + 8] = __float2bfloat16_rn(ot[i][2 + x] * inv);
        }
      }
    } else {
      const int slot = (md.flags & F_ENTERED) ? 0 : 1;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (!oc[x]) continue;
        float* dst = a.part + (((size_t)blockIdx.x * 2 + slot) * a.num_heads + head0 + 2 * c + x) *
                                  part_stride<D>();
#pragma unroll
        for (int i = 0; i < KS; ++i) {
          dst[16 * i + r] = ot[i][x];
          dst[16 * i + r + 8] = ot[i][2 + x];
        }
        if (r == 0) {
          dst[D] = mh[x];
          dst[D + 1] = lh[x];
        }
      }
    }
  }
}

template <int D, int G>
__host__ __device__ constexpr size_t decode_mma_smem_bytes(int ns) {
  return 1024 + 2 * ns * stage_half_bytes<D>() + ns * sizeof(StageMeta) +
         (2 * ns + 2 * kBaseWarps) * sizeof(uint64_t) + (size_t)kBaseWarps * G * (D + 2) * sizeof(float);
}
template <int D, int G>
__host__ __device__ constexpr int mma_ring_stages() {
  return decode_mma_smem_bytes<D, G>(kStages) <= kSmemPerCta ? kStages : kStages - 1;
}
static_assert(decode_mma_smem_bytes<128, 8>(mma_ring_stages<128, 8>()) <= kSmemPerCta,
              "decode CTA smem");

// The tensor-core split kernel: 8 consumer warps + 1 producer warp.  The ring
// starts at the first 1 KiB boundary of the dynamic shared memory (the
// swizzled tensor copies need it).
template <int D, int G>
__global__ void __launch_bounds__((kBaseWarps + 1) * 32, 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const DecodeArgs a,
                      const AppendArgs app) {
  constexpr int RS = mma_ring_stages<D, G>();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ringK = smem;
  uint8_t* ringV = smem + RS * stage_half_bytes<D>();
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + 2 * RS * stage_half_bytes<D>());
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + RS);
  uint64_t* empty = full + RS;
  uint64_t* xfull = empty + RS;
  uint64_t* xfree = xfull + kBaseWarps;
  float* xw = reinterpret_cast<float*>(xfree + kBaseWarps);

  if (threadIdx.x == 0) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = 0; i < RS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kBaseWarps);
    }
    const int ns = kBaseWarps / a.num_kv_heads;
    for (int i = 0; i < kBaseWarps; ++i) {
      mbar_init(&xfull[i], ns > 1 ? ns - 1 : 1);
      mbar_init(&xfree[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if (warp == kBaseWarps)
    decode_producer<D, RS, true>(a, app, &tmK, &tmV, ringK, ringV, meta, full, empty);
  else
    decode_consumer_mma<D, G, RS>(a, app, ringK, ringV, meta, full, empty, xfull, xfree, xw);
  // As in decode_split_kernel: a programmatic dependent completes after its
  // prerequisite grid.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Combines the partials of every sequence that crosses a CTA boundary.
// Block (j, h) handles query head h of the sequence that leaves CTA j, if that
// sequence did not also enter CTA j; its partials are CTA j's "exits" slot
// and the "entered" slots of the following CTAs it reaches.  One thread per
// element of head_dim.  Launched as a programmatic dependent of the split
// kernel: it may start while the split kernel drains and waits for the split
// grid's completion (and memory flush) before reading anything.  Its loads
// take two dependent rounds: split_seq[j-1 .. j+30] (one per lane), then m, l
// and the accumulator element of every part at once.
template <int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(const float* __restrict__ part,
                                                         const int* __restrict__ split_seq,
                                                         int ctas, int num_heads,
                                                         uint16_t* __restrict__ out,
                                                         int64_t out_stride) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int j = blockIdx.x, h = blockIdx.y, e = threadIdx.x, lane = e & 31;
  const int il = j - 1 + lane;
  const int sv = (il >= 0 && il < ctas) ? split_seq[il] : -1;
  const int b = __shfl_sync(0xffffffffu, sv, 1);
  if (b < 0 || __shfl_sync(0xffffffffu, sv, 0) == b) return;
  // Bit k: the sequence also leaves CTA j + k; it ends in the first CTA that
  // it does not leave.
  const unsigned run = __ballot_sync(0xffffffffu, sv == b) >> 1;
  int last = j + (__ffs(~run) - 1);
  if (run == 0x7fffffffu)  // leaves 31 CTAs in a row: walk on
    while (last < ctas - 1 && split_seq[last] == b) ++last;
  if (last > ctas - 1) last = ctas - 1;
  constexpr int S = part_stride<D>();
  const int nparts = last - j + 1;
  float num = 0.f, den = 0.f;
  constexpr int kBatch = 8;
  if (nparts <= kBatch) {
    float av[kBatch], mv[kBatch], lv[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      av[k] = 0.f;
      mv[k] = -INFINITY;
      lv[k] = 0.f;
      if (k < nparts) {
        const float* p = part + (((size_t)(j + k) * 2 + (k == 0 ? 1 : 0)) * num_heads + h) * S;
        av[k] = p[e];
        mv[k] = p[D];
        lv[k] = p[D + 1];
      }
    }
    float M = mv[0];
#pragma unroll
    for (int k = 1; k < kBatch; ++k) M = fmaxf(M, mv[k]);
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (k < nparts) {
        const float w = fast_exp2(mv[k] - M);
        num += w * av[k];
        den += w * lv[k];
      }
    }
  } else {
    float M = -INFINITY;
    for (int i = j; i <= last; ++i)
      M = fmaxf(M, part[(((size_t)i * 2 + (i == j ? 1 : 0)) * num_heads + h) * S + D]);
    for (int i = j; i <= last; ++i) {
      const float* p = part + (((size_t)i * 2 + (i == j ? 1 : 0)) * num_heads + h) * S;
      const float w = fast_exp2(p[D] - M);
      num += w * p[e];
      den += w * p[D + 1];
    }
  }
  const __nv_bfloat16 r = __float2bfloat16_rn(num / den);
  out[(int64_t)b * out_stride + (int64_t)h * D + e] = *reinterpret_cast<const uint16_t*>(&r);
}

// Launches a split kernel, as a programmatic dependent of the stream's
// previous kernel when pdl is set (it may then start beside that kernel).
template <typename... Params, typename... Args>
cudaError_t launch_split(void (*kernel)(Params...), int ctas, size_t smem, cudaStream_t stream,
                         bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3((kBaseWarps + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int D, int G>
cudaError_t launch_decode_t(const DecodeArgs& a, const AppendArgs& app, int ctas,
                            cudaStream_t stream, bool pdl) {
  const size_t smem = decode_smem_bytes<D, G>(kStages);
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_split(decode_split_kernel<D, G>, ctas, smem, stream, pdl, a, app);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, a.num_heads);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, (const float*)a.part,
                            (const int*)a.split_seq, ctas, a.num_heads, a.out, a.out_stride);
}

// Tensor maps of one layer's K and V caches for the tensor-core path.  The
// stage box is {64 columns, T tokens, D / 64 panels, Hkv heads} over a 4-D
// view (column, token row, panel, head) of the [rows, Hkv, D] cache, which
// lands a stage as [head][panel][token][64] in one copy per half; if the
// driver does not take that view, a 3-D map (column, head, row) with a box
// {64, 1, T} per (head, panel) gives the same layout.
bool decode_maps(const DecodeArgs& a, int D, CUtensorMap* mk, CUtensorMap* mv, int* per_head) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!enc) return false;
  const int Hkv = a.num_kv_heads, T = kTokensAllHeads / Hkv;
  const cuuint64_t rows = (cuuint64_t)a.num_blocks * a.block_size;
  {
    cuuint64_t dims[4] = {64, rows, (cuuint64_t)(D / 64), (cuuint64_t)Hkv};
    cuuint64_t strides[3] = {(cuuint64_t)Hkv * D * 2, 128, (cuuint64_t)D * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)T, (cuuint32_t)(D / 64), (cuuint32_t)Hkv};
    cuuint32_t es[4] = {1, 1, 1, 1};
    bool ok = true;
    for (int i = 0; i < 2 && ok; ++i)
      ok = enc(i == 0 ? mk : mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<uint16_t*>(i == 0 ? a.k_cache : a.v_cache), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    if (ok) {
      *per_head = 0;
      return true;
    }
  }
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)T};
  cuuint32_t es[3] = {1, 1, 1};
  for (int i = 0; i < 2; ++i)
    if (enc(i == 0 ? mk : mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<uint16_t*>(i == 0 ? a.k_cache : a.v_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  *per_head = 1;
  return true;
}

cudaError_t launch_merge(const DecodeArgs& a, int D, int ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, a.num_heads);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128)
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<128>, (const float*)a.part,
                              (const int*)a.split_seq, ctas, a.num_heads, a.out, a.out_stride);
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<64>, (const float*)a.part,
                            (const int*)a.split_seq, ctas, a.num_heads, a.out, a.out_stride);
}

template <int D, int G>
cudaError_t launch_decode_mma_t(DecodeArgs a, const AppendArgs& app, int ctas, cudaStream_t stream,
                                bool pdl) {
  CUtensorMap mk, mv;
  if (!decode_maps(a, D, &mk, &mv, &a.tma_per_head)) return cudaErrorInvalidValue;
  const size_t smem = decode_mma_smem_bytes<D, G>(mma_ring_stages<D, G>());
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_split(decode_mma_kernel<D, G>, ctas, smem, stream, pdl, mk, mv, a, app);
  if (e != cudaSuccess) return e;
  return launch_merge(a, D, ctas, stream);
}

// The tensor-core consumers serve groups of 4 and 8 query heads, where the
// CUDA-core consumers are issue-bound (2 FMAs per K/V byte at G = 4); at one
// or two heads per kv head the CUDA-core consumers stream at the HBM rate and
// measured faster (decode B64 at 16/8/128: 97.4 against 99.7 us per call).
template <int D, int G>
constexpr bool use_mma() {
  return G >= 4;
}

template <int D, int G>
cudaError_t launch_decode_any(const DecodeArgs& a, const AppendArgs& app, int ctas,
                              cudaStream_t stream, bool pdl) {
  if constexpr (use_mma<D, G>())
    return launch_decode_mma_t<D, G>(a, app, ctas, stream, pdl);
  else
    return launch_decode_t<D, G>(a, app, ctas, stream, pdl);
}

}  // namespace

bool decode_supported(int num_heads, int num_kv_heads, int head_dim) {
  if (num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads) return false;
  if (num_kv_heads != 1 && num_kv_heads != 2 && num_kv_heads != 4 && num_kv_heads != 8)
    return false;
  const int G = num_heads / num_kv_heads;
  if (head_dim == 128 || head_dim == 64) return G == 1 || G == 2 || G == 4 || G == 8;
  return false;
}

DecodePlan plan_decode(int num_seqs, int num_heads, int head_dim, int max_context_len,
                       int num_sms) {
  // num_sms: the SMs the split kernel may take (one persistent CTA each).
  DecodePlan p{};
  long long upper = (long long)num_seqs * (max_context_len > 0 ? max_context_len : 0);
  long long ctas = (upper + 63) / 64;  // at least 64 tokens per CTA
  if (ctas > num_sms) ctas = num_sms;
  if (ctas < 1) ctas = 1;
  p.ctas = (int)ctas;
  p.part_bytes = (size_t)ctas * 2 * num_heads * (head_dim + 4) * sizeof(float);
  p.split_bytes = (size_t)ctas * sizeof(int);
  p.total_bytes = ((p.part_bytes + 255) / 256) * 256 + ((p.split_bytes + 255) / 256) * 256;
  return p;
}

cudaError_t launch_decode(const uint16_t* q, int64_t q_stride, const uint16_t* k_cache,
                          const uint16_t* v_cache, int64_t num_blocks, int block_size,
                          const int32_t* block_tables, int max_blocks, const int32_t* ctx,
                          int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                          float softmax_scale, const DecodePlan& plan, void* workspace,
                          uint16_t* out, int64_t out_stride, int* status, cudaStream_t stream,
                          const DecodeAppend* app, const DecodeRowsOf* rows_of, bool pdl) {
  DecodeArgs a;
  AppendArgs ap{};
  if (app) {
    ap.k_new = app->k;
    ap.v_new = app->v;
    ap.k_new_stride = app->k_stride;
    ap.v_new_stride = app->v_stride;
    ap.slot_mapping = app->slot_mapping;
    ap.k_cache_w = app->k_cache;
    ap.v_cache_w = app->v_cache;
  }
  a.q = q;
  a.q_stride = q_stride;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.ctx = rows_of ? nullptr : ctx;
  a.cu_q = rows_of ? rows_of->cu_q : nullptr;
  a.cu_k = rows_of ? rows_of->cu_k : nullptr;
  a.cu_off = rows_of ? rows_of->offset : 0;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.part = reinterpret_cast<float*>(workspace);
  a.split_seq = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(workspace) +
                                       ((plan.part_bytes + 255) / 256) * 256);
  a.out = out;
  a.out_stride = out_stride;
  a.status = status;
  a.tma_per_head = 0;
  const int G = num_heads / num_kv_heads;
  if (head_dim == 128) {
    switch (G) {
      case 1: return launch_decode_any<128, 1>(a, ap, plan.ctas, stream, pdl);
      case 2: return launch_decode_any<128, 2>(a, ap, plan.ctas, stream, pdl);
      case 4: return launch_decode_any<128, 4>(a, ap, plan.ctas, stream, pdl);
      case 8: return launch_decode_any<128, 8>(a, ap, plan.ctas, stream, pdl);
    }
  } else if (head_dim == 64) {
    switch (G) {
      case 1: return launch_decode_any<64, 1>(a, ap, plan.ctas, stream, pdl);
      case 2: return launch_decode_any<64, 2>(a, ap, plan.ctas, stream, pdl);
      case 4: return launch_decode_any<64, 4>(a, ap, plan.ctas, stream, pdl);
      case 8: return launch_decode_any<64, 8>(a, ap, plan.ctas, stream, pdl);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvp
