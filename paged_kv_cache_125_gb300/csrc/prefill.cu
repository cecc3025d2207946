// attn_prefill_varlen: causal varlen prefill with a prefix cache, on the
// 5th-generation tensor cores (tcgen05 + tensor memory), fed by TMA.
//
// Source: "Nano vLLM 解读（5）：解析 ModelRunner", prepare_prefill and the
// FlashAttention argument list (cu_seqlens_q / cu_seqlens_k / max_seqlen_q /
// max_seqlen_k; block_tables only when a prefix is cached, in which case the
// keys come from the paged cache); "nano-vLLM-1" "4. prefill 输入打包" (query
// positions start at num_cached_tokens); attention is softmax(QK^T/sqrt(d))V
// with the causal mask of "【nano-vllm 学习】04 …", "KV-Cache … 是什么？".
//
// Work unit ("item"): one sequence b, one kv head g, and a tile of 128 query
// rows = 128/G tokens x the G query heads that share kv head g, so every K/V
// tile in shared memory serves all G heads in one MMA.  Query row (token t,
// head h) sits at absolute position c_b + q0 + t and sees keys 0 .. that
// position.  An item walks kv tiles of 128 keys up to its last visible key.
//
// Persistent CTAs (one per SM), 6 warps:
//   warp 4  TMA producer: Q tile (2 slots), K tiles (2 slots), V tiles
//           (2 slots).  In paged mode a kv tile is loaded as block-sized
//           sub-boxes addressed through the block table (gather folded into
//           the loads).
//   warp 5  MMA issuer + tensor-memory owner.  S_j = Q K_j^T into one of two
//           128-column TMEM buffers (issued two tiles ahead of the PV
//           stream), O += P_j V_j into a third TMEM region.
//   warps 0-3 softmax / correction / epilogue: thread r owns query row r
//           (TMEM lane r).  Reads S with tcgen05.ld, masks only where the
//           tile crosses the diagonal, keeps a running max per row and
//           rescales O only when the max grows by more than 2^8 (exact: O and
//           the row sum share the stale reference), writes P as bf16 into
//           shared memory in the 128-byte-swizzled K-major layout the MMA
//           reads, and at the end of an item normalises O and stores bf16.
#include <cudaTypedefs.h>

#include <mutex>

#include "kvp_device.cuh"

namespace kvp {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per kv tile
constexpr int kSoftmaxWarps = 8;  // two threads per query row, 64 columns each
constexpr int kThreadsPF = (kSoftmaxWarps + 2) * 32;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct PrefillArgs {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_tables;
  int max_blocks;
  int64_t num_blocks;
  int block_size;
  int paged;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int group;        // G
  int tok_per_tile; // 128 / G
  int sub_rows;     // rows per TMA box of a kv tile (paged: min(bs, 128))
  int max_tiles;    // ceil(max_seqlen_q / tok_per_tile)
  float scale_log2;
  uint16_t* out;
  int64_t out_stride;
  int* status;
};

template <int D>
struct Layout {
  static constexpr uint32_t kPanels = D / 64;
  static constexpr uint32_t kPanelBytes = 128 * 128;  // 128 rows x 128 bytes
  static constexpr uint32_t kQBytes = kBM * D * 2;
  static constexpr uint32_t kKVBytes = kBN * D * 2;
  static constexpr uint32_t kPBytes = kBM * kBN * 2;
  static constexpr uint32_t kQ = 0;                    // 2 slots
  static constexpr uint32_t kK = kQ + 2 * kQBytes;     // 2 slots
  static constexpr uint32_t kV = kK + 2 * kKVBytes;    // 2 slots
  static constexpr uint32_t kP = kV + 2 * kKVBytes;    // 1 buffer
  static constexpr uint32_t kX = kP + kPBytes;      // row-half exchange [2][2][128] fp32
  static constexpr uint32_t kBar = kX + 2 * 2 * kBM * 4;
  static constexpr uint32_t kNumBars = 22;
  static constexpr uint32_t kTotal = kBar + kNumBars * 8 + 16;
  // The dynamic shared memory base is 1 KiB aligned on this architecture (the
  // kernel checks it and reports KVP_ERR_DEVICE_DATA otherwise); keep a small
  // slack only.
  static constexpr uint32_t kAlloc = kTotal + 128;
};

// Barrier indices.
enum : int {
  B_QFULL = 0,   // [2]
  B_QEMPTY = 2,  // [2]
  B_KFULL = 4,   // [2]
  B_KEMPTY = 6,  // [2]
  B_VFULL = 8,   // [2]
  B_VEMPTY = 10, // [2]
  B_SFULL = 12,  // [2]
  B_PFULL = 14,
  B_ODONE = 15,
  B_OFREE = 16,
  B_DRAIN = 17,
  B_XCH = 18,    // [4]: the two warps of one lane quarter exchange row halves
};

struct Item {
  int b, g, q0, rows_tok, q_len, cached, k_len, kv_end, n_tiles;
  int q_row0;   // packed row of the item's first query token
  int k_row0;   // packed row of the sequence's first key (packed mode)
};

__device__ __forceinline__ bool decode_item(const PrefillArgs& a, int L, Item& it) {
  const int per_r = a.num_seqs * a.num_kv_heads;
  const int r = L / per_r;
  const int rem = L - r * per_r;
  it.b = rem / a.num_kv_heads;
  it.g = rem - it.b * a.num_kv_heads;
  const int cq0 = a.cu_q[it.b], cq1 = a.cu_q[it.b + 1];
  const int ck0 = a.cu_k[it.b], ck1 = a.cu_k[it.b + 1];
  it.q_len = cq1 - cq0;
  it.k_len = ck1 - ck0;
  if (it.q_len <= 0 || it.k_len < it.q_len) {
    if (it.q_len > 0 && r == 0 && it.g == 0) record_error(a.status, KVP_ERR_DEVICE_DATA);
    return false;
  }
  const int ntiles = (it.q_len + a.tok_per_tile - 1) / a.tok_per_tile;
  if (r >= ntiles) return false;
  const int t = ntiles - 1 - r;  // heaviest tiles (largest t) come first
  it.q0 = t * a.tok_per_tile;
  it.rows_tok = min(a.tok_per_tile, it.q_len - it.q0);
  it.cached = it.k_len - it.q_len;
  it.kv_end = it.cached + it.q0 + it.rows_tok;  // keys visible to the last row
  it.n_tiles = (it.kv_end + kBN - 1) / kBN;
  it.q_row0 = cq0 + it.q0;
  it.k_row0 = ck0;
  return true;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ producer

template <int D>
__device__ void producer_role(const PrefillArgs& a, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                              const CUtensorMap* tmV, uint8_t* smem, uint64_t* bars) {
  using Lay = Layout<D>;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    prefetch_tensormap(tmQ);
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
  }
  const int total_items = a.max_tiles * a.num_seqs * a.num_kv_heads;
  int item_idx = 0;
  uint32_t jt = 0;
  for (int L = blockIdx.x; L < total_items; L += gridDim.x) {
    Item it;
    if (!decode_item(a, L, it)) continue;
    // Q tile: 128/G tokens x G heads x D, one box per 64-column panel.
    {
      const int slot = item_idx & 1;
      const uint32_t par = (item_idx >> 1) & 1;
      if (!mbar_wait(&bars[B_QEMPTY + slot], par ^ 1u, a.status)) return;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[B_QFULL + slot], Lay::kQBytes);
        uint8_t* dst = smem + Lay::kQ + slot * Lay::kQBytes;
        for (int p = 0; p < (int)Lay::kPanels; ++p)
          tma_load_3d(dst + p * Lay::kPanelBytes, tmQ, p * 64, it.g * a.group, it.q_row0,
                      &bars[B_QFULL + slot]);
      }
    }
    // Block ids of this item, 32 logical blocks per warp-wide window.
    int win_base = -1, win_val = -1;
    for (int j = 0; j < it.n_tiles; ++j, ++jt) {
      const int st = jt & 1;
      const uint32_t par = (jt >> 1) & 1;
      // Rows of this tile that exist (keys < k_len); sub-boxes past them are not loaded.
      const int key0 = j * kBN;
      int nsub, rows_per_box;
      if (a.paged) {
        rows_per_box = a.sub_rows;
        const int valid = min(kBN, it.k_len - key0);
        nsub = (valid + rows_per_box - 1) / rows_per_box;
      } else {
        rows_per_box = kBN;
        nsub = 1;
      }
      const uint32_t bytes = (uint32_t)(nsub * rows_per_box * D * 2);
      // physical row of every sub-box (paged: through the block table)
      int rowi[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rowi[i] = 0;
      if (a.paged) {
        for (int i = 0; i < nsub; ++i) {
          const int key = key0 + i * rows_per_box;
          const int lb = key / a.block_size;
          const int wb = lb & ~31;
          if (wb != win_base) {  // warp-uniform
            win_base = wb;
            const int e = wb + lane;
            win_val = e < a.max_blocks ? a.block_tables[(int64_t)it.b * a.max_blocks + e] : -1;
          }
          int phys = __shfl_sync(0xffffffffu, win_val, lb - wb);
          if (phys < 0 || phys >= a.num_blocks) {
            if (lane == 0) record_error(a.status, KVP_ERR_DEVICE_DATA);
            phys = 0;  // never address a block outside the pool
          }
          rowi[i] = phys * a.block_size + (key - lb * a.block_size);
        }
      } else {
        rowi[0] = it.k_row0 + key0;
      }
      for (int kv = 0; kv < 2; ++kv) {
        const int full = kv == 0 ? B_KFULL : B_VFULL;
        const int empty = kv == 0 ? B_KEMPTY : B_VEMPTY;
        if (!mbar_wait(&bars[empty + st], par ^ 1u, a.status)) return;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[full + st], bytes);
          uint8_t* dst = smem + (kv == 0 ? Lay::kK : Lay::kV) + st * Lay::kKVBytes;
          const CUtensorMap* map = kv == 0 ? tmK : tmV;
          for (int i = 0; i < nsub; ++i)
            for (int p = 0; p < (int)Lay::kPanels; ++p)
              tma_load_3d(dst + p * Lay::kPanelBytes + i * rows_per_box * 128, map, p * 64, it.g,
                          rowi[i], &bars[full + st]);
        }
      }
    }
    ++item_idx;
  }
}

// ------------------------------------------------------------------ MMA issuer

// Walks the (item, kv tile) sequence of this CTA.
struct TileIter {
  int L;        // current item index (global)
  int j;        // tile within item
  int item_idx; // items of this CTA so far
  uint32_t jt;  // global tile counter
  Item it;
  bool valid;
};

__device__ __forceinline__ void iter_begin(const PrefillArgs& a, TileIter& t) {
  const int total_items = a.max_tiles * a.num_seqs * a.num_kv_heads;
  t.item_idx = 0;
  t.jt = 0;
  t.j = 0;
  t.valid = false;
  for (t.L = blockIdx.x; t.L < total_items; t.L += gridDim.x)
    if (decode_item(a, t.L, t.it)) {
      t.valid = true;
      return;
    }
}

__device__ __forceinline__ void iter_next(const PrefillArgs& a, TileIter& t) {
  ++t.jt;
  if (++t.j < t.it.n_tiles) return;
  t.j = 0;
  ++t.item_idx;
  const int total_items = a.max_tiles * a.num_seqs * a.num_kv_heads;
  t.valid = false;
  for (t.L += gridDim.x; t.L < total_items; t.L += gridDim.x)
    if (decode_item(a, t.L, t.it)) {
      t.valid = true;
      return;
    }
}

template <int D>
__device__ bool issue_s(const PrefillArgs& a, const TileIter& s, uint8_t* smem, uint64_t* bars,
                        uint32_t tbase) {
  using Lay = Layout<D>;
  const int lane = threadIdx.x & 31;
  const int qslot = s.item_idx & 1;
  if (s.j == 0 && !mbar_wait(&bars[B_QFULL + qslot], (s.item_idx >> 1) & 1, a.status)) return false;
  const int st = s.jt & 1;
  if (!mbar_wait(&bars[B_KFULL + st], (s.jt >> 1) & 1, a.status)) return false;
  tc_fence_after();
  if (lane == 0) {
    const uint32_t qa = smem_u32(smem + Lay::kQ + qslot * Lay::kQBytes);
    const uint32_t ka = smem_u32(smem + Lay::kK + st * Lay::kKVBytes);
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, 0, 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * Lay::kPanelBytes + (kk & 3) * 32;
      umma_f16_ss(tbase + st * kBN, smem_desc(qa + off, 16, 1024, 2),
                  smem_desc(ka + off, 16, 1024, 2), idesc, kk > 0);
    }
    umma_commit(&bars[B_SFULL + st]);
    umma_commit(&bars[B_KEMPTY + st]);
    if (s.j == s.it.n_tiles - 1) umma_commit(&bars[B_QEMPTY + qslot]);
  }
  __syncwarp();
  return true;
}

template <int D>
__device__ void mma_role(const PrefillArgs& a, uint8_t* smem, uint64_t* bars, uint32_t tbase) {
  using Lay = Layout<D>;
  const int lane = threadIdx.x & 31;
  TileIter pv, sx;
  iter_begin(a, pv);
  iter_begin(a, sx);
  // S for the first two tiles
  for (int i = 0; i < 2 && sx.valid; ++i) {
    if (!issue_s<D>(a, sx, smem, bars, tbase)) goto drain;
    iter_next(a, sx);
  }
  while (pv.valid) {
    {
      const uint32_t jt = pv.jt;
      const int st = jt & 1;
      if (!mbar_wait(&bars[B_PFULL], jt & 1, a.status)) goto drain;
      if (pv.j == 0 && pv.item_idx > 0 &&
          !mbar_wait(&bars[B_OFREE], (pv.item_idx - 1) & 1, a.status))
        goto drain;
      if (!mbar_wait(&bars[B_VFULL + st], (jt >> 1) & 1, a.status)) goto drain;
      uint8_t* vs = smem + Lay::kV + st * Lay::kKVBytes;
      // Rows past the sequence's last key may hold stale or poisoned data;
      // P is 0 there, but 0 * NaN is NaN inside the MMA: zero them.
      const int valid_rows = pv.it.k_len - pv.j * kBN;
      if (valid_rows < kBN) {
        const int r0 = valid_rows < 0 ? 0 : valid_rows;
        const int n16 = (kBN - r0) * 8;  // 16-byte chunks per panel
        for (int p = 0; p < (int)Lay::kPanels; ++p)
          for (int i = lane; i < n16; i += 32)
            *reinterpret_cast<uint4*>(vs + p * Lay::kPanelBytes + r0 * 128 + i * 16) =
                make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t pa = smem_u32(smem + Lay::kP);
        const uint32_t va = smem_u32(vs);
        constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, 0, 1);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t ad = smem_desc(pa + (kk >> 2) * Lay::kPanelBytes + (kk & 3) * 32, 16, 1024, 2);
          const uint64_t bd = smem_desc(va + kk * 16 * 128, Lay::kPanelBytes, 1024, 2);
          umma_f16_ss(tbase + 2 * kBN, ad, bd, idesc, (pv.j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_VEMPTY + st]);
        umma_commit(&bars[B_ODONE]);
      }
      __syncwarp();
    }
    if (sx.valid) {
      if (!issue_s<D>(a, sx, smem, bars, tbase)) goto drain;
      iter_next(a, sx);
    }
    iter_next(a, pv);
  }
drain:
  // Every MMA this thread issued has completed before the CTA tears down.
  if (lane == 0) umma_commit(&bars[B_DRAIN]);
  __syncwarp();
  mbar_wait(&bars[B_DRAIN], 0, a.status);
}

// ------------------------------------------------------------------ softmax

template <int D>
__device__ void softmax_role(const PrefillArgs& a, uint8_t* smem, uint64_t* bars, uint32_t tbase) {
  using Lay = Layout<D>;
  constexpr int kHalfCols = kBN / 2;  // S / P columns per thread
  constexpr int kHalfD = D / 2;       // O columns per thread
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;  // TMEM lane quarter, column half
  const int r = quarter * 32 + lane;                // query row == TMEM lane
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  uint8_t* sP = smem + Lay::kP;
  float* xbuf = reinterpret_cast<float*>(smem + Lay::kX);  // [parity][half][row]
  uint64_t* xbar = &bars[B_XCH + quarter];
  uint32_t xcnt = 0;  // exchanges so far (identical in both warps of a quarter)

  // The two threads of a row swap one value through shared memory; bounded
  // wait on the quarter's barrier; double-buffered by exchange parity.
  auto exchange = [&](float mine, float& theirs) -> bool {
    const int par = xcnt & 1;
    xbuf[(par * 2 + half) * kBM + r] = mine;
    __syncwarp();
    if (lane == 0) mbar_arrive(xbar);
    if (!mbar_wait(xbar, (uint32_t)par, a.status)) return false;
    theirs = xbuf[(par * 2 + (half ^ 1)) * kBM + r];
    ++xcnt;
    return true;
  };

  TileIter t;
  iter_begin(a, t);
  const float2 scale2 = make_float2(a.scale_log2, a.scale_log2);
  while (t.valid) {
    const Item it = t.it;
    const int tok = r / a.group, h = r - tok * a.group;
    const bool row_valid = tok < it.rows_tok;
    const int pos = it.cached + it.q0 + (row_valid ? tok : it.rows_tok - 1);
    float m = -INFINITY, l = 0.f;  // l: this thread's half of the row sum
    for (int j = 0; j < it.n_tiles; ++j) {
      const uint32_t jt = t.jt;
      const int st = jt & 1;
      if (!mbar_wait(&bars[B_SFULL + st], (jt >> 1) & 1, a.status)) return;
      tc_fence_after();
      float s[kHalfCols];
#pragma unroll
      for (int c = 0; c < kHalfCols / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_base + st * kBN + half * kHalfCols + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[i]);
      }
      const int lim = pos - j * kBN - half * kHalfCols;  // my columns <= lim are visible
      if (lim < kHalfCols - 1) {
#pragma unroll
        for (int i = 0; i < kHalfCols; ++i)
          if (i > lim) s[i] = -INFINITY;
      }
      float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int i = 4; i < kHalfCols; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
      float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      float other;
      if (!exchange(mx, other)) return;
      mx = fmaxf(mx, other);
      const float mxs = mx * a.scale_log2;
      // The reference max m only moves when the tile's max exceeds it by more
      // than 2^8 (or on the first tile): O and l then get rescaled by alpha.
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        m = mxs;  // key 0 is visible to every row: finite
      } else if (mxs > m + kRescaleThreshold) {
        alpha = fast_exp2(m - mxs);
        m = mxs;
        rescale = true;
      }
      // P = exp2(s * scale_log2 - m) as bf16 pairs, computed while the previous
      // tile's PV still runs on the tensor core.
      const float2 negm = make_float2(-m, -m);
      uint32_t pk[kHalfCols / 2];
      float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kHalfCols / 2; ++i) {
        const float2 x = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), scale2, negm);
        const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
        sum2 = __fadd2_rn(sum2, p);
        pk[i] = pack_bf16x2(p.x, p.y);
      }
      if (j > 0) {
        // PV of the previous tile has finished: O is stable and P is free.
        if (!mbar_wait(&bars[B_ODONE], (jt - 1) & 1, a.status)) return;
        tc_fence_after();
        if (rescale) {
          l *= alpha;
#pragma unroll
          for (int c = 0; c < kHalfD / 32; ++c) {
            uint32_t v[32];
            const uint32_t addr = tbase + lane_base + 2 * kBN + half * kHalfD + c * 32;
            tmem_ld32(addr, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 o = __fmul2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                          make_float2(alpha, alpha));
              v[i] = __float_as_uint(o.x);
              v[i + 1] = __float_as_uint(o.y);
            }
            tmem_st32(addr, v);
          }
          tmem_st_wait();
        }
      }
      l += sum2.x + sum2.y;
      // P into shared memory, 128-byte swizzled K-major (the PV MMA's A
      // operand): this thread's 64 keys are exactly 64-key panel `half`.
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(sP + half * Lay::kPanelBytes + r * 128 + ((c ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_PFULL]);
      iter_next(a, t);
    }
    // Epilogue: O / l -> bf16 -> out; each thread stores its half of the row.
    if (!mbar_wait(&bars[B_ODONE], (t.jt - 1) & 1, a.status)) return;
    tc_fence_after();
    float l_other;
    if (!exchange(l, l_other)) return;
    const float inv = 1.f / (l + l_other);
    uint16_t* orow = a.out + (int64_t)(it.q_row0 + tok) * a.out_stride +
                     (int64_t)(it.g * a.group + h) * D + half * kHalfD;
#pragma unroll
    for (int c = 0; c < kHalfD / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tbase + lane_base + 2 * kBN + half * kHalfD + c * 32, v);
      tmem_ld_wait();
      if (row_valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(v[q * 8 + 0]) * inv, __uint_as_float(v[q * 8 + 1]) * inv);
          u.y = pack_bf16x2(__uint_as_float(v[q * 8 + 2]) * inv, __uint_as_float(v[q * 8 + 3]) * inv);
          u.z = pack_bf16x2(__uint_as_float(v[q * 8 + 4]) * inv, __uint_as_float(v[q * 8 + 5]) * inv);
          u.w = pack_bf16x2(__uint_as_float(v[q * 8 + 6]) * inv, __uint_as_float(v[q * 8 + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + c * 32 + q * 8) = u;
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_OFREE]);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreadsPF, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillArgs a) {
  using Lay = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the 128-byte swizzle needs a 1 KiB aligned base
    if (threadIdx.x == 0) record_error(a.status, KVP_ERR_DEVICE_DATA);
    return;
  }
  uint8_t* smem = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Lay::kNumBars);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_QFULL + i], 1);
      mbar_init(&bars[B_QEMPTY + i], 1);
      mbar_init(&bars[B_KFULL + i], 1);
      mbar_init(&bars[B_KEMPTY + i], 1);
      mbar_init(&bars[B_VFULL + i], 1);
      mbar_init(&bars[B_VEMPTY + i], 1);
      mbar_init(&bars[B_SFULL + i], 1);
    }
    mbar_init(&bars[B_PFULL], kSoftmaxWarps);
    mbar_init(&bars[B_ODONE], 1);
    mbar_init(&bars[B_OFREE], kSoftmaxWarps);
    mbar_init(&bars[B_DRAIN], 1);
    for (int i = 0; i < 4; ++i) mbar_init(&bars[B_XCH + i], 2);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);  // S0 | S1 | O (D columns)
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == kProducerWarp)
    producer_role<D>(a, &tmQ, &tmK, &tmV, smem, bars);
  else if (warp == kMmaWarp)
    mma_role<D>(a, smem, bars, tbase);
  else
    softmax_role<D>(a, smem, bars, tbase);

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 3-D map over [rows, heads, D] bf16 (row stride in elements), 128-byte swizzle,
// box {64, box_heads, box_rows}.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int64_t row_stride,
              int box_heads, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)row_stride * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                     const PrefillArgs& a, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Layout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  prefill_kernel<D><<<grid, kThreadsPF, Layout<D>::kAlloc, stream>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int num_heads, int num_kv_heads, int head_dim, int block_size) {
  if (num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads) return false;
  const int G = num_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  if (head_dim != 64 && head_dim != 128) return false;
  if (block_size < 16 || block_size > 4096 || block_size % 16) return false;
  const int m = block_size / 16;
  return (m & (m - 1)) == 0;
}

int launch_prefill(const uint16_t* q, int64_t q_stride, int64_t total_q, const uint16_t* k,
                   const uint16_t* v, int64_t kv_stride, int64_t total_k,
                   const uint16_t* k_cache, const uint16_t* v_cache, int64_t num_blocks,
                   int block_size, const int32_t* block_tables, int max_blocks,
                   const int32_t* cu_q, const int32_t* cu_k, int max_seqlen_q, int max_seqlen_k,
                   int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                   float softmax_scale, uint16_t* out, int64_t out_stride, int num_sms,
                   int* status, cudaStream_t stream, const char** why) {
  (void)max_seqlen_k;
  if (!get_encoder()) {
    *why = "cuTensorMapEncodeTiled is unavailable";
    return KVP_ERR_CUDA;
  }
  const int G = num_heads / num_kv_heads;
  const int tok = kBM / G;
  const bool paged = block_tables != nullptr;
  const int sub_rows = paged ? (block_size < kBN ? block_size : kBN) : kBN;
  CUtensorMap mq, mk, mv;
  bool ok = make_map(&mq, q, total_q, num_heads, head_dim, q_stride, G, tok);
  if (paged) {
    const int64_t rows = num_blocks * (int64_t)block_size;
    const int64_t rs = (int64_t)num_kv_heads * head_dim;
    ok = ok && make_map(&mk, k_cache, rows, num_kv_heads, head_dim, rs, 1, sub_rows) &&
         make_map(&mv, v_cache, rows, num_kv_heads, head_dim, rs, 1, sub_rows);
  } else {
    ok = ok && make_map(&mk, k, total_k, num_kv_heads, head_dim, kv_stride, 1, kBN) &&
         make_map(&mv, v, total_k, num_kv_heads, head_dim, kv_stride, 1, kBN);
  }
  if (!ok) {
    *why = "tensor map encoding failed (alignment or extent)";
    return KVP_ERR_INVALID_ARG;
  }
  PrefillArgs a;
  a.cu_q = cu_q;
  a.cu_k = cu_k;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.paged = paged ? 1 : 0;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = G;
  a.tok_per_tile = tok;
  a.sub_rows = sub_rows;
  a.max_tiles = (max_seqlen_q + tok - 1) / tok;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.out = out;
  a.out_stride = out_stride;
  a.status = status;
  const long long items = (long long)a.max_tiles * num_seqs * num_kv_heads;
  if (items >= (1ll << 31)) {
    *why = "too many work items";
    return KVP_ERR_UNSUPPORTED;
  }
  const int grid = (int)(items < num_sms ? items : num_sms);
  cudaError_t e = head_dim == 128 ? launch_t<128>(mq, mk, mv, a, grid, stream)
                                  : launch_t<64>(mq, mk, mv, a, grid, stream);
  if (e != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return KVP_ERR_CUDA;
  }
  return KVP_OK;
}

}  // namespace kvp
