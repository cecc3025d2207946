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
// Work unit ("item"): one sequence b, one kv head g and two query tiles A and
// B of 128 rows each.  A tile row is (token, head): 128/G consecutive tokens
// x the G query heads that share kv head g, so one MMA serves the whole GQA
// group; tile B holds the 128/G tokens that follow tile A's.  Query row
// (token t, head h) sits at absolute position c_b + t and sees keys 0 .. that
// position.  An item walks kv tiles of 128 keys up to the last key its last
// row sees; each K/V tile in shared memory feeds both query tiles, which
// halves the K/V bytes moved per FLOP compared with one tile.
//
// Persistent CTAs (one per SM), 12 warps:
//   warp 8  picks the CTA's items (next position of the cost-sorted order
//           from a global counter, heaviest first) and passes each to the
//           other roles through a 2-slot ring in shared memory; and is the
//           TMA producer: the Q pair (one slot), K tiles (2 slots), V tiles
//           (2 slots).  In paged mode a kv tile is loaded as block-sized
//           sub-boxes addressed through the block table (gather folded into
//           the loads); sub-boxes past the sequence's last key are skipped.
//   warp 9  tensor-memory owner; one of its threads issues every MMA.  TMEM
//           columns: S_A | S_B | O_A | O_B (128 each).  Issue order per kv
//           tile j:  PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
//           so each softmax warpgroup computes on one tile while the tensor
//           core works on the other tile (ping-pong).  PV reads P from
//           tensor memory (the A operand of a TS-form MMA).
//   warp 10 V fix-up: zeroes V rows past the last key before PV reads them.
//   warps 0-3 / 4-7  softmax for tile A / B: thread r owns row r (TMEM lane
//           r).  Reads S with tcgen05.ld, masks only where a tile crosses the
//           diagonal, keeps a running max per row and rescales O only when
//           the max grows by more than 2^8 (exact: O and the row sum share the
//           stale reference), writes P as bf16 pairs over the first 64
//           columns of its S region, and at the end of an item normalises O
//           and stores bf16.  The warpgroup of an item's last tile releases
//           the K and Q slots once it sees the S that last read them; a V
//           slot is released by a commit of the MMA thread right after the
//           last PV that reads it (it would otherwise wait for the next S,
//           another batch of MMAs later).
// Synchronisation facts the design relies on: a tcgen05.commit arrives only
// when every earlier MMA of the issuing thread has completed, so the commit
// after S_X(j+1) also says PV_X(j) is done (O_X may be rescaled, and P_X's
// columns, which S_X(j+1) overwrites, have been read).
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "kvp_device.cuh"

namespace kvp {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per kv tile
// Three warpgroups: softmax A (warps 0-3), softmax B (4-7), and a control
// group (warp 8 TMA producer, warp 9 MMA issuer, warp 10 V fix-up, warp 11
// idle).  The launch gives every thread 168 registers (384 x 168 = 64512);
// the control group hands registers back with setmaxnreg and the softmax
// groups take them: 128 x (200 + 200 + 104) = 64512, the launch's total.
constexpr int kThreadsPF = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kVFixWarp = 10;
constexpr int kSoftmaxRegs = 200;
constexpr int kControlRegs = 104;
static_assert(128 * (2 * kSoftmaxRegs + kControlRegs) <= kThreadsPF * 168,
              "register split exceeds the launch's allotment");
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
  int group;         // G
  int tok_per_tile;  // 128 / G
  int sub_rows;      // rows per TMA box of a kv tile (paged: min(bs, 128))
  int max_pairs;     // ceil(max_seqlen_q / (2 * tok_per_tile))
  int dynamic;       // 1: items taken in cost order from a global counter; 0: round-robin
  int cu_in_smem;    // 1: cu_seqlens_q/k are copied into shared memory at kernel start
  unsigned long long* qslot;  // dynamic: (epoch << 32) | next position, one slot per launch
  unsigned int* qdone;        // dynamic: CTAs finished, for the slot's reset
  uint32_t epoch;             // dynamic: this launch's tag in the slot (>= 1)
  float scale_log2;
  uint16_t* out;
  int64_t out_stride;
  int* status;
  // attn_prefill_varlen_append: the grid is a programmatic dependent of the
  // kv_store launch of the step's new rows.  append 1 (paged): uncached keys
  // come from the new rows (maps tmKn / tmVn), and the first read of the cache
  // waits for the store grid (griddepcontrol.wait); append 2 (packed): the
  // keys are the new rows and nothing waits until the end.
  int append;
};

struct Item {
  int b, g, q0, q_len, cached, k_len, n_tiles;
  int first;           // kv tile processed first; tile (first + j) % n_tiles is step j
  int rows_a, rows_b;  // valid tokens in tile A / B (rows_b may be 0)
  int q_row0;          // packed row of tile A's first token
  int k_row0;          // packed row of the sequence's first key (packed mode)
};

constexpr int kCostBins = 256;
constexpr int kCuCap = 520;  // cu_seqlens entries cached in shared memory (num_seqs + 1)
constexpr int kMaxPairs = 4096;  // (pair rank, sequence) entries the cost-sorted order handles
constexpr int kQueueSlots = 64;  // counter slots: prefill calls that may be in flight at once
// Arrivals that free a slot of the item ring: the MMA thread, the 8 softmax
// warps and the V fix-up warp.
constexpr int kItemReaders = 10;

// Per-CTA schedule state in shared memory.
struct Sched {
  uint32_t bins[kCostBins];  // histogram, then next free position per cost
  int count;                 // item positions of the cost-sorted order
  int pad[3];
  Item ring[2];              // items passed from the producer to the other roles
  int cu[2][kCuCap];         // cu_seqlens_q, cu_seqlens_k
  uint8_t cost[kMaxPairs];   // cost bin of each (rank, sequence) pair, 0 = no work
  uint16_t order[kMaxPairs]; // pair index at each pair position of the cost-sorted order
};
constexpr uint32_t kSchedBytes = (sizeof(Sched) + 15) & ~15u;

template <int D>
struct Layout {
  static constexpr uint32_t kPanels = D / 64;
  static constexpr uint32_t kPanelBytes = 128 * 128;  // 128 rows x 128 bytes
  static constexpr uint32_t kQBytes = kBM * D * 2;    // one query tile
  static constexpr uint32_t kKVBytes = kBN * D * 2;
  static constexpr uint32_t kQ = 0;                  // tiles A, B
  static constexpr uint32_t kK = kQ + 2 * kQBytes;   // 2 slots
  static constexpr uint32_t kV = kK + 2 * kKVBytes;  // 2 slots
  static constexpr uint32_t kBar = kV + 2 * kKVBytes;
  static constexpr uint32_t kNumBars = 25;
  static constexpr uint32_t kSched = kBar + kNumBars * 8 + 16;
  static constexpr uint32_t kTotal = kSched + kSchedBytes;
  // The dynamic shared memory base is 1 KiB aligned on this architecture (the
  // kernel checks it and reports KVP_ERR_DEVICE_DATA otherwise).
  static constexpr uint32_t kAlloc = kTotal + 128;
};
static_assert(Layout<128>::kAlloc <= 227 * 1024, "shared memory per CTA");

// Barrier indices.
enum : int {
  B_QFULL = 0,
  B_QEMPTY = 1,
  B_KFULL = 2,   // [2]
  B_KEMPTY = 4,  // [2]
  B_VFULL = 6,   // [2]
  B_VEMPTY = 8,  // [2]
  B_SFULL = 10,  // [2]: tile A, tile B
  B_PFULL = 12,  // [2]
  B_PVDONE = 14, // [2]
  B_OFREE = 16,  // [2]
  B_VREADY = 18, // [2]: V tile loaded and its rows past the last key zeroed
  B_IFULL = 20,  // [2]: item ring slot written by the producer
  B_IEMPTY = 22, // [2]: item ring slot read by every other role
  B_DRAIN = 24,
};

// cu_seqlens as the roles read them: from shared memory when cached there.
struct Cu {
  const int* q;
  const int* k;
};

__device__ __forceinline__ Cu cu_view(const PrefillArgs& a, const Sched* sc) {
  if (a.cu_in_smem) return Cu{sc->cu[0], sc->cu[1]};
  return Cu{a.cu_q, a.cu_k};
}

__device__ __forceinline__ bool decode_item(const PrefillArgs& a, const Cu& cu, int L, Item& it) {
  const int per_r = a.num_seqs * a.num_kv_heads;
  const int r = L / per_r;
  const int rem = L - r * per_r;
  it.b = rem / a.num_kv_heads;
  it.g = rem - it.b * a.num_kv_heads;
  const int cq0 = cu.q[it.b], cq1 = cu.q[it.b + 1];
  const int ck0 = cu.k[it.b], ck1 = cu.k[it.b + 1];
  it.q_len = cq1 - cq0;
  it.k_len = ck1 - ck0;
  // Packed keys of the fused store are the new rows: no cached prefix.
  const bool bad = it.k_len < it.q_len || (a.append == 2 && it.k_len != it.q_len);
  if (it.q_len <= 0 || bad) {
    if (it.q_len > 0 && r == 0 && it.g == 0) record_error(a.status, KVP_ERR_DEVICE_DATA);
    return false;
  }
  const int span = 2 * a.tok_per_tile;
  const int npairs = (it.q_len + span - 1) / span;
  if (r >= npairs) return false;
  const int t = npairs - 1 - r;  // heaviest pairs (largest t) come first
  it.q0 = t * span;
  it.rows_a = min(a.tok_per_tile, it.q_len - it.q0);
  it.rows_b = max(0, min(a.tok_per_tile, it.q_len - it.q0 - a.tok_per_tile));
  it.cached = it.k_len - it.q_len;
  const int kv_end = it.cached + it.q0 + it.rows_a + it.rows_b;  // keys the last row sees
  it.n_tiles = (kv_end + kBN - 1) / kBN;
  it.q_row0 = cq0 + it.q0;
  it.k_row0 = ck0;
  // Fused store: tiles that read the cache (keys below `cached`) wait for the
  // launch's store, so the item takes its uncached tiles first (the online
  // softmax does not depend on the order of the kv tiles).
  const int cache_tiles = a.append == 1 ? (it.cached + kBN - 1) / kBN : 0;
  it.first = cache_tiles < it.n_tiles ? cache_tiles : 0;
  return true;
}

__device__ __forceinline__ int tile_at(const Item& it, int j) {
  const int t = it.first + j;
  return t < it.n_tiles ? t : t - it.n_tiles;
}

__device__ __forceinline__ int total_items(const PrefillArgs& a) {
  return a.max_pairs * a.num_seqs * a.num_kv_heads;
}

// Work order.  An item's cost (kv tiles x query tiles) depends only on its
// sequence and pair rank, not on the kv head, so the order is built over
// (rank, sequence) pairs: every CTA computes the same cost histogram and ranks
// the pairs by cost (ties in index order).  The CTAs then take items from that
// order, heaviest first, through one global counter per launch: a CTA takes
// the next item whenever it is ready (greedy list scheduling), which keeps
// the SMs' finish times together whatever the length mix.
__device__ __forceinline__ bool pair_cost(const PrefillArgs& a, const Cu& cu, int idx, int& v) {
  const int r = idx / a.num_seqs, b = idx - r * a.num_seqs;
  const int q_len = cu.q[b + 1] - cu.q[b];
  const int k_len = cu.k[b + 1] - cu.k[b];
  if (q_len <= 0 || k_len < q_len || (a.append == 2 && k_len != q_len)) {
    if (q_len > 0 && r == 0) record_error(a.status, KVP_ERR_DEVICE_DATA);
    return false;
  }
  const int span = 2 * a.tok_per_tile;
  const int npairs = (q_len + span - 1) / span;
  if (r >= npairs) return false;
  const int q0 = (npairs - 1 - r) * span;
  const int rows_a = min(a.tok_per_tile, q_len - q0);
  const int rows_b = max(0, min(a.tok_per_tile, q_len - q0 - a.tok_per_tile));
  const int n_tiles = (k_len - q_len + q0 + rows_a + rows_b + kBN - 1) / kBN;
  v = min(kCostBins - 1, n_tiles * (rows_b > 0 ? 2 : 1) + 1);
  return true;
}

// First part of the schedule, run by every thread of the CTA: cu_seqlens into
// shared memory, each pair's cost bin, and the per-bin item counts.
__device__ void schedule_costs(const PrefillArgs& a, Sched* sc) {
  const int tid = threadIdx.x, nt = blockDim.x;
  if (a.cu_in_smem)
    for (int i = tid; i <= a.num_seqs; i += nt) {
      sc->cu[0][i] = a.cu_q[i];
      sc->cu[1][i] = a.cu_k[i];
    }
  if (a.dynamic)
    for (int i = tid; i < kCostBins; i += nt) sc->bins[i] = 0;
  __syncthreads();
  if (!a.dynamic) return;
  const Cu cu = cu_view(a, sc);
  const int npi = a.max_pairs * a.num_seqs;
  for (int idx = tid; idx < npi; idx += nt) {
    int v;
    const bool ok = pair_cost(a, cu, idx, v);
    sc->cost[idx] = ok ? (uint8_t)v : (uint8_t)0;
    if (ok) atomicAdd(&sc->bins[v], (uint32_t)a.num_kv_heads);
  }
  __syncthreads();
}

// Second part, one warp (the producer's): the cost-sorted order.  Pairs are
// ranked by cost, descending, ties in index order; a pair's Hkv items take
// consecutive positions, and order[] maps a pair position back to the pair.
__device__ void build_order(const PrefillArgs& a, Sched* sc) {
  const int lane = threadIdx.x & 31;
  const uint32_t H = a.num_kv_heads;
  const int npi = a.max_pairs * a.num_seqs;
  // Exclusive prefix in descending cost: lane 0 owns the 8 highest bins.
  const int base = (31 - lane) * 8;
  uint32_t sum = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) sum += sc->bins[base + k];
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  uint32_t run = incl - sum;
  __syncwarp();
#pragma unroll
  for (int k = 7; k >= 0; --k) {
    const uint32_t c = sc->bins[base + k];
    sc->bins[base + k] = run;
    run += c;
  }
  __syncwarp();
  for (int b0 = 0; b0 < npi; b0 += 32) {
    const int idx = b0 + lane;
    const int v = idx < npi ? sc->cost[idx] : 0;
    const bool ok = v != 0;
    const unsigned same = __match_any_sync(0xffffffffu, ok ? v : -1);
    const unsigned lower = same & ((1u << lane) - 1u);
    uint32_t pos0 = 0;
    if (ok) pos0 = sc->bins[v] + (uint32_t)__popc(lower) * H;
    __syncwarp();
    if (ok && lower == 0) sc->bins[v] += (uint32_t)__popc(same) * H;
    if (ok) sc->order[pos0 / H] = (uint16_t)idx;
    __syncwarp();
  }
  if (lane == 0) sc->count = (int)total;
  __syncwarp();
}

// Next position of the cost-sorted order for this launch (one thread).  The
// slot holds (epoch << 32) | next position.  A slot still tagged with another
// epoch (zero after the previous launch on it reset it, or an older launch
// that stopped early) is moved to this launch's epoch at position 0: a CAS
// against the value last seen, repeated against the value it returns until
// the slot carries this epoch (whichever CTA's CAS lands first does it; an
// increment that lands after it is already a position of this launch).
// Positions are below kMaxPairs x num_kv_heads; 0x3fffffff means none (an
// error was recorded).
__device__ __forceinline__ int queue_fetch(const PrefillArgs& a) {
  unsigned long long v = atomicAdd(a.qslot, 1ull);
  if ((uint32_t)(v >> 32) == a.epoch) return (int)(v & 0xffffffffull);
  const unsigned long long fresh = (unsigned long long)a.epoch << 32;
  unsigned long long cur = v + 1ull;
  for (int tries = 0; (uint32_t)(cur >> 32) != a.epoch; ++tries) {
    if (tries > 4096) {
      record_error(a.status, KVP_ERR_DEVICE_TIMEOUT);
      return 0x3fffffff;
    }
    const unsigned long long prev = atomicCAS(a.qslot, cur, fresh);
    cur = prev == cur ? fresh : prev;
  }
  v = atomicAdd(a.qslot, 1ull);
  if ((uint32_t)(v >> 32) != a.epoch) {  // another launch on this slot: not allowed
    record_error(a.status, KVP_ERR_DEVICE_DATA);
    return 0x3fffffff;
  }
  return (int)(v & 0xffffffffull);
}

// Item k of this CTA, from the producer's ring; false at the end marker (or
// if the wait expired).  The copy is taken before the slot is freed: one
// arrive per reading warp after __syncwarp, or by the MMA thread itself.
__device__ __forceinline__ bool ring_item(const Sched* sc, uint64_t* bars, int k, Item& it,
                                          bool warp_wide, int* status) {
  const int rs = k & 1;
  if (!mbar_wait(&bars[B_IFULL + rs], (k >> 1) & 1, status)) return false;
  it = sc->ring[rs];
  if (warp_wide) __syncwarp();
  if (!warp_wide || (threadIdx.x & 31) == 0) mbar_arrive(&bars[B_IEMPTY + rs]);
  return it.b >= 0;
}

// Transpose of a 4 x 4 matrix of 16-byte chunks held by the 4 lanes of a
// quad: on entry lane j holds chunks 0..3 of its row in w[0..3]; on exit lane
// j holds chunk j of rows 0..3 of the quad.  Two butterfly stages; in each, a
// chunk moves to the partner lane when one bit of its chunk index differs
// from the same bit of the lane index.
__device__ __forceinline__ void quad_transpose16(uint32_t (&w)[4][4], int lane) {
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int k0 = 0; k0 < 4; ++k0) {
      if (k0 & m) continue;
      const int k1 = k0 | m;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t send = hi ? w[k0][i] : w[k1][i];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
        if (hi)
          w[k0][i] = recv;
        else
          w[k1][i] = recv;
      }
    }
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ producer

template <int D>
__device__ void producer_role(const PrefillArgs& a, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                              const CUtensorMap* tmV, const CUtensorMap* tmKn,
                              const CUtensorMap* tmVn, uint8_t* smem, uint64_t* bars, Sched* sc) {
  using Lay = Layout<D>;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    prefetch_tensormap(tmQ);
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
    if (a.append == 1) {
      prefetch_tensormap(tmKn);
      prefetch_tensormap(tmVn);
    }
  }
  if (a.dynamic) build_order(a, sc);
  const Cu cu = cu_view(a, sc);
  // The producer picks this CTA's items and hands each to the other roles
  // through the 2-slot item ring.  Dynamic mode: the next position of the
  // cost-sorted order from the launch's counter, so the heaviest items go
  // first and a CTA takes another one whenever it is ready; the next
  // position is fetched while the current item loads.  Otherwise round-robin
  // over all item indices.
  // The first item of CTA bx is position bx, without a fetch; the counter
  // hands out positions from gridDim.x on.
  int next_pos = blockIdx.x, rr = 0;
  int item_idx = 0;
  uint32_t jt = 0;
  bool stored = false;
  Item it;
  for (;; ++item_idx) {
    bool have = false;
    if (a.dynamic) {
      int pos = __shfl_sync(0xffffffffu, next_pos, 0);
      while (pos < sc->count) {
        const int H = a.num_kv_heads;
        have = decode_item(a, cu, (int)sc->order[pos / H] * H + pos % H, it);
        if (lane == 0) next_pos = (int)gridDim.x + queue_fetch(a);
        if (have) break;
        pos = __shfl_sync(0xffffffffu, next_pos, 0);
      }
    } else {
      for (int L = blockIdx.x + rr * (int)gridDim.x; L < total_items(a); L += gridDim.x) {
        ++rr;
        if (decode_item(a, cu, L, it)) {
          have = true;
          break;
        }
      }
    }
    const int rs = item_idx & 1;
    if (!mbar_wait(&bars[B_IEMPTY + rs], ((item_idx >> 1) & 1) ^ 1u, a.status)) return;
    if (lane == 0) {
      if (have)
        sc->ring[rs] = it;
      else
        sc->ring[rs].b = -1;  // end marker
      mbar_arrive(&bars[B_IFULL + rs]);
    }
    if (!have) break;
    // Q pair: both tiles in one slot (tile B past the sequence is harmless
    // data: its rows are never stored).
    if (!mbar_wait(&bars[B_QEMPTY], (item_idx & 1) ^ 1u, a.status)) return;
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars[B_QFULL], 2 * Lay::kQBytes);
      for (int x = 0; x < 2; ++x)
        for (int p = 0; p < (int)Lay::kPanels; ++p)
          tma_load_3d(smem + Lay::kQ + x * Lay::kQBytes + p * Lay::kPanelBytes, tmQ, p * 64,
                      it.g * a.group, it.q_row0 + x * a.tok_per_tile, &bars[B_QFULL]);
    }
    int win_base = -1, win_val = -1;  // 32 block-table entries per warp-wide window
    for (int j = 0; j < it.n_tiles; ++j, ++jt) {
      const int st = jt & 1;
      const uint32_t par = (jt >> 1) & 1;
      const int key0 = tile_at(it, j) * kBN;
      int nsub, rows_per_box;
      if (a.paged) {
        rows_per_box = a.sub_rows;
        nsub = (min(kBN, it.k_len - key0) + rows_per_box - 1) / rows_per_box;
      } else {
        rows_per_box = kBN;
        nsub = 1;
      }
      const uint32_t bytes = (uint32_t)(nsub * rows_per_box * D * 2);
      int rowi[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rowi[i] = 0;
      uint32_t from_new = 0;  // fused store: sub-boxes read from the new rows
      bool reads_cache = false;
      if (a.paged) {
        for (int i = 0; i < nsub; ++i) {
          const int key = key0 + i * rows_per_box;
          if (a.append == 1 && key >= it.cached) {
            // Entirely in the uncached suffix: the new rows hold these keys.
            from_new |= 1u << i;
            rowi[i] = it.q_row0 - it.q0 + (key - it.cached);
            continue;
          }
          reads_cache = true;
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
      if (reads_cache && a.append == 1 && !stored) {
        // A cache read: the store grid of the step's new rows must be complete.
        if (lane == 0) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        __syncwarp();
        stored = true;
      }
      for (int kv = 0; kv < 2; ++kv) {
        const int full = kv == 0 ? B_KFULL : B_VFULL;
        const int empty = kv == 0 ? B_KEMPTY : B_VEMPTY;
        if (!mbar_wait(&bars[empty + st], par ^ 1u, a.status)) return;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[full + st], bytes);
          uint8_t* dst = smem + (kv == 0 ? Lay::kK : Lay::kV) + st * Lay::kKVBytes;
          for (int i = 0; i < nsub; ++i) {
            const CUtensorMap* map = (from_new >> i & 1u) ? (kv == 0 ? tmKn : tmVn)
                                                          : (kv == 0 ? tmK : tmV);
            for (int p = 0; p < (int)Lay::kPanels; ++p)
              tma_load_3d(dst + p * Lay::kPanelBytes + i * rows_per_box * 128, map, p * 64, it.g,
                          rowi[i], &bars[full + st]);
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ MMA issuer

// S = Q K^T for one query tile: D/16 K-steps of M128 N128 K16.  `dq`, `dk`
// are the descriptors of the tiles' first panels; a K-step moves 32 bytes
// inside a 128-byte swizzled row, and every 4 K-steps the next 64-column panel.
template <int D>
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint64_t dq, uint64_t dk) {
  using Lay = Layout<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, 0, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * Lay::kPanelBytes + (kk & 3) * 32) >> 4;
    umma_f16_ss(d_tmem, dq + off, dk + off, idesc, kk > 0);
  }
}

// O (+)= P V with P read from tensor memory (bf16 pairs written by the
// softmax warps over the first 64 columns of the tile's S region).  V is the
// MN-major B operand: a K-step is 16 key rows (2 KiB).
template <int D>
__device__ __forceinline__ void mma_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t dv, bool acc) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, 0, 1);
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk)
    umma_f16_ts(d_tmem, p_tmem + kk * 8, dv + ((kk * 16 * 128) >> 4), idesc,
                (acc || kk > 0) ? 1u : 0u);
}

// The MMA issuer: one thread.  tcgen05.mma issue keeps pace with execution
// (the queue in front of the tensor core is short), so anything this thread
// does between two batches of MMAs is idle tensor time.  It therefore waits
// for all inputs of a tile step first and then issues PV and the next S of
// the tile back to back; shared-memory fix-ups of V are done by another warp.
template <int D>
__device__ void mma_role(const PrefillArgs& a, uint8_t* smem, uint64_t* bars, uint32_t tbase,
                         const Sched* sc) {
  using Lay = Layout<D>;
  // Descriptors of the first Q tile, K slot and V slot; the others are at
  // fixed byte offsets, added to the address field (bytes >> 4).
  const uint64_t dq0 = smem_desc(smem_u32(smem + Lay::kQ), 16, 1024, 2);
  const uint64_t dk0 = smem_desc(smem_u32(smem + Lay::kK), 16, 1024, 2);
  const uint64_t dv0 = smem_desc(smem_u32(smem + Lay::kV), Lay::kPanelBytes, 1024, 2);
  constexpr uint32_t kQStep = Lay::kQBytes >> 4, kSlotStep = Lay::kKVBytes >> 4;
  uint32_t np[2] = {0, 0};      // PVs issued per tile
  uint32_t nitems[2] = {0, 0};  // items per tile (A: all, B: those with rows)
  int item_idx = 0;
  uint32_t jt = 0;
  Item it;
  for (; ring_item(sc, bars, item_idx, it, false, a.status); ++item_idx) {
    const int ntile = it.rows_b > 0 ? 2 : 1;
    if (!mbar_wait(&bars[B_QFULL], item_idx & 1, a.status)) goto drain;
    if (!mbar_wait(&bars[B_KFULL + (jt & 1)], (jt >> 1) & 1, a.status)) goto drain;
    tc_fence_after();
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      if (x < ntile) {
        mma_qk<D>(tbase + x * kBN, dq0 + x * kQStep, dk0 + (jt & 1) * kSlotStep);
        umma_commit(&bars[B_SFULL + x]);
      }
    }
    for (int j = 0; j < it.n_tiles; ++j, ++jt) {
      const int st = jt & 1;
      const bool more = j + 1 < it.n_tiles;
      const uint32_t jn = jt + 1;
      if (!mbar_wait(&bars[B_VREADY + st], (jt >> 1) & 1, a.status)) goto drain;
      if (more && !mbar_wait(&bars[B_KFULL + (jn & 1)], (jn >> 1) & 1, a.status)) goto drain;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (x < ntile) {
          if (!mbar_wait(&bars[B_PFULL + x], np[x] & 1, a.status)) goto drain;
          if (j == 0 && nitems[x] > 0 &&
              !mbar_wait(&bars[B_OFREE + x], (nitems[x] - 1) & 1, a.status))
            goto drain;
          tc_fence_after();
          mma_pv<D>(tbase + (2 + x) * kBN, tbase + x * kBN, dv0 + st * kSlotStep, j > 0);
          if (x == ntile - 1) umma_commit(&bars[B_VEMPTY + st]);  // last reader of V(j)
          if (more) {
            mma_qk<D>(tbase + x * kBN, dq0 + x * kQStep, dk0 + (jn & 1) * kSlotStep);
            umma_commit(&bars[B_SFULL + x]);
          } else {
            // O_x is final: its epilogue need not wait for the other tile's last P.
            umma_commit(&bars[B_PVDONE + x]);
          }
          ++np[x];
        }
      }
    }
    ++nitems[0];
    if (ntile == 2) ++nitems[1];
  }
drain:
  // Every MMA this thread issued has completed before the CTA tears down.
  umma_commit(&bars[B_DRAIN]);
  mbar_wait(&bars[B_DRAIN], 0, a.status);
}

// V fix-up warp: waits for each V tile and, in paged mode, zeroes the rows
// past the sequence's last key before the MMA may read the tile.  Those rows
// hold whatever the physical block or an earlier tile left there; P is 0 for
// them, but 0 * NaN is NaN inside the MMA.  (Packed mode loads whole boxes:
// rows past the sequence belong to the next one or are filled with zeros.)
template <int D>
__device__ void vfix_role(const PrefillArgs& a, uint8_t* smem, uint64_t* bars, const Sched* sc) {
  using Lay = Layout<D>;
  const int lane = threadIdx.x & 31;
  uint32_t jt = 0;
  Item it;
  for (int k = 0; ring_item(sc, bars, k, it, true, a.status); ++k) {
    for (int j = 0; j < it.n_tiles; ++j, ++jt) {
      const int st = jt & 1;
      if (!mbar_wait(&bars[B_VFULL + st], (jt >> 1) & 1, a.status)) return;
      const int valid_rows = it.k_len - tile_at(it, j) * kBN;
      if (a.paged && valid_rows < kBN) {
        uint8_t* vs = smem + Lay::kV + st * Lay::kKVBytes;
        const int r0 = valid_rows < 0 ? 0 : valid_rows;
        const int n16 = (kBN - r0) * 8;
        for (int p = 0; p < (int)Lay::kPanels; ++p)
          for (int i = lane; i < n16; i += 32)
            *reinterpret_cast<uint4*>(vs + p * Lay::kPanelBytes + r0 * 128 + i * 16) =
                make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_VREADY + st]);
    }
  }
}

// ------------------------------------------------------------------ softmax

template <int D>
__device__ void softmax_role(const PrefillArgs& a, uint8_t* smem, uint64_t* bars, uint32_t tbase,
                             const Sched* sc) {
  using Lay = Layout<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int x = warp >> 2;               // query tile: 0 = A, 1 = B
  const int r = (warp & 3) * 32 + lane;  // row == TMEM lane
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t s_col = tbase + lane_base + x * kBN;
  const uint32_t o_col = tbase + lane_base + 2 * kBN + x * kBN;
  const float2 scale2 = make_float2(a.scale_log2, a.scale_log2);
  uint32_t ns = 0;    // S tiles consumed by this tile's warpgroup
  uint32_t nit = 0;   // items this warpgroup took part in
  uint32_t jt0 = 0;   // kv tiles of all earlier items (ring slot of tile j = (jt0 + j) & 1)
  // The warpgroup of an item's last query tile releases the K and Q slots: it
  // observes S of that tile complete, and that MMA was issued after every
  // earlier MMA that read those slots.  (V slots: MMA commits.)
  const bool releaser = (warp & 3) == 0 && lane == 0;
  Item it;
  for (int k = 0; ring_item(sc, bars, k, it, true, a.status); ++k, jt0 += it.n_tiles) {
    const bool has_b = it.rows_b > 0;
    const int rows = x == 0 ? it.rows_a : it.rows_b;
    if (x == 1 && !has_b) continue;
    const bool last = x == (has_b ? 1 : 0);
    const int tok = r / a.group, h = r - tok * a.group;
    const bool row_valid = tok < rows;
    const int tok0 = it.q0 + x * a.tok_per_tile;  // first token of this tile
    const int pos = it.cached + tok0 + (row_valid ? tok : rows - 1);
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < it.n_tiles; ++j) {
      if (!mbar_wait(&bars[B_SFULL + x], ns & 1, a.status)) return;
      ++ns;
      if (last && releaser) {  // S(j) done: K(j) free
        mbar_arrive(&bars[B_KEMPTY + ((jt0 + j) & 1)]);
        if (j + 1 == it.n_tiles) mbar_arrive(&bars[B_QEMPTY]);
      }
      tc_fence_after();
      // All four 32-column loads in flight, one wait.
      uint32_t sv[kBN / 32][32];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tmem_ld32(s_col + c * 32, sv[c]);
      tmem_ld_wait();
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(sv[c][i]);
      const int lim = pos - tile_at(it, j) * kBN;  // columns <= lim are visible
      if (lim < kBN - 1) {
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i > lim) s[i] = -INFINITY;
      }
      float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int i = 4; i < kBN; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
      const float mxs = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * a.scale_log2;
      // The reference max m only moves when the tile's max exceeds it by more
      // than 2^8 (or on the first tile): O and l then get rescaled by alpha.
      // The S commit of this tile implies the previous PV of this tile is
      // complete, so O may be read and written here.
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        // In kv order the first tile holds key 0, which every row sees; with
        // the uncached tiles first a row may see none of them (m = -inf).
        m = mxs;
      } else if (mxs > m + kRescaleThreshold) {
        alpha = fast_exp2(m - mxs);  // 0 while m is -inf (O and l are still 0)
        m = mxs;
        rescale = true;
      }
      const float mu = m == -INFINITY ? 0.f : m;
      const float2 negm = make_float2(-mu, -mu);
      uint32_t pk[kBN / 2];
      float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kBN / 2; ++i) {
        const float2 xx = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), scale2, negm);
        const float2 p = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
        sum2 = __fadd2_rn(sum2, p);
        pk[i] = pack_bf16x2(p.x, p.y);
      }
      // tcgen05.ld/st are warp-collective (.sync.aligned): the warp takes the
      // branch together when any of its rows rescales; the others have alpha 1.
      if (__any_sync(0xffffffffu, rescale)) {  // S commit => previous PV into O is complete
        l *= alpha;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(o_col + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 o = __fmul2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                        make_float2(alpha, alpha));
            v[i] = __float_as_uint(o.x);
            v[i + 1] = __float_as_uint(o.y);
          }
          tmem_st32(o_col + c * 32, v);
        }
        tmem_st_wait();
      }
      l += sum2.x + sum2.y;
      // P (bf16 pairs) into the first 64 columns of this tile's S region, where
      // the PV MMA reads it as its A operand.  The S columns are free: this
      // thread has read them, and the next S of this tile is issued only after
      // the PV that reads this P.
#pragma unroll
      for (int c = 0; c < kBN / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pk[c * 32 + i];
        tmem_st32(s_col + c * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_PFULL + x]);
    }
    // Epilogue: wait for this tile's last PV, O / l -> bf16 -> out.
    if (!mbar_wait(&bars[B_PVDONE + x], nit & 1, a.status)) return;
    ++nit;
    tc_fence_after();
    uint32_t ov[D / 32][32];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) tmem_ld32(o_col + c * 32, ov[c]);
    tmem_ld_wait();
    // O is in registers: the next item's PV may overwrite it.
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_OFREE + x]);
    // Stores: a lane's row is 2*D contiguous bytes, but lanes of one store
    // instruction would each hit a different cache line.  After a 4x4
    // transpose of 16-byte chunks within each quad of lanes, the quad writes
    // 64 contiguous bytes of one row per instruction.
    const float inv = 1.f / l;
    uint16_t* orow = row_valid ? a.out +
                                     (int64_t)(it.q_row0 + x * a.tok_per_tile + tok) * a.out_stride +
                                     (int64_t)(it.g * a.group + h) * D
                               : nullptr;
    const int qb = lane & ~3, jq = lane & 3;
    uint16_t* qrow[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      qrow[k] = reinterpret_cast<uint16_t*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(orow), qb + k));
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t w[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          {
            const float2 o = __fmul2_rn(make_float2(__uint_as_float(ov[c][8 * k + 2 * i]),
                                                    __uint_as_float(ov[c][8 * k + 2 * i + 1])),
                                        make_float2(inv, inv));
            w[k][i] = pack_bf16x2(o.x, o.y);
          }
      quad_transpose16(w, lane);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (qrow[k] != nullptr)
          *reinterpret_cast<uint4*>(qrow[k] + c * 32 + jq * 8) =
              make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreadsPF, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKn,
                   const __grid_constant__ CUtensorMap tmVn, const PrefillArgs a) {
  using Lay = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the 128-byte swizzle needs a 1 KiB aligned base
    if (threadIdx.x == 0) {
      record_error(a.status, KVP_ERR_DEVICE_DATA);
      if (a.append) asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    return;
  }
  // The next call's store grid (launched as a programmatic dependent, and
  // waiting for this grid before it touches memory) may be scheduled now.
  if (a.append && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint8_t* smem = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Lay::kNumBars);
  Sched* sc = reinterpret_cast<Sched*>(smem + Lay::kSched);
  const int warp = threadIdx.x >> 5;
  schedule_costs(a, sc);

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_QFULL], 1);
    mbar_init(&bars[B_QEMPTY], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_KFULL + i], 1);
      mbar_init(&bars[B_KEMPTY + i], 1);
      mbar_init(&bars[B_VFULL + i], 1);
      mbar_init(&bars[B_VEMPTY + i], 1);
      mbar_init(&bars[B_SFULL + i], 1);
      mbar_init(&bars[B_PFULL + i], 4);
      mbar_init(&bars[B_PVDONE + i], 1);
      mbar_init(&bars[B_OFREE + i], 4);
      mbar_init(&bars[B_VREADY + i], 1);
      mbar_init(&bars[B_IFULL + i], 1);
      mbar_init(&bars[B_IEMPTY + i], kItemReaders);
    }
    mbar_init(&bars[B_DRAIN], 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);  // S_A | S_B | O_A | O_B
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
    if (warp == kProducerWarp)
      producer_role<D>(a, &tmQ, &tmK, &tmV, &tmKn, &tmVn, smem, bars, sc);
    else if (warp == kMmaWarp && (threadIdx.x & 31) == 0)
      mma_role<D>(a, smem, bars, tbase, sc);
    else if (warp == kVFixWarp)
      vfix_role<D>(a, smem, bars, sc);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    softmax_role<D>(a, smem, bars, tbase, sc);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, 512);
  if (a.dynamic && threadIdx.x == 0) {
    // Every fetch of this CTA is done.  The last CTA to get here returns the
    // counter slot to zero, so the same launch parameters (a CUDA graph
    // replay) start from position 0 again.
    __threadfence();
    if (atomicAdd(a.qdone, 1u) == gridDim.x - 1) {
      atomicExch(a.qslot, 0ull);
      atomicExch(a.qdone, 0u);
    }
  }
  // A dependent of the store grid does not complete before it (so the stream
  // order after this call holds for the store as well).
  if (a.append && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Counter slots of the dynamic schedule: one per prefill launch in flight
// (launch n uses slot n % kQueueSlots with epoch n / kQueueSlots + 1).
__device__ unsigned long long g_queue_slot[kQueueSlots];
__device__ unsigned int g_queue_done[kQueueSlots];

// ------------------------------------------------------------------ host side

// Device addresses of the counter slots (looked up once per device) and the
// launch sequence number per device.
constexpr int kMaxQueueDevices = 64;
unsigned long long* g_qslot_ptr[kMaxQueueDevices];
unsigned int* g_qdone_ptr[kMaxQueueDevices];
std::atomic<unsigned long long> g_qseq[kMaxQueueDevices];
std::mutex g_queue_mutex;

struct QueueSlot {
  unsigned long long* next;  // dynamic schedule counter
  unsigned int* done;        // CTAs finished
  uint32_t epoch;
};

bool queue_slot(QueueSlot* q) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxQueueDevices) return false;
  {
    std::lock_guard<std::mutex> lock(g_queue_mutex);
    if (!g_qslot_ptr[dev]) {
      void* ps = nullptr;
      void* pd = nullptr;
      if (cudaGetSymbolAddress(&ps, g_queue_slot) != cudaSuccess ||
          cudaGetSymbolAddress(&pd, g_queue_done) != cudaSuccess)
        return false;
      g_qdone_ptr[dev] = static_cast<unsigned int*>(pd);
      g_qslot_ptr[dev] = static_cast<unsigned long long*>(ps);
    }
  }
  const unsigned long long seq = g_qseq[dev].fetch_add(1);
  q->next = g_qslot_ptr[dev] + seq % kQueueSlots;
  q->done = g_qdone_ptr[dev] + seq % kQueueSlots;
  q->epoch = (uint32_t)(seq / kQueueSlots) + 1u;
  return true;
}

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

// attn_prefill_varlen_append launches the prefill as a programmatic
// dependent of the store grid: its CTAs start on the SMs the (narrow) store
// grid leaves free.
template <int D>
cudaError_t launch_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                     const CUtensorMap& kn, const CUtensorMap& vn, const PrefillArgs& a, int grid,
                     cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Layout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  if (!a.append) {
    prefill_kernel<D><<<grid, kThreadsPF, Layout<D>::kAlloc, stream>>>(q, k, v, kn, vn, a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreadsPF);
  cfg.dynamicSmemBytes = Layout<D>::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_kernel<D>, q, k, v, kn, vn, a);
}

}  // namespace

void* tensor_map_encoder() { return get_encoder() ? reinterpret_cast<void*>(g_encode) : nullptr; }

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
                   int* status, cudaStream_t stream, const char** why,
                   const PrefillAppend* app) {
  (void)max_seqlen_k;
  if (!get_encoder()) {
    *why = "cuTensorMapEncodeTiled is unavailable";
    return KVP_ERR_CUDA;
  }
  const int G = num_heads / num_kv_heads;
  const int tok = kBM / G;
  const bool paged = block_tables != nullptr;
  const int sub_rows = paged ? (block_size < kBN ? block_size : kBN) : kBN;
  CUtensorMap mq, mk, mv, mkn, mvn;
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
  if (ok && paged && app)  // the fused store's new rows, read for uncached keys
    ok = make_map(&mkn, app->k, total_q, num_kv_heads, head_dim, app->stride, 1, sub_rows) &&
         make_map(&mvn, app->v, total_q, num_kv_heads, head_dim, app->stride, 1, sub_rows);
  if (!ok) {
    *why = "tensor map encoding failed (alignment or extent)";
    return KVP_ERR_INVALID_ARG;
  }
  if (!(paged && app)) {
    mkn = mk;
    mvn = mv;
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
  a.max_pairs = (max_seqlen_q + 2 * tok - 1) / (2 * tok);
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.out = out;
  a.out_stride = out_stride;
  a.status = status;
  const long long items = (long long)a.max_pairs * num_seqs * num_kv_heads;
  if (items >= (1ll << 31)) {
    *why = "too many work items";
    return KVP_ERR_UNSUPPORTED;
  }
  const int grid = (int)(items < num_sms ? items : num_sms);
  // With at most one item per CTA (small steps: items <= grid), CTA x takes
  // item x and nothing is scheduled: no cost sort, no counter, cu_seqlens read
  // where the item is decoded.
  const bool one_each = items <= grid;
  a.dynamic = !one_each && (long long)a.max_pairs * num_seqs <= kMaxPairs ? 1 : 0;
  a.qslot = nullptr;
  a.qdone = nullptr;
  a.epoch = 0;
  a.append = app ? (paged ? 1 : 2) : 0;
  if (a.dynamic) {
    QueueSlot qs;
    if (!queue_slot(&qs)) {
      *why = "counter slots of the dynamic schedule unavailable";
      return KVP_ERR_CUDA;
    }
    a.qslot = qs.next;
    a.qdone = qs.done;
    a.epoch = qs.epoch;
  }
  a.cu_in_smem = !one_each && num_seqs + 1 <= kCuCap ? 1 : 0;
  cudaError_t e = head_dim == 128 ? launch_t<128>(mq, mk, mv, mkn, mvn, a, grid, stream)
                                  : launch_t<64>(mq, mk, mv, mkn, mvn, a, grid, stream);
  if (e != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return KVP_ERR_CUDA;
  }
  return KVP_OK;
}

}  // namespace kvp
