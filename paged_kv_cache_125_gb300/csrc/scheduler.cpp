// Host-side block manager and scheduler of a nano-vLLM-style engine, with the
// C ABI of kvpaged_sched.h.  No GPU work: this turns requests into engine
// steps and builds each step's attention metadata.
//
// Sources ("nano-vLLM-1", Senjl's Digital Garden): BlockManager sections
// "1. Block" .. "5. 核心方法三：回收块（deallocate）" (FIFO free list, chained
// hash of full blocks, reference counts, prefix-cache hits confirmed by token
// ids); Scheduler sections "1. 队列与状态机" .. "4. 后处理：postprocess()"
// (prefill first, FCFS; decode with preemption from the tail of `running`);
// ModelRunner "4. prefill 输入打包" / "5. deocde 输入打包" (cu_seqlens,
// positions, slot_mapping, block_tables, context_lens).
#include <algorithm>
#include <cstring>
#include <deque>
#include <memory>
#include <new>
#include <unordered_map>
#include <vector>

#include "kvp_internal.h"
#include "kvpaged_sched.h"

namespace {

enum SeqStatus { kWaiting = 0, kRunning = 1, kFinished = 2 };

struct Seq {
  int64_t id;
  std::vector<int64_t> tokens;
  int num_prompt;
  int num_cached = 0;
  int max_tokens;
  int status = kWaiting;
  std::vector<int32_t> table;

  int len() const { return (int)tokens.size(); }
  int num_blocks(int bs) const { return (len() + bs - 1) / bs; }
  int last_block_tokens(int bs) const { return len() - (num_blocks(bs) - 1) * bs; }
};

struct Block {
  int ref = 0;
  bool has_hash = false;
  uint64_t hash = 0;
  std::vector<int64_t> tokens;
};

// FNV-1a, 64-bit, over the previous block's hash (8 bytes, little endian)
// when there is one, then every token id as 8 little-endian bytes.
uint64_t chain_hash(const int64_t* tok, int n, bool has_prev, uint64_t prev) {
  uint64_t h = 1469598103934665603ull;
  auto mix = [&h](uint64_t v) {
    for (int i = 0; i < 8; ++i) {
      h ^= (v >> (8 * i)) & 0xffu;
      h *= 1099511628211ull;
    }
  };
  if (has_prev) mix(prev);
  for (int i = 0; i < n; ++i) mix((uint64_t)tok[i]);
  return h;
}

class BlockManager {
 public:
  BlockManager(int num_blocks, int bs) : bs_(bs), blocks_(num_blocks), used_(num_blocks, 0) {
    for (int i = 0; i < num_blocks; ++i) free_.push_back(i);
  }

  int num_free() const { return (int)free_.size(); }

  bool can_allocate(const Seq& s) const { return num_free() >= s.num_blocks(bs_); }

  void allocate(Seq& s) {
    bool has_h = false;
    uint64_t h = 0;
    bool miss = false;
    const int nb = s.num_blocks(bs_);
    for (int i = 0; i < nb; ++i) {
      const int64_t* tok = s.tokens.data() + (int64_t)i * bs_;
      const int n = std::min(bs_, s.len() - i * bs_);
      if (n == bs_) {
        h = chain_hash(tok, n, has_h, h);
        has_h = true;
      } else {
        has_h = false;
      }
      int id = -1;
      if (has_h) {
        auto it = map_.find(h);
        if (it != map_.end()) id = it->second;
      }
      if (id == -1 || !same_tokens(blocks_[id], tok, n)) miss = true;
      int got;
      if (miss) {
        got = take(free_.front());
      } else {
        s.num_cached += bs_;
        if (used_[id]) {
          blocks_[id].ref += 1;
          got = id;
        } else {
          got = take(id);
        }
      }
      if (has_h) {
        Block& b = blocks_[got];
        b.has_hash = true;
        b.hash = h;
        b.tokens.assign(tok, tok + n);
        map_[h] = got;
      }
      s.table.push_back(got);
    }
  }

  void deallocate(Seq& s) {
    for (auto it = s.table.rbegin(); it != s.table.rend(); ++it) {
      Block& b = blocks_[*it];
      b.ref -= 1;
      if (b.ref == 0) {
        used_[*it] = 0;
        free_.push_back(*it);
      }
    }
    s.num_cached = 0;
    s.table.clear();
  }

  bool can_append(const Seq& s) const { return num_free() >= (s.len() % bs_ == 1 ? 1 : 0); }

  void may_append(Seq& s) {
    const int r = s.len() % bs_;
    if (r == 1) {
      s.table.push_back(take(free_.front()));
    } else if (r == 0) {
      const int nb = s.num_blocks(bs_);
      const int64_t* tok = s.tokens.data() + (int64_t)(nb - 1) * bs_;
      bool has_prev = false;
      uint64_t prev = 0;
      if (s.table.size() > 1) {
        const Block& pb = blocks_[s.table[s.table.size() - 2]];
        has_prev = pb.has_hash;
        prev = pb.hash;
      }
      const uint64_t h = chain_hash(tok, bs_, has_prev, prev);
      Block& last = blocks_[s.table.back()];
      last.has_hash = true;
      last.hash = h;
      last.tokens.assign(tok, tok + bs_);
      map_[h] = s.table.back();
    }
  }

 private:
  bool same_tokens(const Block& b, const int64_t* tok, int n) const {
    return (int)b.tokens.size() == n && std::equal(b.tokens.begin(), b.tokens.end(), tok);
  }

  // Takes a free block (ref 1, hash cleared), wherever it is in the free list.
  int take(int id) {
    Block& b = blocks_[id];
    b.ref = 1;
    b.has_hash = false;
    b.hash = 0;
    b.tokens.clear();
    free_.erase(std::find(free_.begin(), free_.end(), id));
    used_[id] = 1;
    return id;
  }

  int bs_;
  std::vector<Block> blocks_;
  std::vector<char> used_;
  std::deque<int> free_;
  std::unordered_map<uint64_t, int> map_;
};

}  // namespace

struct kvp_scheduler {
  int bs, max_seqs, max_tokens_per_step;
  BlockManager bm;
  std::unordered_map<int64_t, std::unique_ptr<Seq>> seqs;
  std::deque<Seq*> waiting, running;
  std::vector<Seq*> step;  // sequences of the last scheduled step
  bool step_prefill = false;
  int64_t preemptions = 0;

  kvp_scheduler(int nb, int bs_, int ms, int mt)
      : bs(bs_), max_seqs(ms), max_tokens_per_step(mt), bm(nb, bs_) {}

  void preempt(Seq* s) {
    s->status = kWaiting;
    bm.deallocate(*s);
    waiting.push_front(s);
    ++preemptions;
  }
};

using kvp::set_last_error;

extern "C" {

kvp_scheduler* kvp_sched_create(int num_blocks, int block_size, int max_num_seqs,
                                int max_num_batched_tokens) {
  if (num_blocks <= 0 || block_size <= 0 || max_num_seqs <= 0 || max_num_batched_tokens <= 0) {
    set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_create: non-positive argument");
    return nullptr;
  }
  return new (std::nothrow) kvp_scheduler(num_blocks, block_size, max_num_seqs,
                                          max_num_batched_tokens);
}

void kvp_sched_destroy(kvp_scheduler* s) { delete s; }

int kvp_sched_add(kvp_scheduler* s, int64_t seq_id, const int64_t* token_ids, int num_tokens,
                  int max_tokens) {
  if (!s || !token_ids || num_tokens <= 0 || max_tokens <= 0)
    return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_add: bad argument");
  if (s->seqs.count(seq_id))
    return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_add: duplicate seq_id");
  auto q = std::make_unique<Seq>();
  q->id = seq_id;
  q->tokens.assign(token_ids, token_ids + num_tokens);
  q->num_prompt = num_tokens;
  q->max_tokens = max_tokens;
  s->waiting.push_back(q.get());
  s->seqs.emplace(seq_id, std::move(q));
  return KVP_OK;
}

int kvp_sched_is_finished(const kvp_scheduler* s) {
  return s && s->waiting.empty() && s->running.empty() ? 1 : 0;
}

int kvp_sched_schedule(kvp_scheduler* s, int64_t* seq_ids, int* is_prefill) {
  if (!s || !seq_ids || !is_prefill) return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_schedule: null");
  if (s->waiting.empty() && s->running.empty())
    return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_schedule: nothing queued");
  s->step.clear();
  int num = 0;
  int64_t batched = 0;
  // prefill: FCFS from the head of waiting
  while (!s->waiting.empty() && num < s->max_seqs) {
    Seq* q = s->waiting.front();
    if (batched + q->len() > s->max_tokens_per_step || !s->bm.can_allocate(*q)) break;
    ++num;
    s->bm.allocate(*q);
    batched += q->len() - q->num_cached;
    q->status = kRunning;
    s->waiting.pop_front();
    s->running.push_back(q);
    s->step.push_back(q);
  }
  if (!s->step.empty()) {
    s->step_prefill = true;
  } else {
    // decode: from the head of running, preempting from its tail
    while (!s->running.empty() && num < s->max_seqs) {
      Seq* q = s->running.front();
      s->running.pop_front();
      bool self_preempted = false;
      while (!s->bm.can_append(*q)) {
        if (!s->running.empty()) {
          Seq* t = s->running.back();
          s->running.pop_back();
          s->preempt(t);
        } else {
          s->preempt(q);
          self_preempted = true;
          break;
        }
      }
      if (!self_preempted) {
        ++num;
        s->bm.may_append(*q);
        s->step.push_back(q);
      }
    }
    if (s->step.empty())
      return set_last_error(KVP_ERR_UNSUPPORTED,
                            "kvp_sched_schedule: the pool cannot hold a single sequence");
    for (auto it = s->step.rbegin(); it != s->step.rend(); ++it) s->running.push_front(*it);
    s->step_prefill = false;
  }
  for (size_t i = 0; i < s->step.size(); ++i) seq_ids[i] = s->step[i]->id;
  *is_prefill = s->step_prefill ? 1 : 0;
  return (int)s->step.size();
}

int kvp_sched_step_sizes(const kvp_scheduler* s, int64_t* num_new_tokens, int* max_blocks) {
  if (!s || !num_new_tokens || !max_blocks)
    return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_step_sizes: null");
  int64_t t = 0;
  int mb = 0;
  for (const Seq* q : s->step) {
    t += s->step_prefill ? q->len() - q->num_cached : 1;
    mb = std::max(mb, (int)q->table.size());
  }
  *num_new_tokens = t;
  *max_blocks = mb;
  return KVP_OK;
}

int kvp_sched_prepare(const kvp_scheduler* s, int32_t* cu_q, int32_t* cu_k, int64_t* positions,
                      int32_t* slots, int32_t* ctx, int32_t* tables, int stride, int* max_q,
                      int* max_k, int* has_prefix) {
  if (!s) return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_prepare: null scheduler");
  const int bs = s->bs;
  int mb = 0;
  for (const Seq* q : s->step) mb = std::max(mb, (int)q->table.size());
  if (stride < mb) return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_prepare: stride < max_blocks");
  auto fill_tables = [&]() {
    for (size_t i = 0; i < s->step.size(); ++i) {
      const Seq* q = s->step[i];
      int32_t* row = tables + (int64_t)i * stride;
      for (int j = 0; j < stride; ++j) row[j] = j < (int)q->table.size() ? q->table[j] : -1;
    }
  };
  if (s->step_prefill) {
    if (!cu_q || !cu_k || !positions || !slots || !max_q || !max_k || !has_prefix)
      return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_prepare: null prefill buffer");
    int64_t t = 0;
    int mq = 0, mk = 0;
    bool prefix = false;
    cu_q[0] = cu_k[0] = 0;
    for (size_t i = 0; i < s->step.size(); ++i) {
      const Seq* q = s->step[i];
      const int L = q->len(), c = q->num_cached;
      cu_q[i + 1] = cu_q[i] + (L - c);
      cu_k[i + 1] = cu_k[i] + L;
      mq = std::max(mq, L - c);
      mk = std::max(mk, L);
      prefix = prefix || c > 0;
      for (int p = c; p < L; ++p) {
        positions[t] = p;
        slots[t] = q->table[p / bs] * bs + p % bs;
        ++t;
      }
    }
    *max_q = mq;
    *max_k = mk;
    *has_prefix = prefix ? 1 : 0;
    if (prefix) {
      if (!tables) return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_prepare: null block_tables");
      fill_tables();
    }
  } else {
    if (!positions || !slots || !ctx || !tables)
      return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_prepare: null decode buffer");
    for (size_t i = 0; i < s->step.size(); ++i) {
      const Seq* q = s->step[i];
      positions[i] = q->len() - 1;
      ctx[i] = q->len();
      slots[i] = q->table.back() * bs + q->last_block_tokens(bs) - 1;
    }
    fill_tables();
  }
  return KVP_OK;
}

int kvp_sched_postprocess(kvp_scheduler* s, const int64_t* token_ids, int n) {
  if (!s || (n > 0 && !token_ids) || n != (int)s->step.size())
    return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_postprocess: token count != scheduled");
  for (int i = 0; i < n; ++i) {
    Seq* q = s->step[i];
    q->tokens.push_back(token_ids[i]);
    if (q->len() - q->num_prompt == q->max_tokens) {
      q->status = kFinished;
      s->bm.deallocate(*q);
      s->running.erase(std::find(s->running.begin(), s->running.end(), q));
    }
  }
  s->step.clear();
  return KVP_OK;
}

int64_t kvp_sched_num_preemptions(const kvp_scheduler* s) { return s ? s->preemptions : 0; }

int kvp_sched_num_free_blocks(const kvp_scheduler* s) { return s ? s->bm.num_free() : 0; }

int kvp_sched_seq_state(const kvp_scheduler* s, int64_t seq_id, int* num_tokens,
                        int* num_cached_tokens, int* status, int32_t* table, int cap,
                        int* num_table_entries) {
  if (!s) return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_seq_state: null");
  auto it = s->seqs.find(seq_id);
  if (it == s->seqs.end()) return set_last_error(KVP_ERR_INVALID_ARG, "kvp_sched_seq_state: unknown id");
  const Seq& q = *it->second;
  if (num_tokens) *num_tokens = q.len();
  if (num_cached_tokens) *num_cached_tokens = q.num_cached;
  if (status) *status = q.status;
  if (num_table_entries) *num_table_entries = (int)q.table.size();
  if (table)
    for (int j = 0; j < cap && j < (int)q.table.size(); ++j) table[j] = q.table[j];
  return KVP_OK;
}

}  // extern "C"
