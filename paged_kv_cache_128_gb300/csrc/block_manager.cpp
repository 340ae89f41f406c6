// Host metadata plane: the KV block manager behind the kvbm_* C ABI.
//
// Follows "MiniPaged-Qwen: Paged KV Cache 与 KV Block Manager" §8
// (SequenceState, KVBlockManager), §9 (append_token), §5.3 (release),
// §15 (invariants); "从零实现一个 mini vLLM: Block Manager" (prefill
// allocation, decode slot append, release once, can_allocate /
// can_append_slots, owner table); and the LLM-algo ch.22 "vLLM
// PagedAttention" exercise (atomic prefill, decode rollback, release
// validation, allocation report, capacity ledger).
//
// Free-list policy: take from the front, release to the back in table
// order (no sort), so a seeded initial order and churn carry through.
//
// Prefix sharing and copy-on-write ("paged-attention-impl-detail",
// section Copy-on-Write共享): a forked sequence shares its parent's blocks,
// each block carries a reference count, and a sequence about to write into
// a block that others also hold first copies it to a fresh block (the
// count of the old block drops by one, the new block's count is 1).  A
// released block returns to the free list only when its count reaches 0.
// The copies are queued for the device (kvbm_take_copies).
//
// Design: the free list is a ring buffer of int32; ref_count[b] == 0 iff b
// is free; each sequence keeps its table in a std::vector.  Every mutating
// call validates fully before it changes anything, so a failed call leaves
// the state exactly as it was.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <iterator>
#include <map>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pagedkv.h"

namespace {

struct Sequence {
  int64_t length = 0;            // tokens written == next append position
  std::vector<int32_t> table;    // logical block -> physical block
};

// FIFO of free block ids over a fixed ring of num_blocks entries.
class FreeList {
 public:
  explicit FreeList(int64_t cap) : ring_(static_cast<size_t>(cap)) {}
  int64_t size() const { return size_; }
  int32_t at(int64_t i) const { return ring_[static_cast<size_t>((head_ + i) % cap())]; }
  int32_t pop_front() {
    int32_t b = ring_[static_cast<size_t>(head_)];
    head_ = (head_ + 1) % cap();
    --size_;
    return b;
  }
  void push_back(int32_t b) {
    ring_[static_cast<size_t>((head_ + size_) % cap())] = b;
    ++size_;
  }

 private:
  int64_t cap() const { return static_cast<int64_t>(ring_.size()); }
  std::vector<int32_t> ring_;
  int64_t head_ = 0;
  int64_t size_ = 0;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Set of sequence ids for one call's duplicate checks: open addressing over
// a reused table whose slots are valid only for the current generation, so
// clearing it is one increment and inserting allocates nothing.
class IdSet {
 public:
  // Empty the set, with room for n ids.
  void reset(int64_t n) {
    size_t cap = 16;
    while (cap < 2 * static_cast<size_t>(n) + 1) cap <<= 1;
    if (cap > keys_.size()) {
      keys_.assign(cap, 0);
      gen_.assign(cap, 0);
      cur_ = 0;
    }
    if (++cur_ == 0) {  // generation counter wrapped: every slot is stale again
      std::fill(gen_.begin(), gen_.end(), 0u);
      cur_ = 1;
    }
  }
  // false when id was already in the set
  bool insert(int64_t id) {
    size_t i = find(id);
    if (gen_[i] == cur_) return false;
    gen_[i] = cur_;
    keys_[i] = id;
    return true;
  }
  bool contains(int64_t id) const { return gen_[find(id)] == cur_; }

 private:
  size_t find(int64_t id) const {  // the slot holding id, or the empty slot where it would go
    const size_t mask = keys_.size() - 1;
    size_t i = static_cast<size_t>(static_cast<uint64_t>(id) * 0x9E3779B97F4A7C15ull >> 20) & mask;
    while (gen_[i] == cur_ && keys_[i] != id) i = (i + 1) & mask;
    return i;
  }
  std::vector<int64_t> keys_;
  std::vector<uint32_t> gen_;
  uint32_t cur_ = 0;
};

// Released sequence ids, remembered so that a second release answers
// KV_ERR_DOUBLE_FREE, kept as disjoint inclusive ranges [first, last].  A
// serving loop that numbers its requests in order releases runs of
// consecutive ids, which merge into a few ranges: memory follows the gaps
// between released ids, not their count.  Ids are >= 0.
class IdRanges {
 public:
  size_t count(int64_t id) const {
    auto it = r_.upper_bound(id);  // first range starting after id
    if (it == r_.begin()) return 0;
    --it;
    return id <= it->second ? 1 : 0;
  }
  void insert(int64_t id) {
    if (count(id)) return;
    int64_t last = id;
    if (id < INT64_MAX) {  // absorb a range starting right after id
      auto nx = r_.find(id + 1);
      if (nx != r_.end()) {
        last = nx->second;
        r_.erase(nx);
      }
    }
    auto it = r_.lower_bound(id);
    if (it != r_.begin()) {  // extend a range ending right before id
      auto pv = std::prev(it);
      if (pv->second == id - 1) {
        pv->second = last;
        return;
      }
    }
    r_.emplace(id, last);
  }
  void erase(int64_t id) {
    auto it = r_.upper_bound(id);
    if (it == r_.begin()) return;
    --it;
    if (id > it->second) return;
    const int64_t first = it->first, last = it->second;
    r_.erase(it);
    if (first < id) r_.emplace(first, id - 1);
    if (id < last) r_.emplace(id + 1, last);
  }
  size_t ranges() const { return r_.size(); }

 private:
  std::map<int64_t, int64_t> r_;  // first -> last
};

}  // namespace

struct kvbm_s {
  int64_t num_blocks;
  int32_t block_size;
  FreeList free_list;
  std::vector<int32_t> ref_count;  // table entries referring to each block; 0 = free
  std::unordered_map<int64_t, Sequence> seqs;
  IdRanges released;
  std::vector<int32_t> copy_src, copy_dst;  // copy-on-write copies not yet taken
  IdSet step_ids;                      // kvbm_prepare_step's duplicate checks
  std::vector<const Sequence*> export_rows;  // kvbm_export_update's rows, validated before any write
  std::vector<uint32_t> block_mark;    // kvbm_free_sequence's duplicate-block check, by generation
  uint32_t block_gen = 0;

  kvbm_s(int64_t nb, int32_t bs)
      : num_blocks(nb), block_size(bs), free_list(nb), ref_count(nb, 0), block_mark(nb, 0) {}

  // A fresh generation for block_mark (all marks stale).
  uint32_t next_block_gen() {
    if (++block_gen == 0) {
      std::fill(block_mark.begin(), block_mark.end(), 0u);
      block_gen = 1;
    }
    return block_gen;
  }

  bool is_free(int32_t b) const { return ref_count[static_cast<size_t>(b)] == 0; }
  int32_t take_front() {
    int32_t b = free_list.pop_front();
    ref_count[static_cast<size_t>(b)] = 1;
    return b;
  }
  void give_back(int32_t b) {  // b's count is 0
    free_list.push_back(b);
  }
  // Drop one reference; the block is free again when none is left.
  void unref(int32_t b) {
    if (--ref_count[static_cast<size_t>(b)] == 0) give_back(b);
  }
  // The next write of s lands in its last block while another table also
  // holds that block: it must be copied first.
  bool needs_copy(const Sequence& s) const {
    return s.length % block_size != 0 && !s.table.empty() && ref_count[static_cast<size_t>(s.table.back())] > 1;
  }
  // The slots of positions 0 .. n - 1 of s, in order, to f: block by block,
  // table[k] * bs + off (slot_of without a division per token).
  template <typename F>
  void for_each_slot(const Sequence& s, int64_t n, F&& f) const {
    for (size_t k = 0; n > 0; ++k) {
      const int32_t base = s.table[k] * block_size;
      const int64_t m = n < block_size ? n : block_size;
      for (int64_t off = 0; off < m; ++off) f(base + static_cast<int32_t>(off));
      n -= m;
    }
  }
  // MiniPaged-Qwen §3: slot = table[pos / bs] * bs + pos % bs.
  int32_t slot_of(const Sequence& s, int64_t pos) const {
    return static_cast<int32_t>(static_cast<int64_t>(s.table[static_cast<size_t>(pos / block_size)]) *
                                    block_size +
                                pos % block_size);
  }
  // Blocks a sequence must gain to hold `extra` more tokens: new logical
  // blocks, plus one when its first write needs a copy of a shared block.
  int64_t blocks_needed(const Sequence& s, int64_t extra) const {
    return ceil_div(s.length + extra, block_size) - static_cast<int64_t>(s.table.size()) +
           (extra > 0 && needs_copy(s) ? 1 : 0);
  }
  // MiniPaged-Qwen §9 append_token, with copy-on-write of a shared last
  // block; the caller has checked a block is free.
  int32_t append_one(Sequence& s) {
    if (s.length / block_size == static_cast<int64_t>(s.table.size())) {
      s.table.push_back(take_front());
    } else if (needs_copy(s)) {
      const int32_t old = s.table.back();
      const int32_t fresh = take_front();
      --ref_count[static_cast<size_t>(old)];  // others still hold it: count stays >= 1
      s.table.back() = fresh;
      copy_src.push_back(old);
      copy_dst.push_back(fresh);
    }
    int32_t slot = slot_of(s, s.length);
    s.length += 1;
    return slot;
  }
  Sequence* find(int64_t id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
};

namespace {

template <typename F>
int guarded(F&& f) {
  try {
    return f();
  } catch (const std::bad_alloc&) {
    return KV_ERR_OOM;
  } catch (...) {
    return KV_ERR_INVARIANT;
  }
}

}  // namespace

extern "C" {

const char* kv_status_string(int status) {
  switch (status) {
    case KV_OK: return "ok";
    case KV_ERR_INVALID_ARG: return "invalid argument";
    case KV_ERR_OOM: return "out of KV blocks (OOM)";
    case KV_ERR_UNKNOWN_SEQ: return "unknown sequence id";
    case KV_ERR_DUPLICATE_SEQ: return "sequence already prefilled";
    case KV_ERR_DOUBLE_FREE: return "sequence already released (double free)";
    case KV_ERR_INVARIANT: return "block manager invariant violated";
    case KV_ERR_CUDA: return "CUDA error";
    case KV_ERR_DEVICE_BOUNDS: return "device access outside the KV pool (skipped)";
    case KV_ERR_WORKSPACE: return "workspace too small";
    case KV_ERR_DEVICE_TIMEOUT: return "bounded device wait timed out";
    case KV_ERR_DEVICE_STEP: return "new-token row does not land on its sequence's newest slot";
    default: return "unknown status";
  }
}

int kvbm_create(int64_t num_blocks, int32_t block_size, const int32_t* initial_free_order,
                kvbm_t* out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return KV_ERR_INVALID_ARG;
  if (num_blocks > INT32_MAX / block_size) return KV_ERR_INVALID_ARG;  // slots are int32
  return guarded([&] {
    auto* h = new kvbm_s(num_blocks, block_size);
    if (initial_free_order) {
      std::vector<uint8_t> seen(static_cast<size_t>(num_blocks), 0);
      for (int64_t i = 0; i < num_blocks; ++i) {
        int32_t b = initial_free_order[i];
        if (b < 0 || b >= num_blocks || seen[static_cast<size_t>(b)]) {
          delete h;
          return static_cast<int>(KV_ERR_INVALID_ARG);
        }
        seen[static_cast<size_t>(b)] = 1;
        h->give_back(b);
      }
    } else {
      for (int64_t i = 0; i < num_blocks; ++i) h->give_back(static_cast<int32_t>(i));
    }
    *out = h;
    return static_cast<int>(KV_OK);
  });
}

int kvbm_destroy(kvbm_t h) {
  delete h;
  return KV_OK;
}

int kvbm_can_allocate(kvbm_t h, int64_t num_tokens, int* ok) {
  if (!h || !ok || num_tokens <= 0) return KV_ERR_INVALID_ARG;
  *ok = ceil_div(num_tokens, h->block_size) <= h->free_list.size() ? 1 : 0;
  return KV_OK;
}

int kvbm_allocate_for_prefill(kvbm_t h, int64_t seq_id, int64_t num_tokens, int32_t* slots_out) {
  if (!h || seq_id < 0 || num_tokens <= 0) return KV_ERR_INVALID_ARG;
  if (h->seqs.count(seq_id)) return KV_ERR_DUPLICATE_SEQ;
  int64_t need = ceil_div(num_tokens, h->block_size);
  if (need > h->free_list.size()) return KV_ERR_OOM;  // nothing taken yet: atomic
  return guarded([&] {
    Sequence s;
    s.table.reserve(static_cast<size_t>(need));
    for (int64_t i = 0; i < need; ++i) s.table.push_back(h->take_front());
    s.length = num_tokens;
    if (slots_out) {
      int32_t* out = slots_out;
      h->for_each_slot(s, num_tokens, [&](int32_t slot) { *out++ = slot; });
    }
    h->seqs.emplace(seq_id, std::move(s));
    h->released.erase(seq_id);
    return static_cast<int>(KV_OK);
  });
}

int kvbm_append_slot_for_decode(kvbm_t h, int64_t seq_id, int32_t* slot_out) {
  if (!h) return KV_ERR_INVALID_ARG;
  Sequence* s = h->find(seq_id);
  if (!s) return KV_ERR_UNKNOWN_SEQ;
  if (h->blocks_needed(*s, 1) > h->free_list.size()) return KV_ERR_OOM;
  int32_t slot = h->append_one(*s);
  if (slot_out) *slot_out = slot;
  return KV_OK;
}

int kvbm_append_slots(kvbm_t h, int64_t seq_id, int64_t num_tokens, int32_t* slots_out) {
  if (!h || num_tokens <= 0) return KV_ERR_INVALID_ARG;
  Sequence* s = h->find(seq_id);
  if (!s) return KV_ERR_UNKNOWN_SEQ;
  if (h->blocks_needed(*s, num_tokens) > h->free_list.size()) return KV_ERR_OOM;
  return guarded([&] {
    s->table.reserve(static_cast<size_t>(ceil_div(s->length + num_tokens, h->block_size)));
    for (int64_t t = 0; t < num_tokens; ++t) {
      int32_t slot = h->append_one(*s);
      if (slots_out) slots_out[t] = slot;
    }
    return static_cast<int>(KV_OK);
  });
}

int kvbm_fork(kvbm_t h, int64_t parent_id, int64_t child_id, int64_t prefix_len) {
  if (!h || child_id < 0) return KV_ERR_INVALID_ARG;
  Sequence* p = h->find(parent_id);
  if (!p) return KV_ERR_UNKNOWN_SEQ;
  if (h->seqs.count(child_id)) return KV_ERR_DUPLICATE_SEQ;
  if (prefix_len < 1 || prefix_len > p->length) return KV_ERR_INVALID_ARG;
  return guarded([&] {
    Sequence c;
    const int64_t nb = ceil_div(prefix_len, h->block_size);
    c.table.assign(p->table.begin(), p->table.begin() + nb);
    c.length = prefix_len;
    for (int32_t b : c.table) ++h->ref_count[static_cast<size_t>(b)];
    h->seqs.emplace(child_id, std::move(c));
    h->released.erase(child_id);
    return static_cast<int>(KV_OK);
  });
}

int kvbm_take_copies(kvbm_t h, int32_t* src, int32_t* dst, int64_t cap, int64_t* n_out) {
  if (!h || !n_out) return KV_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(h->copy_src.size());
  *n_out = n;
  if (n == 0 || (!src && !dst)) return KV_OK;  // nothing queued, or a size query
  if (!src || !dst || cap < n) return KV_ERR_INVALID_ARG;
  std::copy(h->copy_src.begin(), h->copy_src.end(), src);
  std::copy(h->copy_dst.begin(), h->copy_dst.end(), dst);
  h->copy_src.clear();
  h->copy_dst.clear();
  return KV_OK;
}

int kvbm_block_refcount(kvbm_t h, int32_t block, int32_t* out) {
  if (!h || !out || block < 0 || block >= h->num_blocks) return KV_ERR_INVALID_ARG;
  *out = h->ref_count[static_cast<size_t>(block)];
  return KV_OK;
}

int kvbm_can_append_slots(kvbm_t h, const int64_t* seq_ids, int64_t n, int* ok) {
  if (!h || !ok || n < 0 || (n > 0 && !seq_ids)) return KV_ERR_INVALID_ARG;
  int64_t need = 0;
  for (int64_t i = 0; i < n; ++i) {
    Sequence* s = h->find(seq_ids[i]);
    if (!s) return KV_ERR_UNKNOWN_SEQ;
    need += h->blocks_needed(*s, 1);
  }
  *ok = need <= h->free_list.size() ? 1 : 0;
  return KV_OK;
}

int kvbm_export(kvbm_t h, const int64_t* seq_ids, int64_t n, int64_t max_blocks,
                int32_t* block_tables, int32_t* seq_lens) {
  if (!h || n < 0 || max_blocks < 0 || (n > 0 && !seq_ids)) return KV_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i) {  // validate everything before writing
    Sequence* s = h->find(seq_ids[i]);
    if (!s) return KV_ERR_UNKNOWN_SEQ;
    if (static_cast<int64_t>(s->table.size()) > max_blocks) return KV_ERR_INVALID_ARG;
    if (s->length > INT32_MAX) return KV_ERR_INVALID_ARG;
  }
  for (int64_t i = 0; i < n; ++i) {
    const Sequence& s = *h->find(seq_ids[i]);
    if (block_tables) {
      int32_t* row = block_tables + i * max_blocks;
      std::copy(s.table.begin(), s.table.end(), row);
      std::fill(row + s.table.size(), row + max_blocks, -1);
    }
    if (seq_lens) seq_lens[i] = static_cast<int32_t>(s.length);
  }
  return KV_OK;
}

int kvbm_export_update(kvbm_t h, const int64_t* seq_ids, int64_t n, int64_t max_blocks, int32_t* block_tables,
                       int64_t* prev_ids, int32_t* prev_nblocks) {
  if (!h || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !block_tables || !prev_ids || !prev_nblocks)))
    return KV_ERR_INVALID_ARG;
  return guarded([&] {
    std::vector<const Sequence*>& rows = h->export_rows;
    rows.resize(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) {  // validate everything before writing
      const Sequence* s = h->find(seq_ids[i]);
      if (!s) return static_cast<int>(KV_ERR_UNKNOWN_SEQ);
      if (static_cast<int64_t>(s->table.size()) > max_blocks) return static_cast<int>(KV_ERR_INVALID_ARG);
      rows[static_cast<size_t>(i)] = s;
    }
    for (int64_t i = 0; i < n; ++i) {
      const Sequence& s = *rows[static_cast<size_t>(i)];
      int32_t* row = block_tables + i * max_blocks;
      const int64_t nb = static_cast<int64_t>(s.table.size());
      std::copy(s.table.begin(), s.table.end(), row);
      // entries past nb: -1 already where the row held this sequence before,
      // up to its previous block count; everything else is written
      const int32_t pn = prev_nblocks[i];
      const int64_t stale = prev_ids[i] == seq_ids[i] && pn >= 0 && pn <= max_blocks ? pn : max_blocks;
      if (stale > nb) std::fill(row + nb, row + stale, -1);
      prev_ids[i] = seq_ids[i];
      prev_nblocks[i] = static_cast<int32_t>(nb);
    }
    return static_cast<int>(KV_OK);
  });
}

int kvbm_decode_step(kvbm_t h, const int64_t* seq_ids, int64_t n, int64_t max_blocks,
                     int32_t* slots_out, int32_t* block_tables, int32_t* seq_lens) {
  if (!h || n < 0 || (n > 0 && !seq_ids) || max_blocks < 0) return KV_ERR_INVALID_ARG;
  return guarded([&] {
    std::vector<Sequence*> seqs(static_cast<size_t>(n));
    IdSet& seen = h->step_ids;
    seen.reset(n);
    int64_t need = 0;
    for (int64_t i = 0; i < n; ++i) {
      if (!seen.insert(seq_ids[i])) return static_cast<int>(KV_ERR_INVALID_ARG);
      Sequence* s = h->find(seq_ids[i]);
      if (!s) return static_cast<int>(KV_ERR_UNKNOWN_SEQ);
      int64_t grow = h->blocks_needed(*s, 1);
      if (ceil_div(s->length + 1, h->block_size) > max_blocks && (block_tables || seq_lens))
        return static_cast<int>(KV_ERR_INVALID_ARG);
      need += grow;
      seqs[static_cast<size_t>(i)] = s;
    }
    if (need > h->free_list.size()) return static_cast<int>(KV_ERR_OOM);
    for (int64_t i = 0; i < n; ++i) {
      int32_t slot = h->append_one(*seqs[static_cast<size_t>(i)]);
      if (slots_out) slots_out[i] = slot;
    }
    if (block_tables || seq_lens) return kvbm_export(h, seq_ids, n, max_blocks, block_tables, seq_lens);
    return static_cast<int>(KV_OK);
  });
}

int kvbm_prepare_step(kvbm_t h, const int64_t* free_ids, int64_t n_free, const int64_t* prefill_ids,
                      const int64_t* prefill_lens, int64_t n_prefill, const int64_t* decode_ids, int64_t n_decode,
                      const int64_t* pad_positions, int64_t n_pad, int64_t max_blocks, int32_t* slot_mapping,
                      int32_t* block_tables, int32_t* seq_lens) {
  if (!h || n_free < 0 || n_prefill < 0 || n_decode < 0 || n_pad < 0 || max_blocks < 0) return KV_ERR_INVALID_ARG;
  if ((n_free && !free_ids) || (n_prefill && (!prefill_ids || !prefill_lens)) || (n_decode && !decode_ids) ||
      (n_pad && !pad_positions))
    return KV_ERR_INVALID_ARG;
  return guarded([&] {
    // 1. releases: validate all, then release all
    for (int64_t i = 0; i < n_free; ++i) {
      if (!h->seqs.count(free_ids[i]))
        return static_cast<int>(h->released.count(free_ids[i]) ? KV_ERR_DOUBLE_FREE : KV_ERR_UNKNOWN_SEQ);
      for (int64_t k = 0; k < i; ++k)
        if (free_ids[k] == free_ids[i]) return static_cast<int>(KV_ERR_DOUBLE_FREE);
    }
    for (int64_t i = 0; i < n_free; ++i) {
      int st = kvbm_free_sequence(h, free_ids[i]);
      if (st != KV_OK) return st;
    }
    // 2-3. validate the prefills and appends and their block need, before any change
    IdSet& seen = h->step_ids;
    seen.reset(n_prefill + n_decode);
    int64_t n_prefill_tokens = 0, need = 0;
    for (int64_t i = 0; i < n_prefill; ++i) {
      if (prefill_ids[i] < 0 || prefill_lens[i] <= 0) return static_cast<int>(KV_ERR_INVALID_ARG);
      if (h->seqs.count(prefill_ids[i])) return static_cast<int>(KV_ERR_DUPLICATE_SEQ);
      if (!seen.insert(prefill_ids[i])) return static_cast<int>(KV_ERR_DUPLICATE_SEQ);
      n_prefill_tokens += prefill_lens[i];
      need += ceil_div(prefill_lens[i], h->block_size);
    }
    std::vector<Sequence*> dec(static_cast<size_t>(n_decode));
    for (int64_t i = 0; i < n_decode; ++i) {
      Sequence* sq = h->find(decode_ids[i]);
      if (!sq) return static_cast<int>(seen.contains(decode_ids[i]) ? KV_ERR_INVALID_ARG : KV_ERR_UNKNOWN_SEQ);
      if (!seen.insert(decode_ids[i])) return static_cast<int>(KV_ERR_INVALID_ARG);
      const int64_t grow = h->blocks_needed(*sq, 1);
      if ((block_tables || seq_lens) && ceil_div(sq->length + 1, h->block_size) > max_blocks)
        return static_cast<int>(KV_ERR_INVALID_ARG);
      need += grow;
      dec[static_cast<size_t>(i)] = sq;
    }
    const int64_t n_slots = n_prefill_tokens + n_decode + n_pad;
    for (int64_t i = 0; i < n_pad; ++i)
      if (pad_positions[i] < 0 || pad_positions[i] >= n_slots || (i && pad_positions[i] <= pad_positions[i - 1]))
        return static_cast<int>(KV_ERR_INVALID_ARG);
    if (need > h->free_list.size()) return static_cast<int>(KV_ERR_OOM);
    // 4. perform: prefills, then appends, writing slots around the padding
    int64_t pos = 0, pad = 0;
    auto put = [&](int32_t slot) {
      while (pad < n_pad && pad_positions[pad] == pos) {
        if (slot_mapping) slot_mapping[pos] = -1;
        ++pos;
        ++pad;
      }
      if (slot_mapping) slot_mapping[pos] = slot;
      ++pos;
    };
    for (int64_t i = 0; i < n_prefill; ++i) {
      Sequence sq;
      const int64_t nb = ceil_div(prefill_lens[i], h->block_size);
      sq.table.reserve(static_cast<size_t>(nb));
      for (int64_t k = 0; k < nb; ++k) sq.table.push_back(h->take_front());
      sq.length = prefill_lens[i];
      h->for_each_slot(sq, prefill_lens[i], put);
      h->seqs.emplace(prefill_ids[i], std::move(sq));
      h->released.erase(prefill_ids[i]);
    }
    for (int64_t i = 0; i < n_decode; ++i) put(h->append_one(*dec[static_cast<size_t>(i)]));
    while (pad < n_pad) {  // trailing padding
      if (slot_mapping) slot_mapping[pos] = -1;
      ++pos;
      ++pad;
    }
    if (block_tables || seq_lens) return kvbm_export(h, decode_ids, n_decode, max_blocks, block_tables, seq_lens);
    return static_cast<int>(KV_OK);
  });
}

int kvbm_free_sequence(kvbm_t h, int64_t seq_id) {
  if (!h) return KV_ERR_INVALID_ARG;
  auto it = h->seqs.find(seq_id);
  if (it == h->seqs.end()) return h->released.count(seq_id) ? KV_ERR_DOUBLE_FREE : KV_ERR_UNKNOWN_SEQ;
  const std::vector<int32_t>& table = it->second.table;
  // LLM-algo ch.22 release checks: in range, no duplicates, none already free.
  const uint32_t gen = h->next_block_gen();
  for (int32_t b : table) {
    if (b < 0 || b >= h->num_blocks) return KV_ERR_INVARIANT;
    if (h->block_mark[static_cast<size_t>(b)] == gen) return KV_ERR_INVARIANT;
    h->block_mark[static_cast<size_t>(b)] = gen;
    if (h->is_free(b)) return KV_ERR_INVARIANT;
  }
  return guarded([&] {
    for (int32_t b : table) h->unref(b);
    h->seqs.erase(it);
    h->released.insert(seq_id);
    return static_cast<int>(KV_OK);
  });
}

int kvbm_num_free_blocks(kvbm_t h, int64_t* out) {
  if (!h || !out) return KV_ERR_INVALID_ARG;
  *out = h->free_list.size();
  return KV_OK;
}

int kvbm_get_free_list(kvbm_t h, int32_t* out, int64_t cap, int64_t* n_out) {
  if (!h || !n_out) return KV_ERR_INVALID_ARG;
  *n_out = h->free_list.size();
  if (!out) return KV_OK;
  if (cap < h->free_list.size()) return KV_ERR_INVALID_ARG;
  for (int64_t i = 0; i < h->free_list.size(); ++i) out[i] = h->free_list.at(i);
  return KV_OK;
}

int kvbm_seq_len(kvbm_t h, int64_t seq_id, int64_t* out) {
  if (!h || !out) return KV_ERR_INVALID_ARG;
  Sequence* s = h->find(seq_id);
  if (!s) return KV_ERR_UNKNOWN_SEQ;
  *out = s->length;
  return KV_OK;
}

int kvbm_get_block_table(kvbm_t h, int64_t seq_id, int32_t* out, int64_t cap, int64_t* n_out) {
  if (!h || !n_out) return KV_ERR_INVALID_ARG;
  Sequence* s = h->find(seq_id);
  if (!s) return KV_ERR_UNKNOWN_SEQ;
  *n_out = static_cast<int64_t>(s->table.size());
  if (!out) return KV_OK;
  if (cap < *n_out) return KV_ERR_INVALID_ARG;
  std::copy(s->table.begin(), s->table.end(), out);
  return KV_OK;
}

int kvbm_check_invariants(kvbm_t h) {
  if (!h) return KV_ERR_INVALID_ARG;
  return guarded([&] {
    // references per block, counted from the tables; no block twice in one
    // table (a block is shared only across sequences)
    std::vector<int32_t> refs(static_cast<size_t>(h->num_blocks), 0);
    for (const auto& kv : h->seqs) {
      const Sequence& s = kv.second;
      if (static_cast<int64_t>(s.table.size()) != ceil_div(s.length, h->block_size))
        return static_cast<int>(KV_ERR_INVARIANT);
      std::unordered_set<int32_t> in_table;
      for (int32_t b : s.table) {
        if (b < 0 || b >= h->num_blocks) return static_cast<int>(KV_ERR_INVARIANT);
        if (!in_table.insert(b).second) return static_cast<int>(KV_ERR_INVARIANT);
        ++refs[static_cast<size_t>(b)];
      }
    }
    int64_t allocated = 0;
    for (int64_t b = 0; b < h->num_blocks; ++b) {
      if (refs[static_cast<size_t>(b)] != h->ref_count[static_cast<size_t>(b)]) return static_cast<int>(KV_ERR_INVARIANT);
      if (refs[static_cast<size_t>(b)] > 0) ++allocated;
    }
    // the free list holds exactly the unreferenced blocks, once each
    std::vector<uint8_t> in_free(static_cast<size_t>(h->num_blocks), 0);
    for (int64_t i = 0; i < h->free_list.size(); ++i) {
      int32_t b = h->free_list.at(i);
      if (b < 0 || b >= h->num_blocks) return static_cast<int>(KV_ERR_INVARIANT);
      if (in_free[static_cast<size_t>(b)] || refs[static_cast<size_t>(b)] != 0)
        return static_cast<int>(KV_ERR_INVARIANT);
      in_free[static_cast<size_t>(b)] = 1;
    }
    if (allocated + h->free_list.size() != h->num_blocks) return static_cast<int>(KV_ERR_INVARIANT);
    return static_cast<int>(KV_OK);
  });
}

int kvbm_stats(kvbm_t h, kvbm_stats_t* out) {
  if (!h || !out) return KV_ERR_INVALID_ARG;
  kvbm_stats_t st{};
  st.num_blocks = h->num_blocks;
  st.block_size = h->block_size;
  st.num_free_blocks = h->free_list.size();
  st.num_sequences = static_cast<int64_t>(h->seqs.size());
  for (const auto& kv : h->seqs) {
    st.logical_tokens += kv.second.length;
    st.allocated_tokens += static_cast<int64_t>(kv.second.table.size()) * h->block_size;
  }
  st.unused_tail_tokens = st.allocated_tokens - st.logical_tokens;
  *out = st;
  return KV_OK;
}

int kvbm_released_ranges(kvbm_t h, int64_t* out) {
  if (!h || !out) return KV_ERR_INVALID_ARG;
  *out = static_cast<int64_t>(h->released.ranges());
  return KV_OK;
}

int kvbm_allocation_report(kvbm_t h, int64_t seq_id, int64_t* logical_tokens,
                           int64_t* allocated_tokens, int64_t* unused_tail_tokens,
                           double* utilization) {
  if (!h) return KV_ERR_INVALID_ARG;
  Sequence* s = h->find(seq_id);
  if (!s) return KV_ERR_UNKNOWN_SEQ;
  int64_t alloc = static_cast<int64_t>(s->table.size()) * h->block_size;
  if (logical_tokens) *logical_tokens = s->length;
  if (allocated_tokens) *allocated_tokens = alloc;
  if (unused_tail_tokens) *unused_tail_tokens = alloc - s->length;
  if (utilization) *utilization = alloc ? static_cast<double>(s->length) / static_cast<double>(alloc) : 0.0;
  return KV_OK;
}

int kvbm_owner_table(kvbm_t h, int64_t* out, int64_t cap) {
  if (!h || !out || cap < h->num_blocks) return KV_ERR_INVALID_ARG;
  std::fill(out, out + h->num_blocks, int64_t{-1});
  for (const auto& kv : h->seqs)
    for (int32_t b : kv.second.table) {
      if (b < 0 || b >= h->num_blocks) return KV_ERR_INVARIANT;
      out[b] = out[b] == -1 ? kv.first : -2;  // -2: held by several sequences
    }
  return KV_OK;
}

int kv_cache_ledger(int64_t num_blocks, int64_t block_size, int64_t num_layers,
                    int64_t num_kv_heads, int64_t head_dim, int64_t dtype_bytes,
                    int64_t* bytes_per_token, int64_t* bytes_per_block, int64_t* total_bytes) {
  if (num_blocks <= 0 || block_size <= 0 || num_layers <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      dtype_bytes <= 0)
    return KV_ERR_INVALID_ARG;
  int64_t per_token = 2 * num_layers * num_kv_heads * head_dim * dtype_bytes;
  int64_t per_block = block_size * per_token;
  if (bytes_per_token) *bytes_per_token = per_token;
  if (bytes_per_block) *bytes_per_block = per_block;
  if (total_bytes) *total_bytes = num_blocks * per_block;
  return KV_OK;
}

}  // extern "C"
