// Host block allocator for the paged KV cache.
//
// Follows the block lifecycle of kasblo.com "vLLMとは？LLMサーバーを高速化する仕組み",
// section "blockはrequestの成長に合わせて割り当てる" (take blocks for the prompt from
// the pool, add one when the current block fills, return a request's blocks when
// it ends, reuse them later) and the reference-counted sharing of section
// "block共有とAutomatic Prefix Caching".  Physical placement is deliberately
// scattered: each free block is drawn at random (seeded) from the free list,
// as in the PagedAttention memory-layout figure of youngju.dev
// "LLM サービング最適化完全ガイド" where a request's blocks need not be adjacent.
//
// The random draw uses splitmix64 so that a seed gives the same placement on
// every host architecture.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "paged_kv.h"
#include "pkv_errors.h"

struct pkv_block_allocator {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  uint64_t rng = 0;
  std::vector<int32_t> free_list;   // unordered; random pick by swap-remove
  std::vector<int32_t> refcount;    // per physical block, 0 = free
  struct Seq {
    std::vector<int32_t> blocks;
    int32_t len = 0;
    bool live = false;
    uint64_t stamp = 0;  // last batch call that listed this sequence
  };
  std::vector<Seq> seqs;
  uint64_t batch_calls = 0;
  std::vector<int32_t> dead_ids;    // reusable sequence ids

  uint64_t next_u64() {
    uint64_t z = (rng += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }

  int32_t pop_block() {
    const uint64_t n = free_list.size();
    const uint64_t idx = next_u64() % n;
    const int32_t blk = free_list[idx];
    free_list[idx] = free_list.back();
    free_list.pop_back();
    refcount[blk] = 1;
    return blk;
  }

  void release_block(int32_t blk) {
    if (--refcount[blk] == 0) free_list.push_back(blk);
  }

  int32_t new_seq_id() {
    if (!dead_ids.empty()) {
      const int32_t id = dead_ids.back();
      dead_ids.pop_back();
      return id;
    }
    seqs.emplace_back();
    return static_cast<int32_t>(seqs.size() - 1);
  }

  bool live(int32_t id) const {
    return id >= 0 && id < static_cast<int32_t>(seqs.size()) && seqs[id].live;
  }

  int32_t blocks_for(int32_t tokens) const { return (tokens + block_size - 1) / block_size; }
};

extern "C" {

pkv_block_allocator* block_allocator_create(int32_t num_blocks, int32_t block_size, uint64_t seed) {
  if (num_blocks <= 0 || block_size <= 0) {
    pkv_set_error("block_allocator_create: num_blocks and block_size must be positive");
    return nullptr;
  }
  auto* a = new pkv_block_allocator();
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->rng = seed;
  a->free_list.resize(num_blocks);
  for (int32_t i = 0; i < num_blocks; ++i) a->free_list[i] = i;
  a->refcount.assign(num_blocks, 0);
  return a;
}

void block_allocator_destroy(pkv_block_allocator* a) { delete a; }

int block_allocator_add_seq(pkv_block_allocator* a, int32_t num_tokens, int32_t* seq_id) {
  if (!a || !seq_id || num_tokens < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "add_seq: bad argument");
  const int32_t need = a->blocks_for(num_tokens);
  if (need > static_cast<int32_t>(a->free_list.size()))
    return pkv_fail(PKV_ERR_NO_BLOCKS, "add_seq: pool has too few free blocks");
  const int32_t id = a->new_seq_id();
  auto& s = a->seqs[id];
  s.blocks.clear();
  for (int32_t j = 0; j < need; ++j) s.blocks.push_back(a->pop_block());
  s.len = num_tokens;
  s.live = true;
  *seq_id = id;
  return PKV_OK;
}

int block_allocator_fork_prefix(pkv_block_allocator* a, int32_t src_seq, int32_t prefix_tokens,
                                int32_t num_tokens, int32_t* seq_id) {
  if (!a || !seq_id || !a->live(src_seq))
    return pkv_fail(PKV_ERR_INVALID_ARG, "fork_prefix: bad allocator or source sequence");
  if (prefix_tokens < 0 || prefix_tokens % a->block_size != 0 ||
      prefix_tokens > a->seqs[src_seq].len || num_tokens < prefix_tokens)
    return pkv_fail(PKV_ERR_INVALID_ARG,
                    "fork_prefix: prefix must be whole blocks of the source and <= num_tokens");
  const int32_t shared = prefix_tokens / a->block_size;
  const int32_t need = a->blocks_for(num_tokens) - shared;
  if (need > static_cast<int32_t>(a->free_list.size()))
    return pkv_fail(PKV_ERR_NO_BLOCKS, "fork_prefix: pool has too few free blocks");
  const int32_t id = a->new_seq_id();  // may grow seqs: take references after this
  auto& src = a->seqs[src_seq];
  auto& s = a->seqs[id];
  s.blocks.assign(src.blocks.begin(), src.blocks.begin() + shared);
  for (int32_t blk : s.blocks) ++a->refcount[blk];
  for (int32_t j = 0; j < need; ++j) s.blocks.push_back(a->pop_block());
  s.len = num_tokens;
  s.live = true;
  *seq_id = id;
  return PKV_OK;
}

int block_allocator_fork(pkv_block_allocator* a, int32_t src_seq, int32_t prefix_tokens, int32_t* seq_id) {
  if (!a || !seq_id || !a->live(src_seq)) return pkv_fail(PKV_ERR_INVALID_ARG, "fork: bad allocator or source");
  if (prefix_tokens < 0 || prefix_tokens > a->seqs[src_seq].len)
    return pkv_fail(PKV_ERR_INVALID_ARG, "fork: prefix must be 0..length of the source");
  const int32_t id = a->new_seq_id();  // may grow seqs: take references after this
  auto& src = a->seqs[src_seq];
  auto& s = a->seqs[id];
  s.blocks.assign(src.blocks.begin(), src.blocks.begin() + a->blocks_for(prefix_tokens));
  for (int32_t blk : s.blocks) ++a->refcount[blk];
  s.len = prefix_tokens;
  s.live = true;
  *seq_id = id;
  return PKV_OK;
}

namespace {
// Block j of sequence s is about to be written: if another sequence holds it
// too, give s a private copy (a fresh block) and report the copy.
void copy_on_write(pkv_block_allocator* a, pkv_block_allocator::Seq& s, int32_t j, int32_t* pair, int32_t* copies) {
  const int32_t old = s.blocks[j];
  if (a->refcount[old] <= 1) return;
  const int32_t fresh = a->pop_block();
  --a->refcount[old];
  s.blocks[j] = fresh;
  pair[0] = old;
  pair[1] = fresh;
  ++*copies;
}
}  // namespace

int block_allocator_append_slot_cow(pkv_block_allocator* a, int32_t seq_id, int32_t* slot, int32_t* copy_pair,
                                    int32_t* num_copies) {
  if (!a || !slot || !copy_pair || !num_copies || !a->live(seq_id))
    return pkv_fail(PKV_ERR_INVALID_ARG, "append_slot_cow: bad argument");
  auto& s = a->seqs[seq_id];
  const int32_t pos = s.len;
  const int32_t j = pos / a->block_size;
  *num_copies = 0;
  if (a->free_list.empty() && (j == static_cast<int32_t>(s.blocks.size()) || a->refcount[s.blocks[j]] > 1))
    return pkv_fail(PKV_ERR_NO_BLOCKS, "append_slot_cow: pool is empty");
  if (j == static_cast<int32_t>(s.blocks.size()))
    s.blocks.push_back(a->pop_block());
  else
    copy_on_write(a, s, j, copy_pair, num_copies);
  *slot = s.blocks[j] * a->block_size + pos % a->block_size;
  s.len = pos + 1;
  return PKV_OK;
}

int block_allocator_step_batch_cow(pkv_block_allocator* a, const int32_t* slot_seq_ids, int32_t n,
                                   int32_t max_blocks, int32_t* tables, int32_t* context_lens, int32_t* copy_pairs,
                                   int32_t* num_copies) {
  if (!a || n < 0 || max_blocks < 0 || !num_copies ||
      (n > 0 && (!slot_seq_ids || !tables || !context_lens || !copy_pairs)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "step_batch_cow: bad argument");
  *num_copies = 0;
  // Check first, so that a failure changes nothing.  A block shared only
  // within this batch is copied for all but the last of its holders to write
  // into it, so count the writers per shared block.
  int32_t need = 0;
  const uint64_t stamp = ++a->batch_calls;
  std::vector<int32_t> writers;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = slot_seq_ids[i];
    if (id < 0) continue;
    if (!a->live(id)) return pkv_fail(PKV_ERR_INVALID_ARG, "step_batch_cow: sequence not live");
    auto& s = a->seqs[id];
    if (s.stamp == stamp) return pkv_fail(PKV_ERR_INVALID_ARG, "step_batch_cow: sequence listed twice");
    s.stamp = stamp;
    if (a->blocks_for(s.len + 1) > max_blocks)
      return pkv_fail(PKV_ERR_INVALID_ARG, "step_batch_cow: a sequence would outgrow max_blocks");
    const int32_t j = s.len / a->block_size;
    if (j == static_cast<int32_t>(s.blocks.size()))
      ++need;
    else if (a->refcount[s.blocks[j]] > 1)
      writers.push_back(s.blocks[j]);
  }
  // Each shared block written by w sequences of the batch needs
  // min(w, refcount - 1) copies: the last holder keeps the original.
  std::sort(writers.begin(), writers.end());
  for (size_t i = 0; i < writers.size();) {
    size_t k = i;
    while (k < writers.size() && writers[k] == writers[i]) ++k;
    const int32_t w = static_cast<int32_t>(k - i), rc = a->refcount[writers[i]];
    need += w < rc - 1 ? w : rc - 1;
    i = k;
  }
  if (need > static_cast<int32_t>(a->free_list.size()))
    return pkv_fail(PKV_ERR_NO_BLOCKS, "step_batch_cow: pool has too few free blocks for this step");
  for (int32_t i = 0; i < n; ++i) {
    int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
    const int32_t id = slot_seq_ids[i];
    int32_t k = 0;
    if (id >= 0) {
      int32_t slot, c = 0;
      block_allocator_append_slot_cow(a, id, &slot, copy_pairs + 2 * static_cast<int64_t>(*num_copies), &c);
      *num_copies += c;
      const auto& s = a->seqs[id];
      for (; k < static_cast<int32_t>(s.blocks.size()); ++k) row[k] = s.blocks[k];
      context_lens[i] = s.len;
    } else {
      context_lens[i] = 0;
    }
    for (; k < max_blocks; ++k) row[k] = -1;
  }
  return PKV_OK;
}

int block_allocator_append_slot(pkv_block_allocator* a, int32_t seq_id, int32_t* slot) {
  if (!a || !slot || !a->live(seq_id)) return pkv_fail(PKV_ERR_INVALID_ARG, "append_slot: bad sequence");
  auto& s = a->seqs[seq_id];
  const int32_t pos = s.len;
  const int32_t j = pos / a->block_size;
  if (j == static_cast<int32_t>(s.blocks.size())) {
    if (a->free_list.empty()) return pkv_fail(PKV_ERR_NO_BLOCKS, "append_slot: pool is empty");
    s.blocks.push_back(a->pop_block());
  } else if (a->refcount[s.blocks[j]] > 1) {
    return pkv_fail(PKV_ERR_SHARED_BLOCK, "append_slot: last block is shared with another sequence");
  }
  *slot = s.blocks[j] * a->block_size + pos % a->block_size;
  s.len = pos + 1;
  return PKV_OK;
}

int block_allocator_append_slots(pkv_block_allocator* a, const int32_t* seq_ids, int32_t n, int32_t* slots) {
  if (!a || n < 0 || (n > 0 && (!seq_ids || !slots))) return pkv_fail(PKV_ERR_INVALID_ARG, "append_slots: bad argument");
  // Check first, so that a failure changes nothing: each sequence is live,
  // appears once, and the pool holds the blocks the batch needs.
  int32_t need = 0;
  const uint64_t stamp = ++a->batch_calls;
  for (int32_t i = 0; i < n; ++i) {
    if (!a->live(seq_ids[i])) return pkv_fail(PKV_ERR_INVALID_ARG, "append_slots: sequence not live");
    auto& s = a->seqs[seq_ids[i]];
    if (s.stamp == stamp) return pkv_fail(PKV_ERR_INVALID_ARG, "append_slots: sequence listed twice");
    s.stamp = stamp;
    const int32_t j = s.len / a->block_size;
    if (j == static_cast<int32_t>(s.blocks.size())) {
      ++need;
    } else if (a->refcount[s.blocks[j]] > 1) {
      return pkv_fail(PKV_ERR_SHARED_BLOCK, "append_slots: a last block is shared with another sequence");
    }
  }
  if (need > static_cast<int32_t>(a->free_list.size()))
    return pkv_fail(PKV_ERR_NO_BLOCKS, "append_slots: pool has too few free blocks for this step");
  for (int32_t i = 0; i < n; ++i) {
    const int rc = block_allocator_append_slot(a, seq_ids[i], &slots[i]);
    if (rc != PKV_OK) return rc;  // unreachable after the checks above
  }
  return PKV_OK;
}

int block_allocator_step_batch(pkv_block_allocator* a, const int32_t* slot_seq_ids, int32_t n, int32_t max_blocks,
                               int32_t* tables, int32_t* context_lens) {
  if (!a || n < 0 || max_blocks < 0 || (n > 0 && (!slot_seq_ids || !tables || !context_lens)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "step_batch: bad argument");
  // Same checks as append_slots, plus the table width, before changing anything.
  int32_t need = 0;
  const uint64_t stamp = ++a->batch_calls;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = slot_seq_ids[i];
    if (id < 0) continue;
    if (!a->live(id)) return pkv_fail(PKV_ERR_INVALID_ARG, "step_batch: sequence not live");
    auto& s = a->seqs[id];
    if (s.stamp == stamp) return pkv_fail(PKV_ERR_INVALID_ARG, "step_batch: sequence listed twice");
    s.stamp = stamp;
    if (a->blocks_for(s.len + 1) > max_blocks)
      return pkv_fail(PKV_ERR_INVALID_ARG, "step_batch: a sequence would outgrow max_blocks");
    const int32_t j = s.len / a->block_size;
    if (j == static_cast<int32_t>(s.blocks.size())) {
      ++need;
    } else if (a->refcount[s.blocks[j]] > 1) {
      return pkv_fail(PKV_ERR_SHARED_BLOCK, "step_batch: a last block is shared with another sequence");
    }
  }
  if (need > static_cast<int32_t>(a->free_list.size()))
    return pkv_fail(PKV_ERR_NO_BLOCKS, "step_batch: pool has too few free blocks for this step");
  for (int32_t i = 0; i < n; ++i) {
    int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
    const int32_t id = slot_seq_ids[i];
    int32_t k = 0;
    if (id >= 0) {
      int32_t slot;
      block_allocator_append_slot(a, id, &slot);  // cannot fail after the checks above
      const auto& s = a->seqs[id];
      for (; k < static_cast<int32_t>(s.blocks.size()); ++k) row[k] = s.blocks[k];
      context_lens[i] = s.len;
    } else {
      context_lens[i] = 0;
    }
    for (; k < max_blocks; ++k) row[k] = -1;
  }
  return PKV_OK;
}

int block_allocator_free_seq(pkv_block_allocator* a, int32_t seq_id) {
  if (!a || !a->live(seq_id)) return pkv_fail(PKV_ERR_INVALID_ARG, "free_seq: bad sequence");
  auto& s = a->seqs[seq_id];
  for (int32_t blk : s.blocks) a->release_block(blk);
  s.blocks.clear();
  s.len = 0;
  s.live = false;
  a->dead_ids.push_back(seq_id);
  return PKV_OK;
}

int block_allocator_block_tables(const pkv_block_allocator* a, const int32_t* seq_ids, int32_t n,
                                 int32_t max_blocks, int32_t* tables, int32_t* context_lens) {
  if (!a || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !tables || !context_lens)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "block_tables: bad argument");
  for (int32_t i = 0; i < n; ++i) {
    if (!a->live(seq_ids[i])) return pkv_fail(PKV_ERR_INVALID_ARG, "block_tables: sequence not live");
    const auto& s = a->seqs[seq_ids[i]];
    if (static_cast<int32_t>(s.blocks.size()) > max_blocks)
      return pkv_fail(PKV_ERR_INVALID_ARG, "block_tables: sequence needs more than max_blocks");
  }
  for (int32_t i = 0; i < n; ++i) {
    const auto& s = a->seqs[seq_ids[i]];
    int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
    int32_t j = 0;
    for (; j < static_cast<int32_t>(s.blocks.size()); ++j) row[j] = s.blocks[j];
    for (; j < max_blocks; ++j) row[j] = -1;
    context_lens[i] = s.len;
  }
  return PKV_OK;
}

int32_t block_allocator_num_free(const pkv_block_allocator* a) {
  return a ? static_cast<int32_t>(a->free_list.size()) : -1;
}

int32_t block_allocator_refcount(const pkv_block_allocator* a, int32_t block) {
  if (!a || block < 0 || block >= a->num_blocks) return -1;
  return a->refcount[block];
}

int32_t block_allocator_seq_len(const pkv_block_allocator* a, int32_t seq_id) {
  if (!a || !a->live(seq_id)) return -1;
  return a->seqs[seq_id].len;
}

int paged_kv_slot_mapping(const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
                          int32_t max_blocks, int32_t block_size, int32_t* slot_mapping) {
  if (num_seqs < 0 || max_blocks < 0 || block_size <= 0 ||
      (num_seqs > 0 && (!block_tables || !context_lens || !slot_mapping)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "slot_mapping: bad argument");
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t L = context_lens[b];
    if (L <= 0) {
      slot_mapping[b] = -1;
      continue;
    }
    const int32_t pos = L - 1;
    const int32_t j = pos / block_size;
    if (j >= max_blocks) return pkv_fail(PKV_ERR_INVALID_ARG, "slot_mapping: context longer than its table");
    const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks + j];
    if (blk < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "slot_mapping: table entry is -1");
    slot_mapping[b] = blk * block_size + pos % block_size;
  }
  return PKV_OK;
}

int paged_kv_slot_mapping_multi(const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
                                int32_t max_blocks, int32_t block_size, int32_t q_len, int32_t* slot_mapping) {
  if (num_seqs < 0 || max_blocks < 0 || block_size <= 0 || q_len < 1 ||
      (num_seqs > 0 && (!block_tables || !context_lens || !slot_mapping)))
    return pkv_fail(PKV_ERR_INVALID_ARG, "slot_mapping_multi: bad argument");
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t L = context_lens[b];
    for (int32_t i = 0; i < q_len; ++i) {
      const int32_t pos = L - q_len + i;
      int32_t& out = slot_mapping[static_cast<int64_t>(b) * q_len + i];
      if (pos < 0) {
        out = -1;
        continue;
      }
      const int32_t j = pos / block_size;
      if (j >= max_blocks) return pkv_fail(PKV_ERR_INVALID_ARG, "slot_mapping_multi: context longer than its table");
      const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks + j];
      if (blk < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "slot_mapping_multi: table entry is -1");
      out = blk * block_size + pos % block_size;
    }
  }
  return PKV_OK;
}

}  // extern "C"
