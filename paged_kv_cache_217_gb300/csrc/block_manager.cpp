// Host block manager: free stack, per-block refcounts, per-sequence block
// tables, slot reservation with copy-on-write.
//
// Follows the KV cache manager of the abeam.tech summary of "Efficient Memory
// Management for Large Language Model Serving with PagedAttention" (section
// "KV キャッシュマネージャ": tokens fill the last block, a new block is taken
// when it is full, a finished request returns its blocks) and its sharing
// section "並列サンプリングやビームサーチでの共有" (samples share prompt
// blocks; a shared block is copied only when a write reaches it). The blog
// "数万トークンでもVRAMが溢れない！..." (section "OSの知恵をGPUへ") fixes that
// sharing is by reference count only and that waste is confined to the last
// block. Readings for what the pages leave open (stack order, copy rule) are
// stated in include/paged_kv.h.
#include <algorithm>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "paged_kv.h"
#include "status.h"

struct pkv_bm {
  struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
  };
  int num_blocks = 0;
  std::vector<int32_t> free_stack;  // top = back()
  std::vector<int32_t> refcount;
  std::unordered_map<int64_t, Seq> seqs;

  int32_t pop() {
    int32_t b = free_stack.back();
    free_stack.pop_back();
    refcount[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--refcount[b] == 0) free_stack.push_back(b);
  }
};

namespace {

// What one append did, so a failed batch can be undone in reverse order.
struct AppendUndo {
  int64_t seq;
  int32_t fresh = -1;     // block pushed onto the table (L % 16 == 0 case)
  int32_t cow_src = -1;   // copy-on-write: old block (refcount was decremented)
  int32_t cow_dst = -1;   // copy-on-write: new block now last in the table
};

pkv_status_t append_one(pkv_bm* bm, int64_t seq_id, int64_t* slot, int64_t* src,
                        int64_t* dst, AppendUndo* undo) {
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return pkv::fail(PKV_ERR_INVALID_ARG, "append_slot: unknown sequence %lld", (long long)seq_id);
  auto& s = it->second;
  const int64_t L = s.len;
  *src = *dst = -1;
  undo->seq = seq_id;
  if (L % PKV_BLOCK_SIZE == 0) {
    if (bm->free_stack.empty()) return pkv::fail(PKV_ERR_OUT_OF_BLOCKS, "append_slot: no free block");
    const int32_t b = bm->pop();
    s.table.push_back(b);
    undo->fresh = b;
  } else {
    const int32_t last = s.table.back();
    if (bm->refcount[last] > 1) {
      if (bm->free_stack.empty()) return pkv::fail(PKV_ERR_OUT_OF_BLOCKS, "append_slot: no free block for copy-on-write");
      const int32_t nb = bm->pop();
      bm->refcount[last] -= 1;
      s.table.back() = nb;
      *src = last;
      *dst = nb;
      undo->cow_src = last;
      undo->cow_dst = nb;
    }
  }
  *slot = int64_t(s.table[L / PKV_BLOCK_SIZE]) * PKV_BLOCK_SIZE + L % PKV_BLOCK_SIZE;
  s.len = L + 1;
  return PKV_OK;
}

void undo_append(pkv_bm* bm, const AppendUndo& u) {
  auto& s = bm->seqs[u.seq];
  s.len -= 1;
  if (u.fresh >= 0) {
    s.table.pop_back();
    bm->refcount[u.fresh] = 0;
    bm->free_stack.push_back(u.fresh);
  } else if (u.cow_dst >= 0) {
    s.table.back() = u.cow_src;
    bm->refcount[u.cow_src] += 1;
    bm->refcount[u.cow_dst] = 0;
    bm->free_stack.push_back(u.cow_dst);
  }
}

}  // namespace

extern "C" {

pkv_status_t pkv_bm_create(int num_blocks, int block_size, const int32_t* initial_free_order,
                           pkv_bm_t** out) {
  if (!out) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_create: out is NULL");
  *out = nullptr;
  if (num_blocks <= 0) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_create: num_blocks must be > 0");
  if (block_size != PKV_BLOCK_SIZE) return pkv::fail(PKV_ERR_UNSUPPORTED, "bm_create: block_size must be 16");
  pkv_bm* bm = new (std::nothrow) pkv_bm();
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_create: out of host memory");
  bm->num_blocks = num_blocks;
  bm->refcount.assign(num_blocks, 0);
  bm->free_stack.resize(num_blocks);
  if (initial_free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
      const int32_t b = initial_free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete bm;
        return pkv::fail(PKV_ERR_INVALID_ARG, "bm_create: initial_free_order is not a permutation");
      }
      seen[b] = 1;
      bm->free_stack[i] = b;
    }
  } else {
    for (int i = 0; i < num_blocks; ++i) bm->free_stack[i] = i;
  }
  *out = bm;
  return pkv::ok();
}

void pkv_bm_destroy(pkv_bm_t* bm) { delete bm; }

pkv_status_t pkv_bm_add_seq(pkv_bm_t* bm, int64_t seq_id, int64_t num_tokens) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_add_seq: NULL handle");
  if (num_tokens < 0) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_add_seq: num_tokens < 0");
  if (bm->seqs.count(seq_id)) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_add_seq: sequence %lld exists", (long long)seq_id);
  const int64_t nb = (num_tokens + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE;
  if (nb > int64_t(bm->free_stack.size()))
    return pkv::fail(PKV_ERR_OUT_OF_BLOCKS, "bm_add_seq: need %lld blocks, %zu free", (long long)nb, bm->free_stack.size());
  pkv_bm::Seq s;
  s.table.reserve(size_t(nb) + 1);
  for (int64_t i = 0; i < nb; ++i) s.table.push_back(bm->pop());
  s.len = num_tokens;
  bm->seqs.emplace(seq_id, std::move(s));
  return pkv::ok();
}

pkv_status_t pkv_bm_fork(pkv_bm_t* bm, int64_t parent, int64_t child) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_fork: NULL handle");
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_fork: unknown parent %lld", (long long)parent);
  if (bm->seqs.count(child)) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_fork: sequence %lld exists", (long long)child);
  pkv_bm::Seq c = it->second;  // copy before emplace (rehash may move it)
  for (int32_t b : c.table)
    if (b >= 0) bm->refcount[b] += 1;  // released entries (-1) are not shared
  bm->seqs.emplace(child, std::move(c));
  return pkv::ok();
}

pkv_status_t pkv_bm_append_slot(pkv_bm_t* bm, int64_t seq_id, int64_t* slot_out,
                                int64_t* cow_src_out, int64_t* cow_dst_out) {
  if (!bm || !slot_out || !cow_src_out || !cow_dst_out)
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_append_slot: NULL argument");
  AppendUndo u;
  int64_t slot, src, dst;
  pkv_status_t st = append_one(bm, seq_id, &slot, &src, &dst, &u);
  if (st != PKV_OK) return st;
  *slot_out = slot;
  *cow_src_out = src;
  *cow_dst_out = dst;
  return pkv::ok();
}

pkv_status_t pkv_bm_append_slots(pkv_bm_t* bm, const int64_t* seq_ids, int n, int64_t* slots_out,
                                 int64_t* pairs_out, int* num_pairs_out) {
  if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots_out || !pairs_out)) || !num_pairs_out)
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_append_slots: bad argument");
  std::vector<AppendUndo> log;
  log.reserve(size_t(n));
  int np = 0;
  for (int i = 0; i < n; ++i) {
    AppendUndo u;
    int64_t src, dst;
    pkv_status_t st = append_one(bm, seq_ids[i], &slots_out[i], &src, &dst, &u);
    if (st != PKV_OK) {
      for (auto r = log.rbegin(); r != log.rend(); ++r) undo_append(bm, *r);
      return st;  // message already recorded by append_one
    }
    log.push_back(u);
    if (src >= 0) {
      pairs_out[2 * np] = src;
      pairs_out[2 * np + 1] = dst;
      ++np;
    }
  }
  *num_pairs_out = np;
  return pkv::ok();
}

pkv_status_t pkv_bm_free_seq(pkv_bm_t* bm, int64_t seq_id) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_free_seq: NULL handle");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_free_seq: unknown sequence %lld", (long long)seq_id);
  for (int32_t b : it->second.table)
    if (b >= 0) bm->release(b);
  bm->seqs.erase(it);
  return pkv::ok();
}

pkv_status_t pkv_bm_beam_reorder(pkv_bm_t* bm, const int64_t* old_ids, int num_old, const int32_t* parents,
                                const int64_t* new_ids, int num_new) {
  if (!bm || num_old < 0 || num_new < 0 || (num_old > 0 && !old_ids) || (num_new > 0 && (!parents || !new_ids)))
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_beam_reorder: bad argument");
  // Validate everything before touching the state.
  std::unordered_map<int64_t, int> old_index;
  for (int i = 0; i < num_old; ++i) {
    if (!bm->seqs.count(old_ids[i]) || !old_index.emplace(old_ids[i], i).second)
      return pkv::fail(PKV_ERR_INVALID_ARG, "bm_beam_reorder: old beam %lld is unknown or repeated",
                       (long long)old_ids[i]);
  }
  std::unordered_map<int64_t, int> seen_new;
  for (int i = 0; i < num_new; ++i) {
    if (parents[i] < 0 || parents[i] >= num_old)
      return pkv::fail(PKV_ERR_INVALID_ARG, "bm_beam_reorder: parent %d of new beam %d outside [0, %d)",
                       int(parents[i]), i, num_old);
    if (!seen_new.emplace(new_ids[i], i).second)
      return pkv::fail(PKV_ERR_INVALID_ARG, "bm_beam_reorder: new beam id %lld repeated", (long long)new_ids[i]);
    if (bm->seqs.count(new_ids[i]) && !old_index.count(new_ids[i]))
      return pkv::fail(PKV_ERR_INVALID_ARG, "bm_beam_reorder: new beam id %lld is a live sequence",
                       (long long)new_ids[i]);
  }
  // Children copy their parents' tables (references only), then the old beams go.
  std::vector<pkv_bm::Seq> children;
  children.reserve(size_t(num_new));
  for (int i = 0; i < num_new; ++i) {
    children.push_back(bm->seqs.find(old_ids[parents[i]])->second);
    for (int32_t b : children.back().table)
      if (b >= 0) bm->refcount[b] += 1;
  }
  for (int i = 0; i < num_old; ++i) {
    auto it = bm->seqs.find(old_ids[i]);
    for (int32_t b : it->second.table)
      if (b >= 0) bm->release(b);
    bm->seqs.erase(it);
  }
  for (int i = 0; i < num_new; ++i) bm->seqs.emplace(new_ids[i], std::move(children[size_t(i)]));
  return pkv::ok();
}

pkv_status_t pkv_bm_add_seq_with_prefix(pkv_bm_t* bm, int64_t seq_id, int64_t num_tokens, int64_t donor,
                                        int64_t prefix_tokens, int64_t* shared_tokens_out) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_add_seq_with_prefix: NULL handle");
  if (num_tokens < 0 || prefix_tokens < 0)
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_add_seq_with_prefix: negative size");
  if (bm->seqs.count(seq_id))
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_add_seq_with_prefix: sequence %lld exists", (long long)seq_id);
  auto dit = bm->seqs.find(donor);
  if (dit == bm->seqs.end())
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_add_seq_with_prefix: unknown donor %lld", (long long)donor);
  const pkv_bm::Seq& d = dit->second;
  const int64_t shared = std::min(std::min(prefix_tokens, num_tokens), d.len) / PKV_BLOCK_SIZE;
  for (int64_t j = 0; j < shared; ++j)
    if (d.table[size_t(j)] < 0)
      return pkv::fail(PKV_ERR_INVALID_ARG, "bm_add_seq_with_prefix: the donor released block %lld of the prefix",
                       (long long)j);
  const int64_t fresh = (num_tokens + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE - shared;
  if (fresh > int64_t(bm->free_stack.size()))
    return pkv::fail(PKV_ERR_OUT_OF_BLOCKS, "bm_add_seq_with_prefix: need %lld fresh blocks, %zu free",
                     (long long)fresh, bm->free_stack.size());
  pkv_bm::Seq s;
  s.table.reserve(size_t(shared + fresh) + 1);
  for (int64_t j = 0; j < shared; ++j) {
    const int32_t b = d.table[size_t(j)];
    bm->refcount[b] += 1;
    s.table.push_back(b);
  }
  for (int64_t j = 0; j < fresh; ++j) s.table.push_back(bm->pop());
  s.len = num_tokens;
  bm->seqs.emplace(seq_id, std::move(s));  // d is not used after this point (rehash)
  if (shared_tokens_out) *shared_tokens_out = shared * PKV_BLOCK_SIZE;
  return pkv::ok();
}

pkv_status_t pkv_bm_release_before(pkv_bm_t* bm, int64_t seq_id, int64_t first_token, int* released_out) {
  if (!bm) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_release_before: NULL handle");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end())
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_release_before: unknown sequence %lld", (long long)seq_id);
  auto& s = it->second;
  if (first_token < 0 || first_token > s.len)
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_release_before: first_token %lld outside [0, %lld]",
                     (long long)first_token, (long long)s.len);
  int released = 0;
  const int64_t whole = first_token / PKV_BLOCK_SIZE;  // blocks wholly before first_token
  for (int64_t j = 0; j < whole; ++j) {
    int32_t& b = s.table[size_t(j)];
    if (b < 0) continue;
    bm->release(b);
    b = -1;
    ++released;
  }
  if (released_out) *released_out = released;
  return pkv::ok();
}

pkv_status_t pkv_bm_block_tables(const pkv_bm_t* bm, const int64_t* seq_ids, int n,
                                 int max_blocks_per_seq, int32_t* table_out, int32_t* lens_out) {
  if (!bm || n < 0 || max_blocks_per_seq < 0 || (n > 0 && (!seq_ids || !table_out || !lens_out)))
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_block_tables: bad argument");
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end())
      return pkv::fail(PKV_ERR_INVALID_ARG, "bm_block_tables: unknown sequence %lld", (long long)seq_ids[i]);
    if (int64_t(it->second.table.size()) > max_blocks_per_seq)
      return pkv::fail(PKV_ERR_INVALID_ARG, "bm_block_tables: sequence %lld has %zu blocks > %d",
                       (long long)seq_ids[i], it->second.table.size(), max_blocks_per_seq);
    if (it->second.len > INT32_MAX) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_block_tables: length overflows int32");
  }
  for (int i = 0; i < n; ++i) {
    const auto& s = bm->seqs.find(seq_ids[i])->second;
    int32_t* row = table_out + size_t(i) * size_t(max_blocks_per_seq);
    std::copy(s.table.begin(), s.table.end(), row);
    std::fill(row + s.table.size(), row + max_blocks_per_seq, -1);
    lens_out[i] = int32_t(s.len);
  }
  return pkv::ok();
}

pkv_status_t pkv_bm_refcount(const pkv_bm_t* bm, int block, int32_t* out) {
  if (!bm || !out || block < 0 || block >= bm->num_blocks)
    return pkv::fail(PKV_ERR_INVALID_ARG, "bm_refcount: bad argument");
  *out = bm->refcount[block];
  return pkv::ok();
}

pkv_status_t pkv_bm_seq_len(const pkv_bm_t* bm, int64_t seq_id, int64_t* out) {
  if (!bm || !out) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_seq_len: bad argument");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return pkv::fail(PKV_ERR_INVALID_ARG, "bm_seq_len: unknown sequence %lld", (long long)seq_id);
  *out = it->second.len;
  return pkv::ok();
}

int pkv_bm_num_free(const pkv_bm_t* bm) { return bm ? int(bm->free_stack.size()) : -1; }

int pkv_bm_num_seqs(const pkv_bm_t* bm) { return bm ? int(bm->seqs.size()) : -1; }

int pkv_bm_free_stack(const pkv_bm_t* bm, int32_t* out, int capacity) {
  if (!bm) return -1;
  const int n = int(bm->free_stack.size());
  if (out) std::copy(bm->free_stack.begin(), bm->free_stack.begin() + std::min(n, std::max(capacity, 0)), out);
  return n;
}

}  // extern "C"
