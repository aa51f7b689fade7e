// Host block allocator: FIFO free list, per-block reference counts, prefix
// sharing by fork and copy-on-write on append.  The cache lives in small
// fixed-size blocks allocated as a sequence grows, with a per-sequence table
// from positions to blocks, and sequences that share a prefix share its
// blocks ("Serving", section 23.4 Paged Attention); a write into a shared
// block copies it first ("Paged Attention: Managing the KV Cache Like Virtual
// Memory", inference-serving tag page).  Full blocks can also be found again
// by the chained hash of their tokens (prefix caching by block hashes, same
// page; hash chains, posts on the pagedattention tag).  The policy is spelled
// out in pa.h.
#include <algorithm>
#include <array>
#include <cstring>
#include <list>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

// FNV-1a, 64-bit: offset basis 14695981039346656037, prime 1099511628211.
uint64_t fnv1a64(const unsigned char* p, size_t n) {
  uint64_t h = 14695981039346656037ull;
  for (size_t k = 0; k < n; ++k) {
    h ^= p[k];
    h *= 1099511628211ull;
  }
  return h;
}

// Chained hash of a full block: the parent's hash as 8 little-endian bytes,
// then the token ids as 4-byte little-endian integers.
uint64_t block_hash(uint64_t parent, const int32_t* tok, int n) {
  std::vector<unsigned char> buf(8 + 4 * static_cast<size_t>(n));
  for (int k = 0; k < 8; ++k) buf[k] = static_cast<unsigned char>(parent >> (8 * k));
  for (int t = 0; t < n; ++t) {
    const uint32_t v = static_cast<uint32_t>(tok[t]);
    for (int k = 0; k < 4; ++k) buf[8 + 4 * t + k] = static_cast<unsigned char>(v >> (8 * k));
  }
  return fnv1a64(buf.data(), buf.size());
}

}  // namespace

struct pa_alloc {
  struct Seq {
    std::vector<int32_t> table;
    long long len = 0;
    bool tracked = true;            // every token so far appended with its id
    std::vector<int32_t> tokens;    // the ids (while tracked)
    std::vector<uint64_t> chain;    // hashes of its full blocks (while tracked)
  };
  struct Entry {
    int32_t block;
    uint64_t parent;
    std::vector<int32_t> tokens;
  };
  int num_blocks = 0;
  int block_size = 0;
  std::list<int32_t> free_list;  // FIFO; cached blocks can leave from the middle
  std::vector<std::list<int32_t>::iterator> free_pos;
  std::vector<char> on_free;
  std::vector<int32_t> refcount;
  std::unordered_map<int, Seq> seqs;
  std::unordered_map<uint64_t, Entry> index;  // hash -> cached full block
  std::vector<uint64_t> key_of;               // block -> its hash while indexed
  std::vector<char> indexed;
  long long queries = 0, hits = 0;

  void push_free(int32_t b) {
    free_list.push_back(b);
    free_pos[b] = std::prev(free_list.end());
    on_free[b] = 1;
  }
  int take() {  // caller checked free_list is non-empty
    int32_t b = free_list.front();
    free_list.pop_front();
    on_free[b] = 0;
    if (indexed[b]) {  // the block is reused: its cached contents go away
      index.erase(key_of[b]);
      indexed[b] = 0;
    }
    refcount[b] = 1;
    return b;
  }
  void share(int32_t b) {
    if (refcount[b] == 0 && on_free[b]) {
      free_list.erase(free_pos[b]);
      on_free[b] = 0;
    }
    refcount[b] += 1;
  }
  // the block that just became full (block k of s) joins the index
  void register_full(Seq& s, int k) {
    const uint64_t parent = k > 0 ? s.chain[k - 1] : 0;
    const int32_t* tok = s.tokens.data() + static_cast<size_t>(k) * block_size;
    const uint64_t h = block_hash(parent, tok, block_size);
    s.chain.push_back(h);
    const int32_t b = s.table[k];
    if (!index.count(h) && !indexed[b]) {
      index.emplace(h, Entry{b, parent, std::vector<int32_t>(tok, tok + block_size)});
      key_of[b] = h;
      indexed[b] = 1;
    }
  }

  int append(int seq, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
    auto it = seqs.find(seq);
    if (it == seqs.end()) return PA_ERR_INVALID;
    Seq& s = it->second;
    const long long pos = s.len;
    int32_t cs = -1, cd = -1;
    if (pos % block_size == 0) {
      if (free_list.empty()) return PA_ERR_OOM;
      s.table.push_back(take());
    } else {
      int32_t last = s.table.back();
      if (refcount[last] > 1) {
        if (free_list.empty()) return PA_ERR_OOM;
        int32_t b = take();
        refcount[last] -= 1;
        s.table.back() = b;
        cs = last;
        cd = b;
      }
    }
    s.len = pos + 1;
    if (slot) *slot = static_cast<int64_t>(s.table[pos / block_size]) * block_size + pos % block_size;
    if (cow_src) *cow_src = cs;
    if (cow_dst) *cow_dst = cd;
    return PA_OK;
  }

  int append_token(int seq, int32_t token, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
    int st = append(seq, slot, cow_src, cow_dst);
    if (st != PA_OK) return st;
    Seq& s = seqs.find(seq)->second;
    if (s.tracked) {
      s.tokens.push_back(token);
      if (s.tokens.size() % block_size == 0) register_full(s, static_cast<int>(s.tokens.size() / block_size) - 1);
    }
    return PA_OK;
  }
};

extern "C" {

int pa_alloc_create(int num_blocks, int block_size, const int32_t* free_order, pa_alloc_t* out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID;
  *out = nullptr;
  pa_alloc* a = new pa_alloc();
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->refcount.assign(num_blocks, 0);
  a->free_pos.resize(num_blocks);
  a->on_free.assign(num_blocks, 0);
  a->key_of.assign(num_blocks, 0);
  a->indexed.assign(num_blocks, 0);
  if (free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int k = 0; k < num_blocks; ++k) {
      int32_t b = free_order[k];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete a;
        return PA_ERR_INVALID;  // not a permutation
      }
      seen[b] = 1;
      a->push_free(b);
    }
  } else {
    for (int b = 0; b < num_blocks; ++b) a->push_free(b);
  }
  *out = a;
  return PA_OK;
}

int pa_alloc_destroy(pa_alloc_t a) {
  delete a;
  return PA_OK;
}

int pa_alloc_seq_add(pa_alloc_t a, int seq_id) {
  if (!a || seq_id < 0 || a->seqs.count(seq_id)) return PA_ERR_INVALID;
  a->seqs.emplace(seq_id, pa_alloc::Seq());
  return PA_OK;
}

int pa_alloc_fork(pa_alloc_t a, int parent, int child) {
  if (!a || child < 0) return PA_ERR_INVALID;
  auto it = a->seqs.find(parent);
  if (it == a->seqs.end() || a->seqs.count(child)) return PA_ERR_INVALID;
  pa_alloc::Seq copy = it->second;
  for (int32_t b : copy.table) a->refcount[b] += 1;
  a->seqs.emplace(child, std::move(copy));
  return PA_OK;
}

int pa_alloc_append_slot(pa_alloc_t a, int seq, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
  if (!a) return PA_ERR_INVALID;
  int st = a->append(seq, slot, cow_src, cow_dst);
  if (st == PA_OK) {
    auto& s = a->seqs.find(seq)->second;
    s.tracked = false;  // its token ids are unknown from here on
    s.tokens.clear();
    s.chain.clear();
  }
  return st;
}

int pa_alloc_append_token(pa_alloc_t a, int seq, int32_t token, int64_t* slot, int32_t* cow_src,
                          int32_t* cow_dst) {
  if (!a) return PA_ERR_INVALID;
  return a->append_token(seq, token, slot, cow_src, cow_dst);
}

int pa_alloc_seq_add_cached(pa_alloc_t a, int seq_id, const int32_t* tokens, int n_tokens, int* n_cached) {
  if (!a || seq_id < 0 || n_tokens < 0 || (n_tokens > 0 && !tokens) || a->seqs.count(seq_id))
    return PA_ERR_INVALID;
  pa_alloc::Seq s;
  uint64_t parent = 0;
  const int bs = a->block_size;
  for (int k = 0; k + 1 <= n_tokens / bs; ++k) {
    const int32_t* tok = tokens + static_cast<size_t>(k) * bs;
    const uint64_t h = block_hash(parent, tok, bs);
    a->queries += 1;
    auto it = a->index.find(h);
    if (it == a->index.end() || it->second.parent != parent ||
        std::memcmp(it->second.tokens.data(), tok, sizeof(int32_t) * bs) != 0)
      break;
    a->hits += 1;
    a->share(it->second.block);
    s.table.push_back(it->second.block);
    s.tokens.insert(s.tokens.end(), tok, tok + bs);
    s.chain.push_back(h);
    s.len += bs;
    parent = h;
  }
  if (n_cached) *n_cached = static_cast<int>(s.len);
  a->seqs.emplace(seq_id, std::move(s));
  return PA_OK;
}

int pa_alloc_block_hash(pa_alloc_t a, int block, uint64_t* hash) {
  if (!a || block < 0 || block >= a->num_blocks) return PA_ERR_INVALID;
  if (!a->indexed[block]) return 0;
  if (hash) *hash = a->key_of[block];
  return 1;
}

int pa_alloc_prefix_stats(pa_alloc_t a, int64_t* queries, int64_t* hits, int64_t* cached_blocks) {
  if (!a) return PA_ERR_INVALID;
  if (queries) *queries = a->queries;
  if (hits) *hits = a->hits;
  if (cached_blocks) *cached_blocks = static_cast<int64_t>(a->index.size());
  return PA_OK;
}

int pa_alloc_extend(pa_alloc_t a, int seq, int n, int64_t* slots, int32_t* cow_src,
                    int32_t* cow_dst, int* n_done) {
  if (!a || n < 0) return PA_ERR_INVALID;
  if (cow_src) *cow_src = -1;
  if (cow_dst) *cow_dst = -1;
  int k = 0;
  int st = PA_OK;
  for (; k < n; ++k) {
    int32_t cs = -1, cd = -1;
    st = a->append(seq, slots ? slots + k : nullptr, &cs, &cd);
    if (st != PA_OK) break;
    if (cs >= 0) {
      if (cow_src) *cow_src = cs;
      if (cow_dst) *cow_dst = cd;
    }
  }
  if (n_done) *n_done = k;
  return st;
}

int pa_alloc_seq_free(pa_alloc_t a, int seq) {
  if (!a) return PA_ERR_INVALID;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_INVALID;
  for (int32_t b : it->second.table) {
    if (--a->refcount[b] == 0) a->push_free(b);
  }
  a->seqs.erase(it);
  return PA_OK;
}

int pa_alloc_table(pa_alloc_t a, int seq, int32_t* out, int cap, int* n_blocks) {
  if (!a || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_INVALID;
  const auto& t = it->second.table;
  int n = static_cast<int>(t.size());
  for (int k = 0; k < n && k < cap; ++k) out[k] = t[k];
  if (n_blocks) *n_blocks = n;
  return PA_OK;
}

int pa_alloc_seq_len(pa_alloc_t a, int seq) {
  if (!a) return PA_ERR_INVALID;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_INVALID;
  return static_cast<int>(it->second.len);
}

int pa_alloc_refcount(pa_alloc_t a, int block) {
  if (!a || block < 0 || block >= a->num_blocks) return PA_ERR_INVALID;
  return a->refcount[block];
}

int pa_cascade_groups(const int32_t* tables, int num_seqs, int max_blocks, const int32_t* seq_lens,
                      int max_members, int32_t* group_start, int32_t* members, int32_t* prefix_blocks,
                      int* n_groups) {
  if (!tables || !seq_lens || !group_start || !members || !prefix_blocks || !n_groups || num_seqs < 0 ||
      max_blocks <= 0 || max_members < 1)
    return PA_ERR_INVALID;
  // sequences by first block, in order of first appearance
  std::vector<int32_t> keys;
  std::unordered_map<int32_t, std::vector<int>> by_first;
  for (int i = 0; i < num_seqs; ++i) {
    if (seq_lens[i] < 16) continue;  // no full block to share
    const int32_t b = tables[static_cast<long long>(i) * max_blocks];
    auto it = by_first.find(b);
    if (it == by_first.end()) {
      keys.push_back(b);
      by_first.emplace(b, std::vector<int>{i});
    } else {
      it->second.push_back(i);
    }
  }
  int ng = 0, nm = 0;
  group_start[0] = 0;
  for (int32_t b : keys) {
    const std::vector<int>& all = by_first[b];
    for (size_t c0 = 0; c0 < all.size(); c0 += static_cast<size_t>(max_members)) {
      const size_t c1 = std::min(all.size(), c0 + static_cast<size_t>(max_members));
      if (c1 - c0 < 2) continue;
      int lim = max_blocks;
      for (size_t k = c0; k < c1; ++k) lim = std::min(lim, seq_lens[all[k]] / 16);
      const int32_t* t0 = tables + static_cast<long long>(all[c0]) * max_blocks;
      int P = 0;
      while (P < lim) {
        bool same = true;
        for (size_t k = c0 + 1; k < c1 && same; ++k)
          same = tables[static_cast<long long>(all[k]) * max_blocks + P] == t0[P];
        if (!same) break;
        ++P;
      }
      if (P < 1) continue;
      for (size_t k = c0; k < c1; ++k) members[nm++] = all[k];
      prefix_blocks[ng] = P;
      group_start[++ng] = nm;
    }
  }
  *n_groups = ng;
  return PA_OK;
}

int pa_alloc_num_free(pa_alloc_t a) {
  if (!a) return PA_ERR_INVALID;
  return static_cast<int>(a->free_list.size());
}

}  // extern "C"
