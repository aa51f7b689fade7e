// Host block allocator: FIFO free list, per-block reference counts, prefix
// sharing by fork and copy-on-write on append.  The cache lives in small
// fixed-size blocks allocated as a sequence grows, with a per-sequence table
// from positions to blocks, and sequences that share a prefix share its
// blocks ("Serving", section 23.4 Paged Attention); a write into a shared
// block copies it first ("Paged Attention: Managing the KV Cache Like Virtual
// Memory", inference-serving tag page).  The policy is spelled out in pa.h.
#include <deque>
#include <unordered_map>
#include <vector>

#include "pa.h"

struct pa_alloc {
  struct Seq {
    std::vector<int32_t> table;
    long long len = 0;
  };
  int num_blocks = 0;
  int block_size = 0;
  std::deque<int32_t> free_list;
  std::vector<int32_t> refcount;
  std::unordered_map<int, Seq> seqs;

  int take() {  // caller checked free_list is non-empty
    int32_t b = free_list.front();
    free_list.pop_front();
    refcount[b] = 1;
    return b;
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
};

extern "C" {

int pa_alloc_create(int num_blocks, int block_size, const int32_t* free_order, pa_alloc_t* out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID;
  *out = nullptr;
  pa_alloc* a = new pa_alloc();
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->refcount.assign(num_blocks, 0);
  if (free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int k = 0; k < num_blocks; ++k) {
      int32_t b = free_order[k];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete a;
        return PA_ERR_INVALID;  // not a permutation
      }
      seen[b] = 1;
      a->free_list.push_back(b);
    }
  } else {
    for (int b = 0; b < num_blocks; ++b) a->free_list.push_back(b);
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
  return a->append(seq, slot, cow_src, cow_dst);
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
    if (--a->refcount[b] == 0) a->free_list.push_back(b);
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

int pa_alloc_num_free(pa_alloc_t a) {
  if (!a) return PA_ERR_INVALID;
  return static_cast<int>(a->free_list.size());
}

}  // extern "C"
