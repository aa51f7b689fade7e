// Cache write: token t's K/V rows go to slot_mapping[t] = block*16 + offset.
// A sequence's cache grows a token at a time into fixed-size blocks
// ("Serving" 23.4 Paged Attention).
#include "pa_internal.h"

namespace pa {

// One thread per 16-byte vector of a row; a row is 16 vectors, so a warp
// writes two full 256-byte rows (coalesced).  Vector x of the launch:
//   t = token, kv = 0 (K) / 1 (V), h = kv head, c = 16-byte chunk.
__global__ void append_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                              const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                              const int64_t* __restrict__ slot_mapping, long long n_vec,
                              int n_kv_heads, long long num_slots, long long* err) {
  const int per_tok = n_kv_heads * 32;
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < n_vec;
       x += (long long)gridDim.x * blockDim.x) {
    long long t = x / per_tok;
    int rem = static_cast<int>(x - t * per_tok);
    int kv = rem / (n_kv_heads * 16);
    int hc = rem - kv * n_kv_heads * 16;   // h*16 + c
    int h = hc >> 4, c = hc & 15;
    long long slot = slot_mapping[t];
    if (slot < 0) continue;                 // padding token
    if (slot >= num_slots) {
      record_error(err, PA_ERR_DEVICE_CHECK, slot);
      continue;
    }
    long long blk = slot >> 4, off = slot & 15;
    long long dst = ((blk * n_kv_heads + h) * kBlock + off) * (kRowBytes / 16) + c;
    long long src = (t * n_kv_heads + h) * (kRowBytes / 16) + c;
    if (kv == 0)
      k_pool[dst] = k_new[src];
    else
      v_pool[dst] = v_new[src];
  }
}

// The fused step's cache write: the new token of every sequence sits at
// position L_i - 1, in slot table[i][(L_i - 1) / 16] * 16 + (L_i - 1) % 16.
// The decode that follows is launched as this kernel's programmatic
// dependent, so it may start right away (griddepcontrol.launch_dependents)
// and waits for this grid only before it reads a tile holding a new token.
// Lengths out of range are left to the decode to report.
__global__ void append_tail_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                   const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                   const int32_t* __restrict__ tables, int max_blocks,
                                   const int32_t* __restrict__ seq_lens, int B, int n_kv_heads,
                                   long long num_blocks, long long* err) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int per_seq = n_kv_heads * 32;
  const long long n_vec = static_cast<long long>(B) * per_seq;
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < n_vec;
       x += (long long)gridDim.x * blockDim.x) {
    const int i = static_cast<int>(x / per_seq);
    const int rem = static_cast<int>(x - static_cast<long long>(i) * per_seq);
    const int kv = rem / (n_kv_heads * 16);
    const int hc = rem - kv * n_kv_heads * 16;  // h*16 + c
    const int h = hc >> 4, c = hc & 15;
    const int L = seq_lens[i];
    if (L <= 0 || L > max_blocks * kBlock) continue;
    const int pos = L - 1;
    const long long blk = tables[static_cast<long long>(i) * max_blocks + pos / kBlock];
    if (blk < 0 || blk >= num_blocks) {
      record_error(err, PA_ERR_DEVICE_CHECK, blk);
      continue;
    }
    const long long dst = ((blk * n_kv_heads + h) * kBlock + (pos & (kBlock - 1))) * (kRowBytes / 16) + c;
    const long long src = (static_cast<long long>(i) * n_kv_heads + h) * (kRowBytes / 16) + c;
    if (kv == 0)
      k_pool[dst] = k_new[src];
    else
      v_pool[dst] = v_new[src];
  }
}

int launch_append_tail(void* k_pool, void* v_pool, int n_kv_heads, long long num_blocks, long long* err,
                       int device, const void* k_new, const void* v_new, const int32_t* tables,
                       int max_blocks, const int32_t* seq_lens, int B, cudaStream_t stream) {
  const long long n_vec = static_cast<long long>(B) * n_kv_heads * 32;
  const int threads = 256;
  const long long want = (n_vec + threads - 1) / threads;
  const long long cap = static_cast<long long>(sm_count(device)) * 2;
  const int blocks = static_cast<int>(want < cap ? (want < 1 ? 1 : want) : cap);
  append_tail_kernel<<<blocks, threads, 0, stream>>>(
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), static_cast<const uint4*>(k_new),
      static_cast<const uint4*>(v_new), tables, max_blocks, seq_lens, B, n_kv_heads, num_blocks, err);
  return cuda_status(cudaGetLastError());
}

}  // namespace pa

using namespace pa;

extern "C" int pa_cache_append(pa_pool_t p, const void* k_new, const void* v_new,
                               const int64_t* slot_mapping, int n_tok, void* stream) {
  if (!p || n_tok < 0) return PA_ERR_INVALID;
  if (n_tok == 0) return PA_OK;
  if (!on_pool_device(p)) return PA_ERR_INVALID;
  if (!k_new || !v_new || !slot_mapping) return PA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return PA_ERR_INVALID;  // rows are moved as 16-byte vectors
  long long n_vec = static_cast<long long>(n_tok) * p->n_kv_heads * 32;
  int threads = 256;
  long long want = (n_vec + threads - 1) / threads;
  int cap = sm_count(p->device) * 8;
  int blocks = static_cast<int>(want < cap ? want : cap);
  if (blocks < 1) blocks = 1;
  append_kernel<<<blocks, threads, 0, as_stream(stream)>>>(
      static_cast<uint4*>(p->k), static_cast<uint4*>(p->v), static_cast<const uint4*>(k_new),
      static_cast<const uint4*>(v_new), slot_mapping, n_vec, p->n_kv_heads,
      static_cast<long long>(p->num_blocks) * kBlock, p->err);
  return cuda_status(cudaGetLastError());
}
