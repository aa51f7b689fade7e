// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

// One pool: K and V arrays [num_blocks][n_kv_heads][16][128] plus a device
// error word.  Fixed-size physical blocks as in "Serving" 23.4.  K and V sit
// in one allocation (V right after K) so that one TMA tensor map covers both:
// it views the pair as a 4-D tensor {64 elements, token rows, 2 row halves,
// K|V} and loads a whole (block, head) tile of K and of V - 16 rows x 128
// elements each - as one box, with the 128-byte swizzle.
struct pa_pool {
  CUtensorMap tmap_kv;  // CUtensorMap carries its own 64-byte alignment
  int num_blocks;
  int n_kv_heads;
  int dtype;          // PA_FP16 | PA_BF16
  int device;
  void* k;            // device
  void* v;            // device
  size_t bytes;       // bytes of one of k / v
  long long* err;     // device: [0] = status code, [1] = detail
};

namespace pa {

constexpr int kBlock = PA_BLOCK_SIZE;     // tokens per block
constexpr int kHeadDim = PA_HEAD_DIM;     // elements per K/V row
constexpr int kRowBytes = kHeadDim * 2;   // one 16-bit row: 256 B
constexpr int kTileBytes = kBlock * kRowBytes;  // one (block, head) tile: 4 KiB

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Maps a CUDA error to a status (and clears sticky-free launch errors).
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

// Records the first device-side error: code in err[0] (0 -> code), detail in
// err[1].  Later errors are dropped.
__device__ inline void record_error(long long* err, long long code, long long detail) {
  if (atomicCAS(reinterpret_cast<unsigned long long*>(err), 0ull,
                static_cast<unsigned long long>(code)) == 0ull) {
    atomicExch(reinterpret_cast<unsigned long long*>(err + 1),
               static_cast<unsigned long long>(detail));
  }
}

// Number of SMs of the current device (cached per device).
int sm_count(int device);

// Entry check of every call that launches kernels: the current device must
// be the pool's (kernels launch on the current device and address the pool's
// memory, so a call from another device is refused before anything is
// launched).  It also clears a pending non-sticky error of an earlier runtime
// call, so that the launch checks that follow report this call's launches.
inline bool on_pool_device(const pa_pool* p) {
  (void)cudaGetLastError();
  int cur = -1;
  return cudaGetDevice(&cur) == cudaSuccess && cur == p->device;
}

// Wait limit for bounded in-kernel waits, in nanoseconds.
long long wait_limit_ns();

// The fused step's cache write (one new token per sequence at position
// L_i - 1), launched on `stream`; the decode follows as its programmatic
// dependent.
int launch_append_tail(void* k_pool, void* v_pool, int n_kv_heads, long long num_blocks, long long* err,
                       int device, const void* k_new, const void* v_new, const int32_t* tables,
                       int max_blocks, const int32_t* seq_lens, int B, cudaStream_t stream);

}  // namespace pa
