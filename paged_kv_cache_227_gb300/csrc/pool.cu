// Pool lifetime, block copy for copy-on-write, the device error word and
// status strings.
#include <cudaTypedefs.h>

#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace pa {

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point so
// the library needs no link-time dependency on the driver library.
static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tile view of the K|V allocation: dims {64 elements, rows, 2 halves, K|V}
// with byte strides {256 (row), 128 (half), bytes of one array}; the box
// {64, 16, 2, 2} is one (block, head) tile of K followed by the same tile of
// V, written to shared memory as [K|V][half][row][128 bytes] with the 128-byte
// swizzle.
static bool encode_pool_map(CUtensorMap* map, void* base, long long rows, size_t array_bytes,
                            int dtype) {
  auto fn = encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim / 2), static_cast<cuuint64_t>(rows), 2, 2};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(kRowBytes), static_cast<cuuint64_t>(kRowBytes / 2),
                           static_cast<cuuint64_t>(array_bytes)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(kHeadDim / 2), static_cast<cuuint32_t>(kBlock), 2, 2};
  cuuint32_t elem[4] = {1, 1, 1, 1};
  CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  4, base, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count(int device) {
  static std::mutex mu;
  static std::vector<int> cache;
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0) return 0;
  if (static_cast<size_t>(device) >= cache.size()) cache.resize(device + 1, 0);
  if (cache[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      (void)cudaGetLastError();  // a failed query leaves no pending error behind
      return 0;
    }
    cache[device] = n;
  }
  return cache[device];
}

static long long g_wait_limit_ns = 2000000000ll;  // 2 s
long long wait_limit_ns() { return g_wait_limit_ns; }

// Whole-block copy: one CTA per (pair, K|V); 16-byte vectors.
__global__ void copy_blocks_kernel(uint4* k, uint4* v, const int32_t* src, const int32_t* dst,
                                   int n, long long num_blocks, int vec_per_block,
                                   long long* err) {
  int j = blockIdx.x >> 1;
  if (j >= n) return;
  uint4* base = (blockIdx.x & 1) ? v : k;
  long long s = src[j], d = dst[j];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0) record_error(err, PA_ERR_DEVICE_CHECK, s < 0 || s >= num_blocks ? s : d);
    return;
  }
  const uint4* from = base + s * vec_per_block;
  uint4* to = base + d * vec_per_block;
  for (int x = threadIdx.x; x < vec_per_block; x += blockDim.x) to[x] = from[x];
}

}  // namespace pa

using namespace pa;

extern "C" {

size_t pa_pool_bytes(int num_blocks, int block_size, int n_kv_heads, int d_head, int dtype) {
  if (num_blocks <= 0 || n_kv_heads <= 0 || block_size != kBlock || d_head != kHeadDim) return 0;
  if (dtype != PA_FP16 && dtype != PA_BF16) return 0;
  return static_cast<size_t>(num_blocks) * n_kv_heads * kBlock * kHeadDim * 2;
}

int pa_pool_create(int num_blocks, int block_size, int n_kv_heads, int d_head, int dtype,
                   pa_pool_t* out) {
  if (!out || num_blocks <= 0 || n_kv_heads <= 0) return PA_ERR_INVALID;
  if (block_size != kBlock || d_head != kHeadDim) return PA_ERR_UNSUPPORTED;
  if (dtype != PA_FP16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  // kernels address token rows (block * heads + head) * 16 with 32-bit ints
  if (static_cast<long long>(num_blocks) * n_kv_heads * kBlock > 0x7fffffffll) return PA_ERR_UNSUPPORTED;
  *out = nullptr;
  pa_pool* p = new pa_pool();
  p->num_blocks = num_blocks;
  p->n_kv_heads = n_kv_heads;
  p->dtype = dtype;
  p->bytes = pa_pool_bytes(num_blocks, block_size, n_kv_heads, d_head, dtype);
  if (cudaGetDevice(&p->device) != cudaSuccess) { delete p; return PA_ERR_CUDA; }
  void* kv = nullptr;
  if (cudaMalloc(&kv, 2 * p->bytes) != cudaSuccess || cudaMalloc(&p->err, 2 * sizeof(long long)) != cudaSuccess) {
    cudaFree(kv); cudaFree(p->err);
    cudaGetLastError();
    delete p;
    return PA_ERR_OOM;
  }
  p->k = kv;
  p->v = static_cast<char*>(kv) + p->bytes;
  const long long rows = static_cast<long long>(num_blocks) * n_kv_heads * kBlock;
  if (!encode_pool_map(&p->tmap_kv, kv, rows, p->bytes, dtype)) {
    cudaFree(kv); cudaFree(p->err);
    delete p;
    return PA_ERR_CUDA;
  }
  if (cudaMemset(kv, 0, 2 * p->bytes) != cudaSuccess ||
      cudaMemset(p->err, 0, 2 * sizeof(long long)) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(kv); cudaFree(p->err);
    delete p;
    return PA_ERR_CUDA;
  }
  *out = p;
  return PA_OK;
}

int pa_pool_destroy(pa_pool_t p) {
  if (!p) return PA_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(p->device);
  cudaDeviceSynchronize();
  cudaFree(p->k);  // K and V share one allocation
  cudaFree(p->err);
  cudaSetDevice(prev);
  delete p;
  return PA_OK;
}

int pa_pool_info(pa_pool_t p, void** k_pool, void** v_pool, size_t* bytes_per_pool) {
  if (!p) return PA_ERR_INVALID;
  if (k_pool) *k_pool = p->k;
  if (v_pool) *v_pool = p->v;
  if (bytes_per_pool) *bytes_per_pool = p->bytes;
  return PA_OK;
}

int pa_pool_shape(pa_pool_t p, int* num_blocks, int* n_kv_heads, int* d_head, int* dtype) {
  if (!p) return PA_ERR_INVALID;
  if (num_blocks) *num_blocks = p->num_blocks;
  if (n_kv_heads) *n_kv_heads = p->n_kv_heads;
  if (d_head) *d_head = kHeadDim;
  if (dtype) *dtype = p->dtype;
  return PA_OK;
}

int pa_copy_blocks(pa_pool_t p, const int32_t* src, const int32_t* dst, int n, void* stream) {
  if (!p || n < 0 || (n > 0 && (!src || !dst))) return PA_ERR_INVALID;
  if (n == 0) return PA_OK;
  if (!on_pool_device(p)) return PA_ERR_INVALID;
  int vec_per_block = p->n_kv_heads * kTileBytes / 16;
  copy_blocks_kernel<<<2 * n, 256, 0, as_stream(stream)>>>(
      static_cast<uint4*>(p->k), static_cast<uint4*>(p->v), src, dst, n, p->num_blocks,
      vec_per_block, p->err);
  return cuda_status(cudaGetLastError());
}

int pa_check(pa_pool_t p, void* stream, int64_t* detail) {
  if (!p) return PA_ERR_INVALID;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return PA_ERR_CUDA;
  long long host[2] = {0, 0};
  if (cudaMemcpy(host, p->err, sizeof host, cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  if (host[0] != 0) {
    const long long zero[2] = {0, 0};
    if (cudaMemcpy(p->err, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return PA_ERR_CUDA;
  }
  if (detail) *detail = host[1];
  return static_cast<int>(host[0]);
}

const char* pa_strerror(int code) {
  switch (code) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported size or type (block size 16, head dim 128, group <= 8)";
    case PA_ERR_OOM: return "out of memory (device allocation or allocator free list)";
    case PA_ERR_CUDA: return "CUDA runtime or launch failure";
    case PA_ERR_DEVICE_CHECK: return "a kernel met an out-of-range block id or slot and skipped it";
    case PA_ERR_TIMEOUT: return "a bounded in-kernel wait ran out";
    case PA_ERR_SCRATCH_LIMIT: return "the call needs more workspace than the library's static scratch holds";
    default: return "unknown status";
  }
}

}  // extern "C"
