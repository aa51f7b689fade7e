// Paged decode attention for sm_103a.
//
// One query token per sequence attends over its cache, which sits in
// fixed-size 16-token blocks found through a per-sequence block table
// ("Serving", section 23.4 Paged Attention).  Decode reads the whole cache
// for one token per sequence, so it is bound by HBM bandwidth ("Serving",
// section 23.2 Prefill and Decode); the design reads every K/V byte exactly
// once, keeps enough bytes in flight to saturate HBM3e, and keeps the SM's
// instruction issue far below the memory time.
//
// Work decomposition.  A segment is one (sequence i, kv head h) pair: its
// nb_i = ceil(L_i/16) tiles of 16 tokens x 128 dims (4 KiB each for K and
// for V).  The whole grouped-query head group (G = Hq/Hkv query heads) of the
// segment is handled by the same CTA, so a tile is fetched once and used by G
// heads.  A CTA is persistent and processes a list of pieces (a contiguous
// range of a segment's tiles) given by one of three schedules:
//   SEGMENT    whole segments, strided over CTAs (no workspace);
//   LEAN       the concatenated tile stream of all segments cut into equal
//              per-CTA ranges (even load for any length mix); a segment cut
//              by a range boundary leaves partial results;
//   PARTITION  fixed partitions of `partition_blocks` tiles per segment.
// A piece that does not cover its whole segment writes a partial record
// (running max m, sum l, unnormalised o, fp32) and bumps the segment's
// counter; the CTA that completes the count merges the records by
// log-sum-exp and writes the output, then resets the counter to zero.
//
// CTA layout: 4 consumer warps + 1 producer warp, two CTAs per SM.  The
// producer walks the block table and streams each (block, head) K and V tile
// into a shared-memory ring of S = 12 stages (8 for G > 4) with TMA tensor
// loads (two 16-row x 128-byte boxes per tile, 128-byte swizzle), completion
// tracked by mbarriers.  Tile n of the CTA's stream goes to stage n % S and
// is consumed by warp n % 4, which runs the online softmax over its own
// tiles; the warps' states are merged at the end of each piece.
//
// Per tile a consumer warp runs two small tensor-core contractions with
// mma.sync m16n8k16 (fp32 accumulate) whose 8 columns are the query heads of
// the group (G <= 8, the rest zero):
//   S^T[t][g] = K[t] . q_g        M = 16 tokens, 8 k-steps of 16 dims
//   O^T[:][g] += V^T P^T          8 m-tiles of 16 dims, k = 16 tokens
// The score fragments are packed and transposed in registers (movmatrix) to
// become the second product's B operand, so P never leaves registers.  P is
// split into a 16-bit high part and the rounded remainder, and both are
// multiplied, which keeps the weights accurate to ~2^-17.  That is 24 MMAs
// per tile; the per-SM rate of this instruction is what bounds the kernel
// once memory keeps up.  Softmax runs in fp32 in the log2 domain with
// a lazily moved running max (rescale only when a new max exceeds the old by
// 2^8).  Positions t >= L are masked by select on S and their V rows are
// zeroed in shared memory, so padding or stale slots (even NaN) never reach
// the output.  ldmatrix reads the swizzled tiles without bank conflicts.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstddef>
#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace pa {

constexpr int kMaxSplitSeqs = 4096;  // sequences per split launch (prefix in shared memory)
constexpr int kMaxCtasPerSm = 4;
constexpr int kLeanMinBlocks = 8;    // smallest LEAN range per CTA
constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;    // log2 units

enum { SCHED_SEGMENT = 0, SCHED_LEAN = 1, SCHED_PARTITION = 2 };

// Compile-time shape of the kernel: 4 consumer warps; 12 ring stages for
// G <= 4 and 8 for larger groups (whose merge buffer is bigger), so that two
// CTAs fit in an SM's shared memory either way.
template <int G>
struct Shape {
  static constexpr int NW = 4;                          // consumer warps (+1 producer)
  static constexpr int kStages = G <= 4 ? 3 * NW : 2 * NW;
  static constexpr int kThreads = (NW + 1) * 32;
};

struct Params {
  CUtensorMap tmap_k;       // token-row views of the pools (see pa_pool)
  CUtensorMap tmap_v;
  const uint16_t* q;        // [B][Hq][128]
  const uint16_t* k_pool;   // [N][Hkv][16][128]
  const uint16_t* v_pool;
  const uint16_t* k_new;    // [B][Hkv][128], fused append only
  const uint16_t* v_new;
  const int32_t* tables;    // [B][max_blocks]
  const int32_t* seq_lens;  // [B]
  void* out;                // [B][Hq][128]
  float* ws;                // partial records
  int* counters;            // [B][Hkv] pieces finished per segment (zero between calls)
  long long* err;
  long long num_blocks;
  int max_blocks;
  int B, Hq, Hkv;
  int out_dtype;
  float qscale;             // scale * log2(e)
  int sched;
  int partition_blocks;     // PARTITION: tiles per partition
  int lean_grid;            // LEAN: number of CTAs the ranges are cut for
  long long wait_limit_ns;
};

// Partial record of one piece: o[G][128], then m[g] at G*128+g and l[g] at
// G*128+64+g (fp32; m in log2 units of the scaled scores).
__host__ __device__ constexpr int record_floats(int G) { return (G + 1) * 128; }

// ---------------------------------------------------------------------------
// PTX helpers: mbarrier, bulk copy, timer, named barriers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
template <int NT>
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}
template <int NT>
__device__ __forceinline__ int consumers_sync_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 2, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "n"(NT)
      : "memory");
  return r;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or
// the wait ran out (then it records PA_ERR_TIMEOUT and raises the abort flag).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           long long limit_ns, long long* err, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      record_error(err, PA_ERR_TIMEOUT, site);
      return false;
    }
  }
}


// TMA tensor load of one box (x = element column, y = row) into shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A B + D for m16n8k16 (fp32 accumulate), all four A and C registers.
template <bool kBf16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if (kBf16)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Transpose of an 8x8 matrix of 16-bit elements held one row-pair per lane
// (row lane/4, columns 2*(lane%4), +1): the result uses the same layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// Two floats -> packed 16-bit pair (x in the low half), and the rounding
// remainders of the pair as a second packed pair.
template <bool kBf16>
__device__ __forceinline__ void split_pack(float x, float y, uint32_t& hi, uint32_t& lo) {
  if (kBf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    float2 hf = __bfloat1622float2(h);
    __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<uint32_t*>(&h);
    lo = *reinterpret_cast<uint32_t*>(&l);
  } else {
    __half2 h = __floats2half2_rn(x, y);
    float2 hf = __half22float2(h);
    __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<uint32_t*>(&h);
    lo = *reinterpret_cast<uint32_t*>(&l);
  }
}
// Byte offset of 16-byte chunk c (0..15) of row r in a tile stored as two
// 128-byte-swizzled boxes [16 rows][64 elements].
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void store_out(void* out, long long idx, float x, int out_dtype) {
  if (out_dtype == PA_FP32)
    static_cast<float*>(out)[idx] = x;
  else if (out_dtype == PA_BF16)
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(x);
  else
    static_cast<__half*>(out)[idx] = __float2half_rn(x);
}

__device__ __forceinline__ int clamp_len(const Params& P, int i) {
  int L = P.seq_lens[i];
  int cap = P.max_blocks * kBlock;
  if (L < 0 || L > cap) {
    record_error(P.err, PA_ERR_DEVICE_CHECK, static_cast<long long>(L));
    L = L < 0 ? 0 : cap;
  }
  return L;
}

__device__ __forceinline__ long long lean_per(const Params& P, const int* pfx) {
  long long T = static_cast<long long>(P.Hkv) * pfx[P.B];
  long long per = (T + P.lean_grid - 1) / P.lean_grid;
  return per < kLeanMinBlocks ? kLeanMinBlocks : per;
}

// ---------------------------------------------------------------------------
// Piece enumeration: every thread of the CTA walks the same list.
// ---------------------------------------------------------------------------
struct Piece {
  int i, h, j0, j1, L;
  bool final_out;
  long long rec;  // partial record index (when !final_out)
};

struct PieceIter {
  const Params& P;
  const int* pfx;  // shared: exclusive prefix over sequences (LEAN: tiles, PARTITION: partitions)
  long long x, x_end;        // SEGMENT / PARTITION cursor
  long long cur, end;        // LEAN cursor
  int li, lh, lj;
  bool first;

  __device__ PieceIter(const Params& p, const int* prefix) : P(p), pfx(prefix) {
    first = true;
    if (P.sched == SCHED_LEAN) {
      long long T = static_cast<long long>(P.Hkv) * pfx[P.B];
      long long per = lean_per(P, pfx);
      cur = per * blockIdx.x;
      end = cur + per < T ? cur + per : T;
      if (cur < end) {
        // largest i with Hkv*pfx[i] <= cur (never an empty sequence)
        int lo = 0, hi = P.B - 1;
        while (lo < hi) {
          int mid = (lo + hi + 1) >> 1;
          if (static_cast<long long>(P.Hkv) * pfx[mid] <= cur) lo = mid; else hi = mid - 1;
        }
        li = lo;
        int nb = pfx[li + 1] - pfx[li];
        long long off = cur - static_cast<long long>(P.Hkv) * pfx[li];
        lh = static_cast<int>(off / nb);
        lj = static_cast<int>(off - static_cast<long long>(lh) * nb);
      }
    } else {
      x = blockIdx.x;
      x_end = P.sched == SCHED_SEGMENT ? static_cast<long long>(P.B) * P.Hkv
                                       : static_cast<long long>(P.Hkv) * pfx[P.B];
    }
  }

  __device__ bool next(Piece& pc) {
    if (P.sched == SCHED_LEAN) {
      if (cur >= end) return false;
      int nb = pfx[li + 1] - pfx[li];
      long long seg_start = static_cast<long long>(P.Hkv) * pfx[li] + static_cast<long long>(lh) * nb;
      long long seg_end = seg_start + nb;
      long long pend = end < seg_end ? end : seg_end;
      pc.i = li;
      pc.h = lh;
      pc.j0 = lj;
      pc.j1 = lj + static_cast<int>(pend - cur);
      pc.L = clamp_len(P, li);
      pc.final_out = (lj == 0 && pend == seg_end);
      pc.rec = 2ll * blockIdx.x + (first ? 0 : 1);
      first = false;
      cur = pend;
      if (cur == seg_end) {
        lj = 0;
        if (++lh == P.Hkv) {
          lh = 0;
          do { ++li; } while (li < P.B && pfx[li + 1] == pfx[li]);
        }
      } else {
        lj = pc.j1;
      }
      return true;
    }
    if (x >= x_end) return false;
    if (P.sched == SCHED_SEGMENT) {
      pc.i = static_cast<int>(x / P.Hkv);
      pc.h = static_cast<int>(x - static_cast<long long>(pc.i) * P.Hkv);
      pc.L = clamp_len(P, pc.i);
      pc.j0 = 0;
      pc.j1 = (pc.L + kBlock - 1) / kBlock;
      pc.final_out = true;
      pc.rec = 0;
    } else {  // PARTITION
      long long u = x / P.Hkv;
      pc.h = static_cast<int>(x - u * P.Hkv);
      int lo = 0, hi = P.B - 1;
      while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (pfx[mid] <= u) lo = mid; else hi = mid - 1;
      }
      pc.i = lo;
      pc.L = clamp_len(P, lo);
      int nb = (pc.L + kBlock - 1) / kBlock;
      int p = static_cast<int>(u - pfx[lo]);
      pc.j0 = p * P.partition_blocks;
      pc.j1 = pc.j0 + P.partition_blocks < nb ? pc.j0 + P.partition_blocks : nb;
      pc.final_out = (pfx[lo + 1] - pfx[lo]) == 1;
      pc.rec = x;
    }
    x += gridDim.x;
    return true;
  }
};

// Records of segment (i, h): how many, and the index of the k-th.
struct SegmentRecords {
  long long c0, s0, per, base;
  int count;
  __device__ SegmentRecords(const Params& P, const int* pfx, int i, int h) {
    if (P.sched == SCHED_LEAN) {
      int nb = pfx[i + 1] - pfx[i];
      per = lean_per(P, pfx);
      s0 = static_cast<long long>(P.Hkv) * pfx[i] + static_cast<long long>(h) * nb;
      c0 = s0 / per;
      count = static_cast<int>((s0 + nb - 1) / per - c0 + 1);
      base = 0;
    } else {
      count = pfx[i + 1] - pfx[i];
      base = static_cast<long long>(pfx[i]) * P.Hkv + h;
      c0 = s0 = per = 0;
    }
  }
  __device__ long long at(const Params& P, int k) const {
    if (P.sched == SCHED_LEAN) return 2 * (c0 + k) + ((k == 0 && s0 > c0 * per) ? 1 : 0);
    return base + static_cast<long long>(k) * P.Hkv;
  }
};


// ---------------------------------------------------------------------------
// Shared memory.  The ring comes first at a 1024-byte aligned base (the
// 128-byte swizzle of TMA boxes needs it); the mbarriers need 8 bytes.
// ---------------------------------------------------------------------------
template <int G>
struct __align__(1024) Smem {
  static constexpr int NW = Shape<G>::NW;
  static constexpr int S = Shape<G>::kStages;
  uint8_t stage[S][kStageBytes];
  __align__(16) float ow[NW][G][kHeadDim];
  __align__(8) unsigned long long full[S];
  unsigned long long empty[S];
  float mw[NW][G];
  float lw[NW][G];
  int stage_blk[S];
  int issued[S];
  int consumed[S];
  int abort_flag;
  int merge_flag;
  int pfx[1];  // [B + 1], dynamic tail
};

template <int G>
constexpr bool smem_layout_ok() {
  return offsetof(Smem<G>, stage) == 0 && offsetof(Smem<G>, ow) % 16 == 0 &&
         offsetof(Smem<G>, full) % 8 == 0 && offsetof(Smem<G>, empty) % 8 == 0 &&
         kStageBytes % 1024 == 0 && Shape<G>::kStages % Shape<G>::NW == 0;
}
static_assert(smem_layout_ok<1>() && smem_layout_ok<2>() && smem_layout_ok<3>() &&
                  smem_layout_ok<4>() && smem_layout_ok<5>() && smem_layout_ok<6>() &&
                  smem_layout_ok<7>() && smem_layout_ok<8>(),
              "shared-memory layout breaks a swizzle, vector or mbarrier alignment");

// Dynamic shared memory to request: the struct, the prefix array, and slack
// to align the base to 1024 bytes.
template <int G>
constexpr size_t smem_bytes(int B) {
  return sizeof(Smem<G>) + sizeof(int) * static_cast<size_t>(B + 1) + 1024;
}
// ---------------------------------------------------------------------------
// The decode kernel.
// ---------------------------------------------------------------------------
template <int G, bool kBf16, bool kFused>
__global__ void __launch_bounds__(Shape<G>::kThreads)
    decode_kernel(const __grid_constant__ Params P) {
  constexpr int NW = Shape<G>::NW;
  constexpr int NS = Shape<G>::kStages;
  constexpr int NT = NW * 32;  // consumer threads
  extern __shared__ uint8_t smem_raw[];
  Smem<G>& S = *reinterpret_cast<Smem<G>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // --- set-up: barriers, prefix over sequences -----------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&S.full[s]), 1);
      mbar_init(smem_addr(&S.empty[s]), 1);
      S.issued[s] = 0;
      S.consumed[s] = 0;
    }
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (P.sched != SCHED_SEGMENT && warp == 0) {
    // exclusive prefix of per-sequence counts (tiles for LEAN, partitions for
    // PARTITION), 32 sequences at a time
    int carry = 0;
    for (int base = 0; base < P.B; base += 32) {
      int i = base + lane;
      int c = 0;
      if (i < P.B) {
        int L = P.seq_lens[i];
        int cap = P.max_blocks * kBlock;
        L = L < 0 ? 0 : (L > cap ? cap : L);
        int nb = (L + kBlock - 1) / kBlock;
        c = P.sched == SCHED_LEAN ? nb : (nb + P.partition_blocks - 1) / P.partition_blocks;
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (i < P.B) S.pfx[i] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) S.pfx[P.B] = carry;
  }
  __syncthreads();

  volatile int* abort_flag = &S.abort_flag;

  if (warp == NW) {
    // ======================= producer warp =================================
    PieceIter it(P, S.pfx);
    Piece pc;
    long long n = 0;
    bool ok = true;
    while (ok && it.next(pc)) {
      const int32_t* row = P.tables + static_cast<long long>(pc.i) * P.max_blocks;
      for (int jb = pc.j0; ok && jb < pc.j1; jb += 32) {
        int cnt = pc.j1 - jb < 32 ? pc.j1 - jb : 32;
        int my_blk = lane < cnt ? row[jb + lane] : 0;
        for (int k = 0; k < cnt; ++k, ++n) {
          int blk = __shfl_sync(0xffffffffu, my_blk, k);
          int s = static_cast<int>(n % NS);
          if (lane == 0) {
            if (n >= NS)
              ok = wait_phase(smem_addr(&S.empty[s]), static_cast<uint32_t>(((n / NS) - 1) & 1),
                              abort_flag, P.wait_limit_ns, P.err, 1);
            if (ok) {
              bool valid = blk >= 0 && blk < P.num_blocks;
              S.stage_blk[s] = valid ? blk : -1;
              S.issued[s] += 1;
              uint32_t fb = smem_addr(&S.full[s]);
              if (valid) {
                mbar_arrive_expect_tx(fb, kStageBytes);
                const int y = (blk * P.Hkv + pc.h) * kBlock;  // first token row of the tile
                const uint32_t dst = smem_addr(S.stage[s]);
                tma_load_2d(dst, &P.tmap_k, 0, y, fb);
                tma_load_2d(dst + 2048, &P.tmap_k, kHeadDim / 2, y, fb);
                tma_load_2d(dst + kTileBytes, &P.tmap_v, 0, y, fb);
                tma_load_2d(dst + kTileBytes + 2048, &P.tmap_v, kHeadDim / 2, y, fb);
              } else {
                record_error(P.err, PA_ERR_DEVICE_CHECK, static_cast<long long>(blk));
                mbar_arrive(fb);
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
        }
      }
    }
  } else {
    // ======================= consumer warps ================================
    // MMA fragment coordinates: row group r4 = lane / 4, column pair c4 = lane % 4.
    //   scores  S^T[t][g]: rows t = r4, r4+8 (tokens), columns g = 2*c4, 2*c4+1
    //   output  O^T[d][g]: rows d = 16*mt + r4, +8, the same columns g
    const int r4 = lane >> 2;
    const int c4 = lane & 3;
    const int g0 = 2 * c4;       // first of this lane's two query heads
    const int tid = threadIdx.x;
    // ldmatrix row addresses: lane group lm supplies matrix lm, row lr.  Both
    // operands read [tok 0-7, chunk c], [tok 0-7, chunk c+1]... in the order
    // (tok 0-7, c), (tok 8-15, c) for K and (tok 0-7, c), (tok 0-7, c+1) for V.
    const int lm = lane >> 3, lr = lane & 7;
    const int k_tok = lr + 8 * (lm & 1), k_cadd = lm >> 1;  // A = K tile rows (tokens)
    const int v_tok = lr + 8 * (lm >> 1), v_cadd = lm & 1;  // A = V^T via transposed loads

    // zero rows of empty sequences (split schedules; SEGMENT pieces write them)
    if (P.sched != SCHED_SEGMENT) {
      for (int i = blockIdx.x; i < P.B; i += gridDim.x) {
        if (S.pfx[i + 1] != S.pfx[i]) continue;
        for (int x = tid; x < P.Hq * kHeadDim; x += NT)
          store_out(P.out, static_cast<long long>(i) * P.Hq * kHeadDim + x, 0.f, P.out_dtype);
      }
    }

    PieceIter it(P, S.pfx);
    Piece pc;
    long long n = 0;  // tile counter of the CTA's stream
    bool ok = true;
    while (it.next(pc)) {
      const long long n0 = n;
      const int nblk = pc.j1 - pc.j0;
      n += nblk;
      // B fragments of Q^T: column g = r4 of the group (zero past G), k = dims
      uint32_t qb[8][2];
      if (r4 < G) {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            P.q + (static_cast<long long>(pc.i) * P.Hq + pc.h * G + r4) * kHeadDim);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          qb[ks][0] = qrow[8 * ks + c4];
          qb[ks][1] = qrow[8 * ks + 4 + c4];
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) qb[ks][0] = qb[ks][1] = 0u;
      }
      float o[8][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
      const int nb_total = (pc.L + kBlock - 1) / kBlock;

      // first tile of this warp in the piece
      int first = static_cast<int>((warp - (n0 % NW) + NW) % NW);
      for (int b = first; ok && b < nblk; b += NW) {
        const long long nn = n0 + b;
        const int s = static_cast<int>(nn % NS);
        const uint32_t parity = static_cast<uint32_t>((nn / NS) & 1);
        bool got = wait_phase(smem_addr(&S.full[s]), parity, abort_flag, P.wait_limit_ns, P.err, 2);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          ok = false;
          break;
        }
        const int j = pc.j0 + b;
        const int blk = S.stage_blk[s];
        uint8_t* Ks = S.stage[s];
        uint8_t* Vs = Ks + kTileBytes;
        const uint32_t ks_addr = smem_addr(Ks), vs_addr = smem_addr(Vs);
        const int valid_tokens = pc.L - j * kBlock < kBlock ? pc.L - j * kBlock : kBlock;
        bool touched = false;
        if (blk >= 0) {
          if (kFused && j == nb_total - 1) {
            // the new token: use the caller's k_new/v_new for position L-1
            // and write it to its slot in the pool
            const int tn = (pc.L - 1) & (kBlock - 1);
            const int c = lane & 15;
            const long long src = (static_cast<long long>(pc.i) * P.Hkv + pc.h) * kHeadDim;
            const long long dst =
                ((static_cast<long long>(blk) * P.Hkv + pc.h) * kBlock + tn) * kHeadDim;
            const uint16_t* from = (lane < 16 ? P.k_new : P.v_new) + src;
            uint4 val = *reinterpret_cast<const uint4*>(from + 8 * c);
            *reinterpret_cast<uint4*>((lane < 16 ? Ks : Vs) + swz(tn, c)) = val;
            uint16_t* pool_w = const_cast<uint16_t*>(lane < 16 ? P.k_pool : P.v_pool);
            *reinterpret_cast<uint4*>(pool_w + dst + 8 * c) = val;
            touched = true;
          }
          if (valid_tokens < kBlock) {
            // V rows past the sequence end may hold anything (even NaN):
            // zero them so that 0-weight rows contribute exactly 0
            const int nz = (kBlock - valid_tokens) * 16;
            for (int x = lane; x < nz; x += 32)
              *reinterpret_cast<uint4*>(Vs + swz(valid_tokens + (x >> 4), x & 15)) = make_uint4(0, 0, 0, 0);
            touched = true;
          }
          if (touched) __syncwarp();
          // ---- S^T = K Q^T: M = 16 tokens, N = 8 heads, 8 k-steps of 16 dims
          float st[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(ks_addr + swz(k_tok, 2 * ks + k_cadd), a0, a1, a2, a3);
            mma16816<kBf16>(st, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
          }
          // ---- online softmax of columns g0, g0+1 over tokens r4, r4+8
          float mx[2];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            st[c] = r4 < valid_tokens ? st[c] * P.qscale : -INFINITY;
            st[2 + c] = r4 + 8 < valid_tokens ? st[2 + c] * P.qscale : -INFINITY;
            mx[c] = fmaxf(st[c], st[2 + c]);
#pragma unroll
            for (int msk = 4; msk < 32; msk <<= 1) mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], msk));
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (mx[c] > m_run[c] + kRescaleThreshold) {  // uniform across the column's lanes
              const float mn = fmaxf(m_run[c], mx[c]);
              const float alpha = fast_exp2(m_run[c] - mn);
              l_run[c] *= alpha;
#pragma unroll
              for (int mt = 0; mt < 8; ++mt) {
                o[mt][c] *= alpha;
                o[mt][2 + c] *= alpha;
              }
              m_run[c] = mn;
            }
          }
          float p[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            p[k] = fast_exp2(st[k] - m_run[k & 1]);
            l_run[k & 1] += p[k];
          }
          // B fragments of P^T (k = tokens, n = heads): transpose the packed
          // 8x8 blocks (tokens 0-7 and 8-15) of the score fragment
          uint32_t h0, l0, h1, l1;
          split_pack<kBf16>(p[0], p[1], h0, l0);
          split_pack<kBf16>(p[2], p[3], h1, l1);
          h0 = movmatrix_t(h0);
          l0 = movmatrix_t(l0);
          h1 = movmatrix_t(h1);
          l1 = movmatrix_t(l1);
          // ---- O^T += V^T P^T: M = 16 dims per m-tile (8 m-tiles), N = 8 heads, K = 16 tokens
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(vs_addr + swz(v_tok, 2 * mt + v_cadd), a0, a1, a2, a3);
            mma16816<kBf16>(o[mt], a0, a1, a2, a3, h0, h1);
            mma16816<kBf16>(o[mt], a0, a1, a2, a3, l0, l1);
          }
        }
        __syncwarp();
        if (touched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) {
          S.consumed[s] += 1;
          mbar_arrive(smem_addr(&S.empty[s]));
        }
      }

      // ---- merge the NW warps' states for this piece
      float lsum[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        lsum[c] = l_run[c];
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) lsum[c] += __shfl_xor_sync(0xffffffffu, lsum[c], msk);
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (g0 + c < G) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            S.ow[warp][g0 + c][16 * mt + r4] = o[mt][c];
            S.ow[warp][g0 + c][16 * mt + r4 + 8] = o[mt][2 + c];
          }
          if (r4 == 0) {
            S.mw[warp][g0 + c] = m_run[c];
            S.lw[warp][g0 + c] = lsum[c];
          }
        }
      }
      consumers_sync<NT>();
      for (int x = tid; x < G * kHeadDim; x += NT) {
        const int g = x / kHeadDim, e = x % kHeadDim;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, S.mw[w][g]);
        float Ls = 0.f, Os = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            float f = fast_exp2(S.mw[w][g] - M);
            Ls = fmaf(S.lw[w][g], f, Ls);
            Os = fmaf(S.ow[w][g][e], f, Os);
          }
        }
        if (pc.final_out) {
          long long idx = (static_cast<long long>(pc.i) * P.Hq + pc.h * G + g) * kHeadDim + e;
          store_out(P.out, idx, Ls > 0.f ? Os / Ls : 0.f, P.out_dtype);
        } else {
          float* rec = P.ws + pc.rec * record_floats(G);
          rec[g * kHeadDim + e] = Os;
          if (e == 0) {
            rec[G * kHeadDim + g] = M;
            rec[G * kHeadDim + 64 + g] = Ls;
          }
        }
      }
      if (!pc.final_out) {
        // ---- log-sum-exp merge by the CTA that completes the segment:
        //   M = max_p m_p;  out = sum_p 2^(m_p-M) o_p / sum_p 2^(m_p-M) l_p
        __threadfence();
        consumers_sync<NT>();
        const SegmentRecords recs(P, S.pfx, pc.i, pc.h);
        int* counter = P.counters + static_cast<long long>(pc.i) * P.Hkv + pc.h;
        if (tid == 0) S.merge_flag = atomicAdd(counter, 1) == recs.count - 1;
        consumers_sync<NT>();
        if (S.merge_flag) {
          __threadfence();
          for (int x = tid; x < G * kHeadDim; x += NT) {
            const int g = x / kHeadDim, e = x % kHeadDim;
            float M = -INFINITY;
            for (int k = 0; k < recs.count; ++k)
              M = fmaxf(M, __ldcg(P.ws + recs.at(P, k) * record_floats(G) + G * kHeadDim + g));
            float Ls = 0.f, Os = 0.f;
            for (int k = 0; k < recs.count; ++k) {
              const float* rec = P.ws + recs.at(P, k) * record_floats(G);
              float f = fast_exp2(__ldcg(rec + G * kHeadDim + g) - M);
              Ls = fmaf(__ldcg(rec + G * kHeadDim + 64 + g), f, Ls);
              Os = fmaf(__ldcg(rec + g * kHeadDim + e), f, Os);
            }
            long long idx = (static_cast<long long>(pc.i) * P.Hq + pc.h * G + g) * kHeadDim + e;
            store_out(P.out, idx, Ls > 0.f ? Os / Ls : 0.f, P.out_dtype);
          }
          if (tid == 0) *counter = 0;
        }
      }
      // all consumers agree whether to stop; also guards the shared scratch
      if (consumers_sync_or<NT>(ok ? 0 : 1)) break;
    }
  }

  // --- drain: never leave a bulk copy in flight into this CTA's memory ------
  __syncthreads();
  if (threadIdx.x == 0 && S.abort_flag) {
    for (int s = 0; s < NS; ++s) {
      if (S.issued[s] > S.consumed[s]) {
        uint32_t parity = static_cast<uint32_t>((S.issued[s] - 1) & 1);
        long long t0 = global_ns();
        while (!mbar_try_wait(smem_addr(&S.full[s]), parity) && global_ns() - t0 < P.wait_limit_ns) {
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Host side: dispatch over (G, dtype, fused).
// ---------------------------------------------------------------------------

// Library-owned timing events (pa_profile_start / pa_profile_stop).
static std::vector<cudaEvent_t> g_prof_events;  // [2 * capacity]
static int g_prof_next = 0;

static void profile_release() {
  for (cudaEvent_t e : g_prof_events) cudaEventDestroy(e);
  g_prof_events.clear();
  g_prof_next = 0;
}

template <int G, bool kBf16, bool kFused>
static int occupancy_for(size_t bytes) {
  static std::mutex mu;
  static int cached_dev = -1;
  static size_t cached_bytes = 0;
  static int cached_occ = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if (dev == cached_dev && bytes == cached_bytes) return cached_occ;
  if (cudaFuncSetAttribute(decode_kernel<G, kBf16, kFused>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes<G>(kMaxSplitSeqs))) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<G, kBf16, kFused>,
                                                    Shape<G>::kThreads, bytes) != cudaSuccess)
    return 0;
  if (occ > kMaxCtasPerSm) occ = kMaxCtasPerSm;
  cached_dev = dev;
  cached_bytes = bytes;
  cached_occ = occ;
  return occ;
}

template <int G, bool kBf16, bool kFused>
static int launch_typed(Params& P, int device, cudaStream_t stream) {
  int B_smem = P.sched == SCHED_SEGMENT ? 0 : P.B;
  size_t bytes = smem_bytes<G>(B_smem);
  int occ = occupancy_for<G, kBf16, kFused>(bytes);
  if (occ <= 0) return PA_ERR_CUDA;
  long long slots = static_cast<long long>(sm_count(device)) * occ;
  long long grid;
  if (P.sched == SCHED_SEGMENT) {
    long long segs = static_cast<long long>(P.B) * P.Hkv;
    grid = segs < slots ? segs : slots;
  } else if (P.sched == SCHED_LEAN) {
    grid = slots;
    P.lean_grid = static_cast<int>(grid);
  } else {
    long long parts = static_cast<long long>(P.B) * P.Hkv *
                      ((P.max_blocks + P.partition_blocks - 1) / P.partition_blocks);
    grid = parts < slots ? parts : slots;
  }
  if (grid < 1) grid = 1;
  const bool timed = 2 * static_cast<size_t>(g_prof_next) < g_prof_events.size();
  if (timed && cudaEventRecord(g_prof_events[2 * g_prof_next], stream) != cudaSuccess) return PA_ERR_CUDA;
  decode_kernel<G, kBf16, kFused>
      <<<static_cast<int>(grid), Shape<G>::kThreads, bytes, stream>>>(P);
  if (timed) {
    if (cudaEventRecord(g_prof_events[2 * g_prof_next + 1], stream) != cudaSuccess) return PA_ERR_CUDA;
    ++g_prof_next;
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <bool kBf16, bool kFused>
static int launch_g(int G, Params& P, int device, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_typed<1, kBf16, kFused>(P, device, stream);
    case 2: return launch_typed<2, kBf16, kFused>(P, device, stream);
    case 3: return launch_typed<3, kBf16, kFused>(P, device, stream);
    case 4: return launch_typed<4, kBf16, kFused>(P, device, stream);
    case 5: return launch_typed<5, kBf16, kFused>(P, device, stream);
    case 6: return launch_typed<6, kBf16, kFused>(P, device, stream);
    case 7: return launch_typed<7, kBf16, kFused>(P, device, stream);
    case 8: return launch_typed<8, kBf16, kFused>(P, device, stream);
    default: return PA_ERR_UNSUPPORTED;
  }
}

// Workspace layout: partial records, then the per-segment counters at a
// 256-byte aligned offset.
struct WorkspaceLayout {
  size_t records_bytes, counters_offset, total;
};

static bool workspace_layout(const pa_pool* p, int B, int Hq, int max_blocks, int partition_blocks,
                             WorkspaceLayout* out) {
  if (!p || B <= 0 || Hq <= 0 || max_blocks <= 0 || partition_blocks < 0) return false;
  if (Hq % p->n_kv_heads) return false;
  int G = Hq / p->n_kv_heads;
  if (G > PA_MAX_GROUP) return false;
  size_t rec = sizeof(float) * record_floats(G);
  size_t n_rec;
  if (partition_blocks == 0)  // LEAN: two records per CTA of the largest grid
    n_rec = 2 * static_cast<size_t>(sm_count(p->device)) * kMaxCtasPerSm;
  else
    n_rec = static_cast<size_t>(B) * p->n_kv_heads *
            ((max_blocks + partition_blocks - 1) / partition_blocks);
  out->records_bytes = rec * n_rec;
  out->counters_offset = (out->records_bytes + 255) / 256 * 256;
  out->total = out->counters_offset + sizeof(int) * static_cast<size_t>(B) * p->n_kv_heads;
  return true;
}

static int decode_common(pa_pool_t p, const void* q, const void* k_new, const void* v_new,
                         const int32_t* tables, int max_blocks, const int32_t* seq_lens, int B,
                         int Hq, float scale, void* out, int out_dtype, int sched,
                         int partition_blocks, void* ws, size_t ws_bytes, void* stream) {
  if (!p || !q || !tables || !seq_lens || !out || B <= 0 || Hq <= 0 || max_blocks <= 0)
    return PA_ERR_INVALID;
  if (out_dtype != PA_FP16 && out_dtype != PA_BF16 && out_dtype != PA_FP32) return PA_ERR_INVALID;
  if (Hq % p->n_kv_heads) return PA_ERR_INVALID;
  const int G = Hq / p->n_kv_heads;
  if (G > PA_MAX_GROUP) return PA_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(q) & 15) return PA_ERR_INVALID;
  const bool fused = k_new != nullptr;
  if (fused && ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15))
    return PA_ERR_INVALID;
  WorkspaceLayout lay{};
  if (sched != SCHED_SEGMENT) {
    if (B > kMaxSplitSeqs) return PA_ERR_UNSUPPORTED;
    if (!workspace_layout(p, B, Hq, max_blocks, partition_blocks, &lay)) return PA_ERR_INVALID;
    if (!ws || ws_bytes < lay.total || (reinterpret_cast<uintptr_t>(ws) & 15)) return PA_ERR_INVALID;
  }
  Params P{};
  P.tmap_k = p->tmap_k;
  P.tmap_v = p->tmap_v;
  P.q = static_cast<const uint16_t*>(q);
  P.k_pool = static_cast<const uint16_t*>(p->k);
  P.v_pool = static_cast<const uint16_t*>(p->v);
  P.k_new = static_cast<const uint16_t*>(k_new);
  P.v_new = static_cast<const uint16_t*>(v_new);
  P.tables = tables;
  P.seq_lens = seq_lens;
  P.out = out;
  P.ws = static_cast<float*>(ws);
  P.counters = ws ? reinterpret_cast<int*>(static_cast<char*>(ws) + lay.counters_offset) : nullptr;
  P.err = p->err;
  P.num_blocks = p->num_blocks;
  P.max_blocks = max_blocks;
  P.B = B;
  P.Hq = Hq;
  P.Hkv = p->n_kv_heads;
  P.out_dtype = out_dtype;
  P.qscale = scale * kLog2e;
  P.sched = sched;
  P.partition_blocks = partition_blocks > 0 ? partition_blocks : 1;
  P.lean_grid = 1;
  P.wait_limit_ns = wait_limit_ns();
  cudaStream_t st = as_stream(stream);
  const bool bf16 = p->dtype == PA_BF16;
  if (bf16)
    return fused ? launch_g<true, true>(G, P, p->device, st) : launch_g<true, false>(G, P, p->device, st);
  return fused ? launch_g<false, true>(G, P, p->device, st) : launch_g<false, false>(G, P, p->device, st);
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_profile_start(int capacity) {
  if (capacity < 0) return PA_ERR_INVALID;
  profile_release();
  g_prof_events.resize(2 * static_cast<size_t>(capacity), nullptr);
  for (auto& e : g_prof_events) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      profile_release();
      return PA_ERR_CUDA;
    }
  }
  return PA_OK;
}

int pa_profile_stop(float* ms, int cap) {
  if (cap < 0 || (cap > 0 && !ms)) return PA_ERR_INVALID;
  int n = g_prof_next;
  int status = PA_OK;
  for (int k = 0; k < n && k < cap; ++k) {
    if (cudaEventSynchronize(g_prof_events[2 * k + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms[k], g_prof_events[2 * k], g_prof_events[2 * k + 1]) != cudaSuccess)
      status = PA_ERR_CUDA;
  }
  profile_release();
  return status == PA_OK ? n : status;
}

int pa_decode(pa_pool_t p, const void* q, const int32_t* block_tables, int max_blocks_per_seq,
              const int32_t* seq_lens, int num_seqs, int n_q_heads, float scale, void* out,
              int out_dtype, void* stream) {
  return decode_common(p, q, nullptr, nullptr, block_tables, max_blocks_per_seq, seq_lens,
                       num_seqs, n_q_heads, scale, out, out_dtype, SCHED_SEGMENT, 0, nullptr, 0,
                       stream);
}

size_t pa_decode_workspace_bytes(pa_pool_t p, int num_seqs, int n_q_heads, int max_blocks_per_seq,
                                 int partition_blocks) {
  WorkspaceLayout lay{};
  if (!workspace_layout(p, num_seqs, n_q_heads, max_blocks_per_seq, partition_blocks, &lay)) return 0;
  return lay.total;
}

int pa_decode_split(pa_pool_t p, const void* q, const int32_t* block_tables,
                    int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int n_q_heads,
                    float scale, void* out, int out_dtype, int partition_blocks, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (partition_blocks < 0) return PA_ERR_INVALID;
  int sched = partition_blocks == 0 ? SCHED_LEAN : SCHED_PARTITION;
  return decode_common(p, q, nullptr, nullptr, block_tables, max_blocks_per_seq, seq_lens,
                       num_seqs, n_q_heads, scale, out, out_dtype, sched, partition_blocks,
                       workspace, workspace_bytes, stream);
}

int pa_append_decode(pa_pool_t p, const void* q, const void* k_new, const void* v_new,
                     const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                     int num_seqs, int n_q_heads, float scale, void* out, int out_dtype,
                     int partition_blocks, void* workspace, size_t workspace_bytes, void* stream) {
  if (!k_new || !v_new || partition_blocks < 0) return PA_ERR_INVALID;
  int sched = partition_blocks == 0 ? SCHED_LEAN : SCHED_PARTITION;
  return decode_common(p, q, k_new, v_new, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                       n_q_heads, scale, out, out_dtype, sched, partition_blocks, workspace,
                       workspace_bytes, stream);
}

}  // extern "C"
