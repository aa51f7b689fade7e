// Paged decode attention for sm_103a.
//
// One query token per sequence attends over its cache, which sits in
// fixed-size 16-token blocks found through a per-sequence block table
// ("Serving", section 23.4 Paged Attention).  Decode reads the whole cache
// for one token per sequence, so it is bound by HBM bandwidth ("Serving",
// section 23.2 Prefill and Decode); the design keeps every K/V byte read
// exactly once and keeps enough bytes in flight to saturate HBM3e.
//
// Work decomposition.  A segment is one (sequence i, kv head h) pair: its
// nb_i = ceil(L_i/16) tiles of 16 tokens x 128 dims (4 KiB each for K and
// for V).  The whole grouped-query head group (G = Hq/Hkv query heads) of the
// segment is handled by the same CTA, so a tile is fetched once and used by G
// heads.  A CTA is persistent and processes a list of pieces (a contiguous
// range of a segment's tiles) given by one of three schedules:
//   SEGMENT    whole segments, strided over CTAs (no workspace);
//   LEAN       the concatenated tile stream of all segments cut into equal
//              per-CTA ranges (perfect balance for any length mix); a segment
//              cut by a range boundary leaves partial results;
//   PARTITION  fixed partitions of `partition_blocks` tiles per segment.
// Partial results (running max m, sum l, unnormalised o, fp32) are merged by
// a log-sum-exp kernel.
//
// CTA layout: 4 consumer warps + 1 producer warp.  The producer walks the
// block table and streams each (block, head) K and V tile (contiguous in the
// [block][head][16][128] pool) into an 8-stage shared-memory ring with
// cp.async.bulk, completion tracked by mbarriers.  Tile n of the CTA's stream
// goes to stage n % 8 and is consumed by warp n % 4, which runs the online
// softmax over its own tiles; the 4 warps' states are merged per piece.
//
// Per tile a consumer warp computes, in fp32:
//   scores  s[t][g] = <q_g * scale * log2(e), K[t]>   (8 lanes per token row,
//           partial dots reduced across lanes by a reduce-scatter butterfly)
//   online softmax with a lazily moved running max (rescale only when a new
//           max exceeds the old by 2^8), p = 2^(s - m)
//   o[g][:] += sum_t p[t][g] V[t][:]                    (16 lanes per row)
// Positions t >= L are masked by select, never by multiplying, so padding or
// stale slots (even NaN) never reach the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstddef>
#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace pa {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 8;
constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
constexpr int kMaxSplitSeqs = 8192;          // sequences per split launch
constexpr int kMaxCtasPerSm = 4;
constexpr int kLeanMinBlocks = 8;            // smallest LEAN range per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;    // log2 units

enum { SCHED_SEGMENT = 0, SCHED_LEAN = 1, SCHED_PARTITION = 2 };

struct Params {
  const uint16_t* q;        // [B][Hq][128]
  const uint16_t* k_pool;   // [N][Hkv][16][128]
  const uint16_t* v_pool;
  const uint16_t* k_new;    // [B][Hkv][128], fused append only
  const uint16_t* v_new;
  const int32_t* tables;    // [B][max_blocks]
  const int32_t* seq_lens;  // [B]
  void* out;                // [B][Hq][128]
  float* ws;                // partial records
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
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ int consumers_sync_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 2, 128, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred)
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

// 16-bit -> fp32 for 8 packed elements.
template <bool kBf16>
__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (kBf16) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
      float2 t = __half22float2(h);
      f[2 * k] = t.x;
      f[2 * k + 1] = t.y;
    }
  }
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
  // SEGMENT / PARTITION cursor
  long long x, x_end;
  // LEAN cursor
  long long cur, end;
  int li, lh, lj;
  bool first;

  __device__ PieceIter(const Params& p, const int* prefix) : P(p), pfx(prefix) {
    first = true;
    if (P.sched == SCHED_LEAN) {
      long long T = static_cast<long long>(P.Hkv) * pfx[P.B];
      long long per = (T + P.lean_grid - 1) / P.lean_grid;
      if (per < kLeanMinBlocks) per = kLeanMinBlocks;
      cur = per * blockIdx.x;
      end = cur + per < T ? cur + per : T;
      if (cur < end) {
        // largest i with Hkv*pfx[i] <= cur
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

// ---------------------------------------------------------------------------
// Shared memory.
// ---------------------------------------------------------------------------
// Arrays read or written with 16-byte vector accesses come first and are
// 16-byte aligned (checked below); the mbarriers need 8-byte alignment.
template <int G>
struct __align__(128) Smem {
  uint8_t stage[kStages][kStageBytes];
  __align__(16) float ow[kConsumerWarps][G][kHeadDim];
  __align__(16) float pbuf[kConsumerWarps][kBlock][G <= 4 ? 4 : 8];
  __align__(8) unsigned long long full[kStages];
  unsigned long long empty[kStages];
  float mw[kConsumerWarps][G];
  float lw[kConsumerWarps][G];
  int stage_blk[kStages];
  int issued[kStages];
  int consumed[kStages];
  int abort_flag;
  int pfx[1];  // [B + 1], dynamic tail
};

template <int G>
constexpr bool smem_layout_ok() {
  return offsetof(Smem<G>, stage) == 0 && offsetof(Smem<G>, ow) % 16 == 0 &&
         offsetof(Smem<G>, pbuf) % 16 == 0 && offsetof(Smem<G>, full) % 8 == 0 &&
         offsetof(Smem<G>, empty) % 8 == 0 && kStageBytes % 128 == 0;
}
static_assert(smem_layout_ok<1>() && smem_layout_ok<2>() && smem_layout_ok<3>() &&
                  smem_layout_ok<4>() && smem_layout_ok<5>() && smem_layout_ok<6>() &&
                  smem_layout_ok<7>() && smem_layout_ok<8>(),
              "shared-memory layout breaks a vector or mbarrier alignment");

template <int G>
constexpr size_t smem_bytes(int B) {
  return sizeof(Smem<G>) + sizeof(int) * static_cast<size_t>(B + 1);
}

// ---------------------------------------------------------------------------
// The decode kernel.
// ---------------------------------------------------------------------------
template <int G, bool kBf16, bool kFused>
__global__ void __launch_bounds__(kThreads) decode_kernel(const Params P) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<G>& S = *reinterpret_cast<Smem<G>*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // --- set-up: barriers, prefix over sequences -----------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
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
  const long long head_stride = static_cast<long long>(kBlock) * kHeadDim;  // elements per tile

  if (warp == kConsumerWarps) {
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
          int s = static_cast<int>(n % kStages);
          if (lane == 0) {
            if (n >= kStages)
              ok = wait_phase(smem_addr(&S.empty[s]), static_cast<uint32_t>(((n / kStages) - 1) & 1),
                              abort_flag, P.wait_limit_ns, P.err, 1);
            if (ok) {
              bool valid = blk >= 0 && blk < P.num_blocks;
              S.stage_blk[s] = valid ? blk : -1;
              S.issued[s] += 1;
              uint32_t fb = smem_addr(&S.full[s]);
              if (valid) {
                mbar_arrive_expect_tx(fb, kStageBytes);
                long long off = (static_cast<long long>(blk) * P.Hkv + pc.h) * head_stride;
                bulk_copy_g2s(smem_addr(S.stage[s]), P.k_pool + off, kTileBytes, fb);
                bulk_copy_g2s(smem_addr(S.stage[s] + kTileBytes), P.v_pool + off, kTileBytes, fb);
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
    constexpr int TPL = G <= 4 ? 8 : 16;   // lanes per token row in the score phase
    constexpr int CH = 16 / TPL;           // 16-byte chunks per lane
    constexpr int TPP = 32 / TPL;          // tokens per pass
    constexpr int NP = kBlock / TPP;       // passes per tile
    constexpr int PB = G <= 4 ? 4 : 8;     // pbuf row stride
    const int cg = lane % TPL;
    const int ts = lane / TPL;
    const int kq = (lane >> 1) & (NP - 1);  // pass index this lane owns after the reduction
    const int tq = kq * TPP + ts;           // token this lane owns after the reduction
    const int c16 = lane & 15;              // value phase: chunk
    const int r16 = lane >> 4;              // value phase: token parity

    PieceIter it(P, S.pfx);
    Piece pc;
    long long n = 0;  // tile counter of the CTA's stream
    bool ok = true;
    while (it.next(pc)) {
      const long long n0 = n;
      const int nblk = pc.j1 - pc.j0;
      n += nblk;
      // query group of this piece, pre-scaled into log2 units
      float qf[G][CH][8];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint16_t* qrow = P.q + (static_cast<long long>(pc.i) * P.Hq + pc.h * G + g) * kHeadDim;
#pragma unroll
        for (int u = 0; u < CH; ++u) {
          uint4 raw = *reinterpret_cast<const uint4*>(qrow + 8 * (cg + TPL * u));
          unpack8<kBf16>(raw, qf[g][u]);
#pragma unroll
          for (int e = 0; e < 8; ++e) qf[g][u][e] *= P.qscale;
        }
      }
      float o[G][8];
      float m_run[G], l_run[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[g][e] = 0.f;
      }
      const int nb_total = (pc.L + kBlock - 1) / kBlock;

      // first tile of this warp in the piece
      int first = static_cast<int>((warp - (n0 % kConsumerWarps) + kConsumerWarps) % kConsumerWarps);
      for (int b = first; ok && b < nblk; b += kConsumerWarps) {
        const long long nn = n0 + b;
        const int s = static_cast<int>(nn % kStages);
        const uint32_t parity = static_cast<uint32_t>((nn / kStages) & 1);
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
        const int valid_tokens = pc.L - j * kBlock < kBlock ? pc.L - j * kBlock : kBlock;
        bool patched = false;
        if (blk >= 0) {
          if (kFused && j == nb_total - 1) {
            // the new token: use the caller's k_new/v_new for position L-1
            // and write it to its slot in the pool
            const int tn = (pc.L - 1) & (kBlock - 1);
            const long long src = (static_cast<long long>(pc.i) * P.Hkv + pc.h) * kHeadDim;
            const long long dst =
                ((static_cast<long long>(blk) * P.Hkv + pc.h) * kBlock + tn) * kHeadDim;
            const uint16_t* from = (lane < 16 ? P.k_new : P.v_new) + src;
            uint4 val = *reinterpret_cast<const uint4*>(from + 8 * c16);
            uint8_t* tile = lane < 16 ? Ks : Vs;
            *reinterpret_cast<uint4*>(tile + tn * kRowBytes + 16 * c16) = val;
            uint16_t* pool_w = const_cast<uint16_t*>(lane < 16 ? P.k_pool : P.v_pool);
            *reinterpret_cast<uint4*>(pool_w + dst + 8 * c16) = val;
            patched = true;
            __syncwarp();
          }
          // ---- scores: partial dot products over this lane's chunks
          float part[NP][G];
#pragma unroll
          for (int k = 0; k < NP; ++k) {
            const int t = k * TPP + ts;
#pragma unroll
            for (int g = 0; g < G; ++g) part[k][g] = 0.f;
#pragma unroll
            for (int u = 0; u < CH; ++u) {
              uint4 raw = *reinterpret_cast<const uint4*>(Ks + t * kRowBytes + 16 * (cg + TPL * u));
              float kf[8];
              unpack8<kBf16>(raw, kf);
#pragma unroll
              for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < 8; ++e) part[k][g] = fmaf(qf[g][u][e], kf[e], part[k][g]);
            }
          }
          // ---- reduce-scatter across the TPL lanes of a row
#pragma unroll
          for (int lvl = 0; (NP >> (lvl + 1)) >= 1; ++lvl) {
            const int m = TPL >> (lvl + 1);
            const int half = NP >> (lvl + 1);
            const bool hi = (lane & m) != 0;
#pragma unroll
            for (int kk = 0; kk < half; ++kk)
#pragma unroll
              for (int g = 0; g < G; ++g) {
                float keep = hi ? part[kk + half][g] : part[kk][g];
                float send = hi ? part[kk][g] : part[kk + half][g];
                part[kk][g] = keep + __shfl_xor_sync(0xffffffffu, send, m);
              }
          }
#pragma unroll
          for (int g = 0; g < G; ++g) part[0][g] += __shfl_xor_sync(0xffffffffu, part[0][g], 1);
          // ---- online softmax (log2 domain)
          const bool tvalid = tq < valid_tokens;
          float sc[G], bm[G];
#pragma unroll
          for (int g = 0; g < G; ++g) {
            sc[g] = tvalid ? part[0][g] : -INFINITY;
            bm[g] = sc[g];
#pragma unroll
            for (int msk = 2; msk < 32; msk <<= 1)
              bm[g] = fmaxf(bm[g], __shfl_xor_sync(0xffffffffu, bm[g], msk));
          }
          bool grow = false;
#pragma unroll
          for (int g = 0; g < G; ++g) grow |= bm[g] > m_run[g] + kRescaleThreshold;
          if (grow) {  // warp-uniform
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float mn = fmaxf(m_run[g], bm[g]);
              float alpha = fast_exp2(m_run[g] - mn);
              l_run[g] *= alpha;
#pragma unroll
              for (int e = 0; e < 8; ++e) o[g][e] *= alpha;
              m_run[g] = mn;
            }
          }
          float (*pb)[PB] = S.pbuf[warp];
          if ((lane & 1) == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float p = fast_exp2(sc[g] - m_run[g]);
              l_run[g] += p;
              pb[tq][g] = p;
            }
          }
          __syncwarp();
          // ---- o += p V
#pragma unroll
          for (int k = 0; k < kBlock / 2; ++k) {
            const int t = 2 * k + r16;
            if (t < valid_tokens) {
              uint4 raw = *reinterpret_cast<const uint4*>(Vs + t * kRowBytes + 16 * c16);
              float vf[8];
              unpack8<kBf16>(raw, vf);
              float p[PB];
#pragma unroll
              for (int g4 = 0; g4 < PB; g4 += 4) {
                float4 pp = *reinterpret_cast<const float4*>(&pb[t][g4]);
                p[g4] = pp.x; p[g4 + 1] = pp.y; p[g4 + 2] = pp.z; p[g4 + 3] = pp.w;
              }
#pragma unroll
              for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < 8; ++e) o[g][e] = fmaf(p[g], vf[e], o[g][e]);
            }
          }
          __syncwarp();
        }
        if (patched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) {
          S.consumed[s] += 1;
          mbar_arrive(smem_addr(&S.empty[s]));
        }
      }

      // ---- merge the 4 warps' states for this piece
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], 16);
        float l = l_run[g];
#pragma unroll
        for (int msk = 1; msk < 32; msk <<= 1) l += __shfl_xor_sync(0xffffffffu, l, msk);
        l_run[g] = l;
      }
      if (lane < 16) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float4* dst = reinterpret_cast<float4*>(&S.ow[warp][g][8 * lane]);
          dst[0] = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
          dst[1] = make_float4(o[g][4], o[g][5], o[g][6], o[g][7]);
        }
      }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          S.mw[warp][g] = m_run[g];
          S.lw[warp][g] = l_run[g];
        }
      }
      consumers_sync();
      const int e = threadIdx.x;  // 0..127: output element
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, S.mw[w][g]);
        float Ls = 0.f, Os = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
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
      // all consumers agree whether to stop; also guards S.ow/mw/lw reuse
      if (consumers_sync_or(ok ? 0 : 1)) break;
    }
  }

  // --- drain: never leave a bulk copy in flight into this CTA's memory ------
  __syncthreads();
  if (threadIdx.x == 0 && S.abort_flag) {
    for (int s = 0; s < kStages; ++s) {
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
// Log-sum-exp merge of partial records: one CTA (128 threads) per segment.
//   M = max_p m_p;  out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p
// Also writes the zero rows of empty sequences.
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(128) merge_kernel(const Params P) {
  const int i = blockIdx.x / P.Hkv;
  const int h = blockIdx.x - i * P.Hkv;
  const int e = threadIdx.x;
  __shared__ long long red[2][4];
  int L = P.seq_lens[i];
  const int cap = P.max_blocks * kBlock;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int nb = (L + kBlock - 1) / kBlock;
  const long long row0 = (static_cast<long long>(i) * P.Hq + h * G) * kHeadDim;
  if (nb == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) store_out(P.out, row0 + g * kHeadDim + e, 0.f, P.out_dtype);
    return;
  }
  // prefix (sequences before i) and total of per-sequence counts
  long long before = 0, total = 0;
  for (int j = e; j < P.B; j += 128) {
    int Lj = P.seq_lens[j];
    Lj = Lj < 0 ? 0 : (Lj > cap ? cap : Lj);
    int nbj = (Lj + kBlock - 1) / kBlock;
    int c = P.sched == SCHED_LEAN ? nbj : (nbj + P.partition_blocks - 1) / P.partition_blocks;
    total += c;
    if (j < i) before += c;
  }
#pragma unroll
  for (int msk = 16; msk >= 1; msk >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, msk);
    total += __shfl_xor_sync(0xffffffffu, total, msk);
  }
  if ((e & 31) == 0) {
    red[0][e >> 5] = before;
    red[1][e >> 5] = total;
  }
  __syncthreads();
  before = red[0][0] + red[0][1] + red[0][2] + red[0][3];
  total = red[1][0] + red[1][1] + red[1][2] + red[1][3];

  long long rec0, step = 0;
  int count;
  // LEAN: the records of the CTAs whose ranges cut this segment
  long long c0 = 0, s0 = 0, per = 1;
  if (P.sched == SCHED_LEAN) {
    long long T = static_cast<long long>(P.Hkv) * total;
    per = (T + P.lean_grid - 1) / P.lean_grid;
    if (per < kLeanMinBlocks) per = kLeanMinBlocks;
    s0 = static_cast<long long>(P.Hkv) * before + static_cast<long long>(h) * nb;
    c0 = s0 / per;
    long long c1 = (s0 + nb - 1) / per;
    if (c0 == c1) return;  // written directly by the decode kernel
    count = static_cast<int>(c1 - c0 + 1);
    rec0 = 0;
  } else {
    int parts = (nb + P.partition_blocks - 1) / P.partition_blocks;
    if (parts == 1) return;
    count = parts;
    rec0 = before * P.Hkv + h;
    step = P.Hkv;
  }
  const int RF = record_floats(G);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
    for (int p = 0; p < count; ++p) {
      long long r = P.sched == SCHED_LEAN
                        ? 2 * (c0 + p) + ((p == 0 && s0 > c0 * per) ? 1 : 0)
                        : rec0 + p * step;
      M = fmaxf(M, P.ws[r * RF + G * kHeadDim + g]);
    }
    float Ls = 0.f, Os = 0.f;
    for (int p = 0; p < count; ++p) {
      long long r = P.sched == SCHED_LEAN
                        ? 2 * (c0 + p) + ((p == 0 && s0 > c0 * per) ? 1 : 0)
                        : rec0 + p * step;
      const float* rec = P.ws + r * RF;
      float f = fast_exp2(rec[G * kHeadDim + g] - M);
      Ls = fmaf(rec[G * kHeadDim + 64 + g], f, Ls);
      Os = fmaf(rec[g * kHeadDim + e], f, Os);
    }
    store_out(P.out, row0 + g * kHeadDim + e, Ls > 0.f ? Os / Ls : 0.f, P.out_dtype);
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
static int occupancy_for(int B) {
  static std::mutex mu;
  static int cached_dev = -1, cached_B = -1, cached_occ = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if (dev == cached_dev && B == cached_B) return cached_occ;
  size_t bytes = smem_bytes<G>(B);
  if (cudaFuncSetAttribute(decode_kernel<G, kBf16, kFused>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<G, kBf16, kFused>, kThreads,
                                                    bytes) != cudaSuccess)
    return 0;
  if (occ > kMaxCtasPerSm) occ = kMaxCtasPerSm;
  cached_dev = dev;
  cached_B = B;
  cached_occ = occ;
  return occ;
}

template <int G, bool kBf16, bool kFused>
static int launch_typed(Params& P, int device, cudaStream_t stream) {
  int B_smem = P.sched == SCHED_SEGMENT ? 0 : P.B;
  int occ = occupancy_for<G, kBf16, kFused>(B_smem);
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
      <<<static_cast<int>(grid), kThreads, smem_bytes<G>(B_smem), stream>>>(P);
  if (timed) {
    if (cudaEventRecord(g_prof_events[2 * g_prof_next + 1], stream) != cudaSuccess) return PA_ERR_CUDA;
    ++g_prof_next;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (P.sched != SCHED_SEGMENT) {
    merge_kernel<G><<<P.B * P.Hkv, 128, 0, stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
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

static int choose_partition(int partition_blocks) {
  return partition_blocks;  // 0 -> LEAN
}

// Upper bound on the CTAs of a LEAN launch (for workspace sizing).
static long long lean_grid_bound(int device) {
  return static_cast<long long>(sm_count(device)) * kMaxCtasPerSm;
}

static size_t workspace_bytes_for(const pa_pool* p, int B, int Hq, int max_blocks, int partition_blocks) {
  if (!p || B <= 0 || Hq <= 0 || max_blocks <= 0 || partition_blocks < 0) return 0;
  if (Hq % p->n_kv_heads) return 0;
  int G = Hq / p->n_kv_heads;
  if (G > PA_MAX_GROUP) return 0;
  size_t rec = sizeof(float) * record_floats(G);
  if (choose_partition(partition_blocks) == 0) return rec * 2 * lean_grid_bound(p->device);
  size_t parts = static_cast<size_t>(B) * p->n_kv_heads *
                 ((max_blocks + partition_blocks - 1) / partition_blocks);
  return rec * parts;
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
  if (sched != SCHED_SEGMENT) {
    if (B > kMaxSplitSeqs) return PA_ERR_UNSUPPORTED;
    size_t need = workspace_bytes_for(p, B, Hq, max_blocks, partition_blocks);
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15)) return PA_ERR_INVALID;
  }
  Params P{};
  P.q = static_cast<const uint16_t*>(q);
  P.k_pool = static_cast<const uint16_t*>(p->k);
  P.v_pool = static_cast<const uint16_t*>(p->v);
  P.k_new = static_cast<const uint16_t*>(k_new);
  P.v_new = static_cast<const uint16_t*>(v_new);
  P.tables = tables;
  P.seq_lens = seq_lens;
  P.out = out;
  P.ws = static_cast<float*>(ws);
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
  return workspace_bytes_for(p, num_seqs, n_q_heads, max_blocks_per_seq, partition_blocks);
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
