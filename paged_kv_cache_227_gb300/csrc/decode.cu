// Paged decode attention for sm_103a.
//
// One query token per sequence attends over its cache, which sits in
// fixed-size 16-token blocks found through a per-sequence block table
// ("Serving", section 23.4 Paged Attention).  Decode reads the whole cache
// for one token per sequence, so it is bound by HBM bandwidth ("Serving",
// section 23.2 Prefill and Decode); the design reads every K/V byte exactly
// once, keeps enough bytes in flight to saturate HBM3e, and keeps the SM's
// instruction issue and its synchronisation well below the memory time.
//
// Work decomposition.  A segment is one (sequence i, kv head h) pair: its
// nb_i = ceil(L_i/16) tiles of 16 tokens x 128 dims (4 KiB each for K and
// for V).  A tile is fetched once and used by all G = Hq/Hkv query heads of
// the group.  The unit of work is one WARP: every warp of the persistent grid
// is an independent pipeline with its own list of pieces (a contiguous range
// of one segment's tiles) given by one of three schedules:
//   SEGMENT    whole segments, strided over warps (no workspace);
//   LEAN       the concatenated tile stream of all segments cut into equal
//              per-warp ranges (even load for any length mix); a segment cut
//              by a range boundary leaves partial results;
//   PARTITION  fixed partitions of `partition_blocks` tiles per segment.
// A piece that does not cover its whole segment writes a partial record
// (running max m, sum l, unnormalised o, fp32); a second kernel, launched as a
// programmatic dependent of this one, merges each cut segment's records by
// log-sum-exp in their fixed order.  Partial records need no fence, atomic or
// counter, so no warp ever stalls on another warp's progress.
//
// Per warp: a private ring of S shared-memory stages.  The warp streams its
// tiles in with TMA tensor loads (one 8 KiB box per tile: the K and the V
// tile, each as two 16-row x 128-byte swizzled halves; completion on an
// mbarrier) and refills a stage the moment it has finished with it.  Per
// tile (software-pipelined: the score product of tile j+1 is issued before
// the value product of tile j):
//   scores  S^T[t][g] = K[t] . q_g with mma.sync m16n8k16 (M = 16 tokens,
//           N = 8 query heads of the group, 8 k-steps of 16 dims, fp32
//           accumulate, 4 independent accumulators); ldmatrix reads the
//           swizzled K tile without bank conflicts;
//   online softmax in fp32 in the log2 domain with a lazily moved running
//           max (rescale only when a new max exceeds the old by 2^8);
//   values  for G <= 4, O^T += V^T P with mma.sync (M = 128 dims in 8
//           m-tiles read by ldmatrix.trans, N = 8 columns holding the high
//           and the low 16-bit halves of each head's weights, so the weights
//           keep ~17 bits; fp32 accumulate); for G > 4, o[g][:] +=
//           p[t][g] V[t][:] in fp32 on the FMA pipes (packed two-wide FMAs).
// Positions t >= L are masked by select in the scores and skipped in the
// values, so padding or stale slots (even NaN) never reach the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstddef>
#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace pa {

constexpr int kMaxSplitSeqs = 4096;  // sequences per split launch (prefix in shared memory)
constexpr int kMaxCtasPerSm = 4;
constexpr int kLeanMinBlocks = 4;    // smallest LEAN range per warp
// LEAN balances cost, not tiles: each (sequence, kv head) segment counts
// kLeanPieceCost extra units ahead of its tiles, the measured cost of
// starting a piece (its q, table window and record) in tile-equivalents, so
// a warp whose range crosses several short segments gets fewer tiles.
constexpr int kLeanPieceCost = 1;
// The same for segments of packed query tokens (16 columns): a piece there
// also costs its 8.7 KB record and a merge of 16 columns; swept 1-20 on the
// batch-64 LLaMA-3-8B layout with 4 new tokens per sequence, 8-20 flat, 12
// best (60.3 us against 71.2 us at 1).
constexpr int kLeanPieceCostPacked = 12;
constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;    // log2 units

enum { SCHED_SEGMENT = 0, SCHED_LEAN = 1, SCHED_PARTITION = 2 };

// Compile-time shape of the kernel: NW warps per CTA, SW ring stages per warp.
template <int G>
struct Shape {
  static constexpr int NW = 2;
  static constexpr int SW = 3;
  static constexpr int kMinCtas = 4;  // CTAs per SM the register budget is sized for
  static constexpr int kThreads = NW * 32;
  static constexpr int PB = G <= 4 ? 4 : 8;  // row stride of the per-warp p buffer
};

struct Params {
  CUtensorMap tmap_kv;      // tile view of the K|V allocation (see pa_pool)
  const uint16_t* q;        // [B][Hq][128]
  const uint16_t* k_pool;   // [N][Hkv][16][128]
  const uint16_t* v_pool;
  const uint16_t* k_new;    // [B][Hkv][128], fused append only
  const uint16_t* v_new;
  const int32_t* tables;    // [rows][max_blocks]
  const int32_t* table_offs;  // [B]: element offset of sequence i's table row, or null (i * max_blocks)
  float* lse;               // [B][Hq] log2-sum-exp of the scaled scores (log2 units), or null
  const int32_t* ext_ntok;  // [B]: query tokens packed in sequence i's columns, or null (1)
  int ext_g;                // columns per packed token (the real group size)
  const int32_t* ext_qbase;  // [B]: q / out row of sequence i's first packed token (its ext_ntok[i]
                             // tokens are the rows that follow), or -1 (none); null: q and out are
                             // [B][Hq][128]
  int ext_hq;                // with ext_qbase: heads of a q / out row ([rows][ext_hq][128])
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
  int lean_units;           // LEAN: number of warps the ranges are cut for
  int lean_cost;            // LEAN: units counted ahead of each segment's tiles
  long long wait_limit_ns;
  int launch_flags;         // kLaunch* (host side; kLaunchSecondary also read by the kernel)
};

// Launch variants of one decode call (host side).  Secondary: the decode is
// the programmatic dependent of the kernel before it in the stream, needs
// nothing that kernel writes, and completes only after it (one thread waits
// for it at the end), so the merge that depends on this decode also sees
// that kernel's writes.  NoMerge / MergeOnly: launch one of the two kernels.
// AfterPlan: the decode is the programmatic dependent of a kernel that writes
// its lengths, table offsets and row maps, and waits for it before reading them.
constexpr int kLaunchSecondary = 1, kLaunchNoMerge = 2, kLaunchMergeOnly = 4, kLaunchAfterPlan = 8;

// Partial record of one piece: the unnormalised output o of its columns in
// C = record_cols(G) columns' room, then m[g] at C*128+g and l[g] at
// C*128+64+g (fp32; m in log2 units of the scaled scores).  o is stored
// o[g][128] by the FMA and 4-column tensor-core paths, and in fragment order
// by the 8-column tensor-core path of the extended kernel (see
// frag_record_index), which writes it with whole-warp 16-byte stores.
__host__ __device__ constexpr int record_cols(int G) { return G <= 4 ? G : (G + 7) / 8 * 8; }
__host__ __device__ constexpr int record_floats(int G) { return (record_cols(G) + 1) * 128; }
// Fragment order: float4 number ((hf*2 + e)*4 + k)*32 + lane holds, for the
// lane's column 8hf + 2(lane%4) + e, dims 32k + lane/4 + {0, 8, 16, 24}.
// Returns that float4's index for column g, and the merge lane ml = 8k + r
// whose dims are 32k + r + {0, 8, 16, 24}.
__host__ __device__ constexpr int frag_record_index(int g, int ml) {
  return (((g >> 3) * 2 + (g & 1)) * 4 + (ml >> 3)) * 32 + 4 * (ml & 7) + ((g & 7) >> 1);
}
// Columns of one segment of packed query tokens (two halves of the MMA's 8).
constexpr int kMaxPackedCols = 16;

// Element offset in q and out of column g of kv head h of a sequence whose
// packed tokens are rows r0 .. r0 + nt - 1 (ext_g columns each), or -1 when
// the column carries no query: column g is token g / ext_g's query head
// h * ext_g + g % ext_g.
__device__ __forceinline__ long long packed_io_offset(const Params& P, int r0, int nt, int h, int g) {
  const int tt = g / P.ext_g;
  if (r0 < 0 || tt >= nt) return -1;
  return (static_cast<long long>(r0 + tt) * P.ext_hq + h * P.ext_g + (g - tt * P.ext_g)) * 128;
}

// ---------------------------------------------------------------------------
// PTX helpers.
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
__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// L2 policy for the K/V stream: evict first, so that the tiles, read once,
// do not push out what is read again (q rows, tables, the partial records
// the merge kernel reads back).
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// TMA tensor load of the 4-D box at (0, y, 0, 0) into shared memory: one
// (block, head) tile of K and of V, with L2 cache policy `pol`.
__device__ __forceinline__ void tma_load_tile(uint32_t dst, const CUtensorMap* map, int y, uint32_t bar,
                                              uint64_t pol) {
  const int z = 0;
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(z), "r"(y), "r"(z), "r"(z), "r"(bar), "l"(pol)
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
// Transpose of an 8x8 16-bit matrix held one 32-bit pair per lane (lane t:
// row t/4, columns 2(t%4), 2(t%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// Two fp32 values as a 16-bit pair (a in the low half), rounded to nearest;
// pack_lo packs what rounding left over, so hi + lo carries a to ~2^-17.
template <bool kBf16>
__device__ __forceinline__ uint32_t pack_hi(float a, float b) {
  if (kBf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <bool kBf16>
__device__ __forceinline__ uint32_t pack_lo(float a, float b) {
  if (kBf16) {
    const float ra = a - __bfloat162float(__float2bfloat16_rn(a));
    const float rb = b - __bfloat162float(__float2bfloat16_rn(b));
    __nv_bfloat162 h = __floats2bfloat162_rn(ra, rb);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  const float ra = a - __half2float(__float2half_rn(a));
  const float rb = b - __half2float(__float2half_rn(b));
  __half2 h = __floats2half2_rn(ra, rb);
  return *reinterpret_cast<uint32_t*>(&h);
}
// D = A B + D for m16n8k16 (fp32 accumulate).
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
// Byte offset of 16-byte chunk c (0..15) of row r in a tile stored as two
// 128-byte-swizzled boxes [16 rows][64 elements] (the TMA 128-byte swizzle
// XORs the chunk index with the row index modulo 8 inside each 1024-byte
// span).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
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

// 16-bit -> fp32 pairs for 8 packed elements (element 2k in .x, 2k+1 in .y).
template <bool kBf16>
__device__ __forceinline__ void unpack8(const uint4& v, float2 f[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (kBf16) {
      f[k] = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
      f[k] = __half22float2(h);
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

// Four consecutive outputs starting at an index that is a multiple of 4.
__device__ __forceinline__ void store_out4(void* out, long long idx, float a, float b, float c, float d,
                                           int out_dtype) {
  if (out_dtype == PA_FP32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = make_float4(a, b, c, d);
  } else if (out_dtype == PA_BF16) {
    __nv_bfloat162 h0 = __floats2bfloat162_rn(a, b), h1 = __floats2bfloat162_rn(c, d);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) =
        make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
  } else {
    __half2 h0 = __floats2half2_rn(a, b), h1 = __floats2half2_rn(c, d);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) =
        make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
  }
}

// Eight consecutive outputs starting at an index that is a multiple of 8.
__device__ __forceinline__ void store_out8(void* out, long long idx, const float v[8], int out_dtype) {
  if (out_dtype == PA_FP32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (out_dtype == PA_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&h);
      } else {
        __half2 h = __floats2half2_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
  }
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
  const long long num = static_cast<long long>(P.Hkv) * pfx[P.B] + P.lean_units - 1;
  const long long per = num < 0x7fffffffll ? static_cast<int>(num) / P.lean_units : num / P.lean_units;
  return per < kLeanMinBlocks ? kLeanMinBlocks : per;
}

// ---------------------------------------------------------------------------
// Piece enumeration for one warp (unit u of n_units): the warp walks the
// same list twice, once to issue its loads and once to consume them.
// ---------------------------------------------------------------------------
struct Piece {
  int i, h, j0, j1, L;
  bool final_out;
  long long rec;  // partial record index (when !final_out)
};

struct PieceIter {
  const Params& P;
  const int* pfx;   // shared: exclusive prefix over sequences (LEAN: units = tiles + lean_cost per
                    // segment, PARTITION: partitions)
  const int* lens;  // shared: clamped lengths (split schedules), or null (read from P.seq_lens)
  int unit, n_units;
  long long x, x_end;        // SEGMENT / PARTITION cursor
  long long cur, end;        // LEAN cursor (units)
  int li, lh;
  bool first;

  __device__ PieceIter(const Params& p, const int* prefix, const int* lengths, int u, int nu)
      : P(p), pfx(prefix), lens(lengths), unit(u), n_units(nu) {
    first = true;
    if (P.sched == SCHED_LEAN) {
      long long T = static_cast<long long>(P.Hkv) * pfx[P.B];
      long long per = lean_per(P, pfx);
      cur = per * unit;
      end = cur + per < T ? cur + per : T;
      if (cur < end) {
        // largest i with Hkv*pfx[i] <= cur (never an empty sequence)
        int lo = 0, hi = P.B - 1;
        while (lo < hi) {
          int mid = (lo + hi + 1) >> 1;
          if (static_cast<long long>(P.Hkv) * pfx[mid] <= cur) lo = mid; else hi = mid - 1;
        }
        li = lo;
        const int cnt = pfx[li + 1] - pfx[li];
        lh = static_cast<int>((cur - static_cast<long long>(P.Hkv) * pfx[li]) / cnt);
      }
    } else {
      x = unit;
      x_end = P.sched == SCHED_SEGMENT ? static_cast<long long>(P.B) * P.Hkv
                                       : static_cast<long long>(P.Hkv) * pfx[P.B];
    }
  }

  __device__ int len(int i) const { return lens ? lens[i] : clamp_len(P, i); }

  __device__ bool next(Piece& pc) {
    if (P.sched == SCHED_LEAN) {
      if (cur >= end) return false;
      // segment (li, lh): units [seg_start, seg_end), its tiles from rs on
      const int cnt = pfx[li + 1] - pfx[li];
      const long long seg_start = static_cast<long long>(P.Hkv) * pfx[li] + static_cast<long long>(lh) * cnt;
      const long long rs = seg_start + P.lean_cost, seg_end = seg_start + cnt;
      if (end <= rs) {  // the range ends before this segment's tiles
        cur = end;
        return false;
      }
      const long long from = cur > rs ? cur : rs;
      const long long pend = end < seg_end ? end : seg_end;
      pc.i = li;
      pc.h = lh;
      pc.j0 = static_cast<int>(from - rs);
      pc.j1 = static_cast<int>(pend - rs);
      pc.L = len(li);
      pc.final_out = (from == rs && pend == seg_end);
      pc.rec = 2ll * unit + (first ? 0 : 1);
      first = false;
      cur = pend;
      if (cur == seg_end && ++lh == P.Hkv) {
        lh = 0;
        do { ++li; } while (li < P.B && pfx[li + 1] == pfx[li]);
      }
      return true;
    }
    if (x >= x_end) return false;
    if (P.sched == SCHED_SEGMENT) {
      pc.i = static_cast<int>(x / P.Hkv);
      pc.h = static_cast<int>(x - static_cast<long long>(pc.i) * P.Hkv);
      pc.L = len(pc.i);
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
      pc.L = len(lo);
      int nb = (pc.L + kBlock - 1) / kBlock;
      int p = static_cast<int>(u - pfx[lo]);
      pc.j0 = p * P.partition_blocks;
      pc.j1 = pc.j0 + P.partition_blocks < nb ? pc.j0 + P.partition_blocks : nb;
      pc.final_out = (pfx[lo + 1] - pfx[lo]) == 1;
      pc.rec = x;
    }
    x += n_units;
    return true;
  }
};

// Records of segment (i, h): how many, and the index of the k-th.
struct SegmentRecords {
  long long c0, s0, per, base;
  int count;
  __device__ SegmentRecords(const Params& P, const int* pfx, int i, int h) {
    if (P.sched == SCHED_LEAN) {
      const int cnt = pfx[i + 1] - pfx[i];
      const int nb = cnt - P.lean_cost;
      per = lean_per(P, pfx);
      s0 = static_cast<long long>(P.Hkv) * pfx[i] + static_cast<long long>(h) * cnt;  // segment's units start
      const long long rs = s0 + P.lean_cost;                                          // its tiles start
      const long long last = rs + nb - 1;
      if (last < 0x7fffffffll && per < 0x7fffffffll) {
        c0 = static_cast<int>(rs) / static_cast<int>(per);
        count = static_cast<int>(last) / static_cast<int>(per) - static_cast<int>(c0) + 1;
      } else {
        c0 = rs / per;
        count = static_cast<int>(last / per - c0 + 1);
      }
      base = 0;
    } else {
      count = pfx[i + 1] - pfx[i];
      base = static_cast<long long>(pfx[i]) * P.Hkv + h;
      c0 = s0 = per = 0;
    }
  }
  __device__ long long at(const Params& P, int k) const {
    // warp c0 holds an earlier piece (the previous segment's tiles end at
    // s0) when its range starts before s0: then this is its second record
    if (P.sched == SCHED_LEAN) return 2 * (c0 + k) + ((k == 0 && s0 > c0 * per) ? 1 : 0);
    return base + static_cast<long long>(k) * P.Hkv;
  }
};

// Exclusive prefix over sequences of the per-sequence counts (tiles for
// LEAN, partitions for PARTITION) into pfx[0..B], and, when lens is given, the
// clamped lengths into lens[0..B).  All threads of the block load the
// lengths; warp 0 scans.  Ends with a block barrier.
__device__ void block_prefix(const Params& P, int* pfx, int* lens, bool report, int* rows = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cap = P.max_blocks * kBlock;
  for (int i = threadIdx.x; i < P.B; i += blockDim.x) {
    int L = P.seq_lens[i];
    if (L < 0 || L > cap) {
      if (report) record_error(P.err, PA_ERR_DEVICE_CHECK, static_cast<long long>(L));
      L = L < 0 ? 0 : cap;
    }
    if (lens) lens[i] = L;
    if (rows) {
      rows[i] = P.table_offs[i];
      rows[P.B + i] = P.ext_ntok ? P.ext_ntok[i] : 1;
      rows[2 * P.B + i] = P.ext_qbase ? P.ext_qbase[i] : -1;
    }
    const int nb = (L + kBlock - 1) / kBlock;
    pfx[i + 1] = P.sched == SCHED_LEAN ? (nb ? nb + P.lean_cost : 0)
                                       : (nb + P.partition_blocks - 1) / P.partition_blocks;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < P.B; base += 32) {
      const int i = base + lane;
      const int c = i < P.B ? pfx[i + 1] : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      __syncwarp();
      if (i < P.B) pfx[i + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pfx[0] = 0;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Shared memory.  The rings come first at a 1024-byte aligned base (the
// 128-byte swizzle of TMA boxes needs it); p buffers are 16-byte aligned.
// ---------------------------------------------------------------------------
template <int G>
struct __align__(1024) Smem {
  static constexpr int NW = Shape<G>::NW;
  static constexpr int SW = Shape<G>::SW;
  uint8_t stage[NW][SW][kStageBytes];
  __align__(16) float pbuf[NW][kBlock][Shape<G>::PB];
  __align__(8) unsigned long long full[NW][SW];
  int stage_blk[NW][SW];
  int abort_flag;
  int pfx[1];  // dynamic tail: prefix [B + 1], then clamped lengths [B]
};

template <int G>
constexpr bool smem_layout_ok() {
  return offsetof(Smem<G>, stage) == 0 && offsetof(Smem<G>, pbuf) % 16 == 0 &&
         offsetof(Smem<G>, full) % 8 == 0 && kStageBytes % 1024 == 0;
}
static_assert(smem_layout_ok<1>() && smem_layout_ok<2>() && smem_layout_ok<3>() &&
                  smem_layout_ok<4>() && smem_layout_ok<5>() && smem_layout_ok<6>() &&
                  smem_layout_ok<7>() && smem_layout_ok<8>() && smem_layout_ok<16>(),
              "shared-memory layout breaks a swizzle, vector or mbarrier alignment");

// Dynamic shared memory to request: the struct, the prefix array, and slack
// to align the base to 1024 bytes.
template <int G>
constexpr size_t smem_bytes(int B, bool rows = false) {
  return sizeof(Smem<G>) + sizeof(int) * static_cast<size_t>((rows ? 5 : 2) * B + 1) + 1024;
}

// ---------------------------------------------------------------------------
// The decode kernel.
// ---------------------------------------------------------------------------
template <int G, bool kBf16, bool kFused, bool kExt>
__global__ void __launch_bounds__(Shape<G>::kThreads, Shape<G>::kMinCtas) decode_kernel(const __grid_constant__ Params P) {
  constexpr int NW = Shape<G>::NW;
  constexpr int SW = Shape<G>::SW;
  constexpr int PB = Shape<G>::PB;
  extern __shared__ uint8_t smem_raw[];
  Smem<G>& S = *reinterpret_cast<Smem<G>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // --- set-up: barriers, prefix over sequences -----------------------------
  if (threadIdx.x == 0) {
    for (int w = 0; w < NW; ++w)
      for (int s = 0; s < SW; ++s) mbar_init(smem_addr(&S.full[w][s]), 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // tail of shared memory: prefix [B+1], lengths [B], and (kExt) per sequence
  // its table offset [B], packed tokens [B] and first q / out row [B]
  int* const S_rows = kExt ? S.pfx + 2 * P.B + 1 : nullptr;
  // (a planning kernel before this one writes the lengths and maps read here)
  if (kExt && (P.launch_flags & kLaunchAfterPlan)) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (P.sched != SCHED_SEGMENT) block_prefix(P, S.pfx, S.pfx + P.B + 1, blockIdx.x == 0, S_rows);
  // element offset of column g of kv head h of sequence i in q and out, or -1
  auto io_at = [&](int i, int h, int g) -> long long {
    if (kExt && P.ext_qbase) return packed_io_offset(P, S_rows[2 * P.B + i], S_rows[P.B + i], h, g);
    return (static_cast<long long>(i) * P.Hq + h * G + g) * kHeadDim;
  };
  // a dependent launch that follows (the merge kernel, or the prefix pass
  // of a cascade) may start its own set-up now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // zero rows of empty sequences (split schedules; SEGMENT pieces write them)
  if (P.sched != SCHED_SEGMENT) {
    for (int i = blockIdx.x; i < P.B; i += gridDim.x) {
      if (S.pfx[i + 1] != S.pfx[i]) continue;
      if constexpr (kExt) {
        if (P.ext_qbase && S_rows[2 * P.B + i] < 0) continue;  // a packed slot with no query rows
        // one warp per column; columns that carry no query are skipped
        for (int col = warp; col < P.Hq; col += NW) {
          const long long at = io_at(i, col / G, col % G);
          if (at < 0) continue;
          for (int d = lane; d < kHeadDim; d += 32) store_out(P.out, at + d, 0.f, P.out_dtype);
        }
      } else {
        for (int x = threadIdx.x; x < P.Hq * kHeadDim; x += blockDim.x)
          store_out(P.out, static_cast<long long>(i) * P.Hq * kHeadDim + x, 0.f, P.out_dtype);
      }
      if (kExt && P.lse)
        for (int x = threadIdx.x; x < P.Hq; x += blockDim.x) P.lse[static_cast<long long>(i) * P.Hq + x] = -INFINITY;
    }
  }

  volatile int* abort_flag = &S.abort_flag;
  const int* S_lens = P.sched != SCHED_SEGMENT ? S.pfx + P.B + 1 : nullptr;
  const int unit = blockIdx.x * NW + warp;
  const int n_units = gridDim.x * NW;
  uint8_t* ring = S.stage[warp][0];
  const uint32_t ring_addr = smem_addr(ring);
  const uint32_t full0 = smem_addr(&S.full[warp][0]);

  // MMA fragment coordinates: row group r4 = lane / 4, column pair c4.
  //   scores S^T[t][g]: rows t = r4, r4 + 8 (tokens), columns g = 2*c4, +1
  const int r4 = lane >> 2;
  const int c4 = lane & 3;
  const int g0 = 2 * c4;
  // ldmatrix: lane group lm supplies matrix lm, row lr: [tok 0-7 | 8-15] x [chunk +0 | +1]
  const int lm = lane >> 3, lr = lane & 7;
  const int k_tok = lr + 8 * (lm & 1), k_cadd = lm >> 1;
  // ldmatrix.trans of V^T: matrix lm covers tokens 8*(lm/2).. and dims 8*(lm%2).. of an m-tile
  const int v_tok = lr + 8 * (lm >> 1), v_cadd = lm & 1;
  // Value product.  Mode 1 (G <= 4): tensor cores, the high and low weight
  // halves of all heads in the 8 columns of one m16n8k16 product.  Mode 2
  // (G > 4, extended kernel): tensor cores, the high halves and the low
  // halves in one product each.  Mode 0 (G > 4): packed fp32 FMAs, measured
  // faster than mode 2 for the plain decode of G = 6.
  constexpr int kPvMode = G <= 4 ? 1 : (kExt ? 2 : 0);
  constexpr bool kMmaPv = kPvMode != 0;
  // Column halves: the extended kernel takes up to 16 columns as two groups
  // of 8 (the MMA's n), which share each K/V tile, its wait and its operand
  // loads.  kSc: independent score accumulators per half.
  constexpr int NCH = G > 8 ? 2 : 1;
  constexpr int kSc = NCH == 1 ? 4 : 2;
  static_assert(G <= 8 || kPvMode == 2, "more than 8 columns only in the extended kernel");
  // value phase: lane owns 16-byte chunk c16 of the V rows of token parity r16
  const int c16 = lane & 15;
  const int r16 = lane >> 4;

  // ---- issue side: walks the piece list SW tiles ahead of the consumer.
  // Block ids come from 32-entry windows of a piece's table row held one per
  // lane; the window after the current one (the rest of this piece, or the
  // first of the next piece) is already being loaded, so an issue never waits
  // on the table.  Entering a piece also prefetches the piece after it's q
  // rows (and new K/V rows) into L2.
  const uint64_t kv_policy = evict_first_policy();
  PieceIter iss(P, S.pfx, S_lens, unit, n_units);
  PieceIter cit = iss;  // the consumer walks the same list
  Piece ip, inx;  // current and next piece of the issue side
  bool ihave = iss.next(ip);
  bool inx_have = ihave && iss.next(inx);
  int ij = ihave ? ip.j0 : 0;
  int tb_base = ij, tb_val = 0, tb_nv = 0;
  int n_issued = 0;
  bool append_seen = false;  // fused step: the append grid has completed
  auto window = [&](const Piece& pp, int base) -> int {
    const int jj = base + lane;
    const long long off = kExt ? static_cast<long long>(S_rows[pp.i]) : static_cast<long long>(pp.i) * P.max_blocks;
    return jj < pp.j1 ? P.tables[off + jj] : 0;
  };
  auto prefetch_rows = [&](const Piece& pp) {
    if constexpr (kExt) {
      if (lane < 2 * G) {
        const long long at = io_at(pp.i, pp.h, lane >> 1);
        if (at >= 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(P.q + at + 64 * (lane & 1)));
      }
    } else {
      const long long qrow = (static_cast<long long>(pp.i) * P.Hq + pp.h * G) * kHeadDim;
      if (lane < 2 * G) asm volatile("prefetch.global.L2 [%0];" ::"l"(P.q + qrow + 64 * lane));
    }
  };
  auto load_following = [&]() {
    if (tb_base + 32 < ip.j1) {
      tb_nv = window(ip, tb_base + 32);
    } else if (inx_have) {
      tb_nv = window(inx, inx.j0);
      prefetch_rows(inx);
    }
  };
  if (ihave) {
    tb_val = window(ip, ij);
    load_following();
  }
  auto issue = [&](int stage) {
    while (ihave && ij >= ip.j1) {  // enter the next piece: its first window is tb_nv
      ip = inx;
      ihave = inx_have;
      if (!ihave) return;
      inx_have = iss.next(inx);
      ij = ip.j0;
      tb_base = ij;
      tb_val = tb_nv;
      load_following();
    }
    if (!ihave) return;
    if (ij - tb_base >= 32) {  // the next window of the same piece
      tb_base += 32;
      tb_val = tb_nv;
      load_following();
    }
    const int blk = __shfl_sync(0xffffffffu, tb_val, ij - tb_base);
    if (kFused && !append_seen && ij == (ip.L + kBlock - 1) / kBlock - 1) {
      // the sequence's last tile holds its new token, which the append grid
      // (this grid's programmatic prerequisite) writes: wait for it once
      asm volatile("griddepcontrol.wait;" ::: "memory");
      append_seen = true;
    }
    if (lane == 0) {
      const bool valid = blk >= 0 && blk < P.num_blocks;
      S.stage_blk[warp][stage] = valid ? blk : -1;
      const uint32_t fb = full0 + 8 * stage;
      if (valid) {
        mbar_arrive_expect_tx(fb, kStageBytes);
        const int y = (blk * P.Hkv + ip.h) * kBlock;  // first token row of the tile
        tma_load_tile(ring_addr + stage * kStageBytes, &P.tmap_kv, y, fb, kv_policy);
      } else {
        record_error(P.err, PA_ERR_DEVICE_CHECK, static_cast<long long>(blk));
        mbar_arrive(fb);
      }
    }
    ++ij;
    ++n_issued;
  };
  // ---- consume side -----------------------------------------------------------
  Piece pc;
  bool have_pc = cit.next(pc);
  // B fragments of Q^T: column g = 8 hf + r4 of the group (zero past G), k = dims
  uint32_t qb[NCH][8][2];
  auto load_q = [&]() {
#pragma unroll
    for (int hf = 0; hf < NCH; ++hf) {
      const int col = 8 * hf + r4;
      long long at;
      if constexpr (kExt)
        at = col < G ? io_at(pc.i, pc.h, col) : -1;
      else
        at = col < G ? (static_cast<long long>(pc.i) * P.Hq + pc.h * G + col) * kHeadDim : -1;
      if (at >= 0) {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(P.q + at);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          qb[hf][ks][0] = qrow[8 * ks + c4];
          qb[hf][ks][1] = qrow[8 * ks + 4 + c4];
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) qb[hf][ks][0] = qb[hf][ks][1] = 0u;
      }
    }
  };
  if (have_pc) load_q();  // in flight while the first loads are issued
#pragma unroll 1
  for (int s = 0; s < SW; ++s) issue(s);

  int n = 0;  // tiles consumed by this warp
  bool ok = true;
  float (*pb)[PB] = S.pbuf[warp];
  while (ok && have_pc) {
    // value accumulators.  Tensor-core path (G <= 4): oc[mt] is the m16n8
    // fragment of O^T for dims 16mt..16mt+15: this lane holds dims 16mt+r4
    // and 16mt+r4+8 of columns 2c4, 2c4+1, where columns 0-3 accumulate the
    // high halves and columns 4-7 the low halves of the weights of heads 0-3.
    // FMA path (G > 4): o[g][e] holds dims 8*c16+2e, +1 of head g over the
    // tokens of parity r16.
    // Mode 2: oc[hf] holds the products with the high halves of the 8
    // columns of half hf (columns 8hf + 2c4, +1 for this lane), oc2 those
    // with the low halves; with two halves both go into oc (registers).
    constexpr bool kLoApart = kPvMode == 2 && NCH == 1;
    float oc[NCH][kMmaPv ? 8 : 1][4];
    float oc2[kLoApart ? 8 : 1][4];
    float2 o[kMmaPv ? 1 : G][4];
#pragma unroll
    for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
      for (int mt = 0; mt < (kMmaPv ? 8 : 1); ++mt) oc[hf][mt][0] = oc[hf][mt][1] = oc[hf][mt][2] = oc[hf][mt][3] = 0.f;
#pragma unroll
    for (int mt = 0; mt < (kLoApart ? 8 : 1); ++mt) oc2[mt][0] = oc2[mt][1] = oc2[mt][2] = oc2[mt][3] = 0.f;
#pragma unroll
    for (int g = 0; g < (kMmaPv ? 1 : G); ++g)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[g][e] = make_float2(0.f, 0.f);
    float m_run[NCH][2], l_run[NCH][2];
#pragma unroll
    for (int hf = 0; hf < NCH; ++hf) {
      m_run[hf][0] = m_run[hf][1] = -INFINITY;
      l_run[hf][0] = l_run[hf][1] = 0.f;
    }
    const int nb_total = (pc.L + kBlock - 1) / kBlock;
    // extended kernel: the sequence packs ntok query tokens, ext_g columns
    // each; token t of them sees ntok - 1 - t fewer positions (causal).
    // cut[hf][c]: positions column 8hf + g0 + c does not see.
    int cut[NCH][2];
#pragma unroll
    for (int hf = 0; hf < NCH; ++hf) cut[hf][0] = cut[hf][1] = 0;
    if constexpr (kExt) {
      const int nt = S_rows[P.B + pc.i];
      if (nt > 1) {
#pragma unroll
        for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int x = nt - 1 - (8 * hf + g0 + c) / P.ext_g;
            cut[hf][c] = x < 0 ? 0 : x;
          }
      }
    }

    // prepare(): wait for the tile's stage, read its block id, and on the
    // tensor-core path clear the V rows past the sequence's end (0 x NaN would
    // poison the product; the weights there are exactly zero).
    auto prepare = [&](int jj, int nn, int& blk_out, bool& touched_out) -> bool {
      const int s = nn % SW;
      const uint32_t parity = static_cast<uint32_t>((nn / SW) & 1);
      bool got = wait_phase(full0 + 8 * s, parity, abort_flag, P.wait_limit_ns, P.err, 2);
      got = __all_sync(0xffffffffu, got);
      touched_out = false;
      blk_out = -1;
      if (!got) return false;
      const int blk = S.stage_blk[warp][s];
      blk_out = blk;
      if (blk >= 0 && jj == nb_total - 1) {
        uint8_t* Ks = ring + s * kStageBytes;
        const int valid = pc.L - jj * kBlock;
        if (kMmaPv && valid < kBlock) {
          for (int x = valid * 16 + lane; x < kBlock * 16; x += 32)
            *reinterpret_cast<uint4*>(Ks + kTileBytes + swz(x >> 4, x & 15)) = make_uint4(0u, 0u, 0u, 0u);
          touched_out = true;
        }
        if (touched_out) __syncwarp();
      }
      return true;
    };
    // S^T = K Q^T for the tile in stage s, in kSc independent accumulators
    // per half (each K fragment serves both halves)
    auto scores = [&](int s, float (&acc)[NCH][kSc][4]) {
      const uint32_t ks_addr = ring_addr + s * kStageBytes;
#pragma unroll
      for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
        for (int c = 0; c < kSc; ++c) acc[hf][c][0] = acc[hf][c][1] = acc[hf][c][2] = acc[hf][c][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ks_addr + swz(k_tok, 2 * ks + k_cadd), a0, a1, a2, a3);
#pragma unroll
        for (int hf = 0; hf < NCH; ++hf)
          mma16816<kBf16>(acc[hf][ks % kSc], a0, a1, a2, a3, qb[hf][ks][0], qb[hf][ks][1]);
      }
    };

    float acc[NCH][kSc][4];
    int cur_blk = -1;
    bool cur_touched = false;
    if (pc.j1 > pc.j0) {
      if (!prepare(pc.j0, n, cur_blk, cur_touched))
        ok = false;
      else if (cur_blk >= 0)
        scores(n % SW, acc);
    }
    for (int j = pc.j0; ok && j < pc.j1; ++j) {
      const int s = n % SW;
      const uint8_t* Vs = ring + s * kStageBytes + kTileBytes;
      const int valid_tokens = pc.L - j * kBlock < kBlock ? pc.L - j * kBlock : kBlock;
      float p[NCH][4];
      if (cur_blk >= 0) {
        float st[NCH][4];
#pragma unroll
        for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if constexpr (kSc == 4)
              st[hf][c] = (acc[hf][0][c] + acc[hf][1][c]) + (acc[hf][2][c] + acc[hf][3][c]);
            else
              st[hf][c] = acc[hf][0][c] + acc[hf][1][c];
          }
        // ---- online softmax of columns 8hf + g0, +1 over tokens r4, r4+8.
        // Each lane checks its own scores against the running max; only when
        // one of them exceeds it by more than 2^8 does the warp reduce the
        // tile's column maxima and move the running max (rare after the first
        // tile).
        float mx[NCH][2];
        bool grow = false;
#pragma unroll
        for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            // (rows past a column's last position; the cut can reach into the
            // tile before the last one)
            const int vt = kExt ? pc.L - j * kBlock - cut[hf][c] : valid_tokens;
            st[hf][c] = r4 < vt ? st[hf][c] * P.qscale : -INFINITY;
            st[hf][2 + c] = r4 + 8 < vt ? st[hf][2 + c] * P.qscale : -INFINITY;
            mx[hf][c] = fmaxf(st[hf][c], st[hf][2 + c]);
            grow = grow || mx[hf][c] > m_run[hf][c] + kRescaleThreshold;
          }
        if (__any_sync(0xffffffffu, grow)) {  // warp-uniform
#pragma unroll
          for (int hf = 0; hf < NCH; ++hf) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int msk = 4; msk < 32; msk <<= 1)
                mx[hf][c] = fmaxf(mx[hf][c], __shfl_xor_sync(0xffffffffu, mx[hf][c], msk));
            float alpha[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const float mn = fmaxf(m_run[hf][c], mx[hf][c]);
              // (extended kernel: a column with no position seen yet stays at
              // -inf and keeps its zero state)
              alpha[c] = kExt && mn == -INFINITY ? 1.f : fast_exp2(m_run[hf][c] - mn);
              l_run[hf][c] *= alpha[c];
              m_run[hf][c] = mn;
            }
            if constexpr (kPvMode == 1) {
              // columns 4-7 (low halves) belong to the heads of lane c4 - 2
              const float x0 = __shfl_xor_sync(0xffffffffu, alpha[0], 2);
              const float x1 = __shfl_xor_sync(0xffffffffu, alpha[1], 2);
              const float a0 = c4 < 2 ? alpha[0] : x0, a1 = c4 < 2 ? alpha[1] : x1;
#pragma unroll
              for (int mt = 0; mt < 8; ++mt) {
                oc[hf][mt][0] *= a0;
                oc[hf][mt][1] *= a1;
                oc[hf][mt][2] *= a0;
                oc[hf][mt][3] *= a1;
              }
            } else if constexpr (kPvMode == 2) {
#pragma unroll
              for (int mt = 0; mt < 8; ++mt) {
                oc[hf][mt][0] *= alpha[0];
                oc[hf][mt][1] *= alpha[1];
                oc[hf][mt][2] *= alpha[0];
                oc[hf][mt][3] *= alpha[1];
                if constexpr (kLoApart) {
                  oc2[mt][0] *= alpha[0];
                  oc2[mt][1] *= alpha[1];
                  oc2[mt][2] *= alpha[0];
                  oc2[mt][3] *= alpha[1];
                }
              }
            } else {
#pragma unroll
              for (int g = 0; g < (kMmaPv ? 1 : G); ++g) {
                const float al = __shfl_sync(0xffffffffu, alpha[g & 1], g >> 1);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  o[g][e].x *= al;
                  o[g][e].y *= al;
                }
              }
            }
          }
        }
#pragma unroll
        for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // (extended kernel: a column may see no position of a piece yet)
            p[hf][k] = kExt && st[hf][k] == -INFINITY ? 0.f : fast_exp2(st[hf][k] - m_run[hf][k & 1]);
            l_run[hf][k & 1] += p[hf][k];
          }
        if constexpr (!kMmaPv) {
          if (g0 < G) {
            pb[r4][g0] = p[0][0];
            pb[r4 + 8][g0] = p[0][2];
          }
          if (g0 + 1 < G) {
            pb[r4][g0 + 1] = p[0][1];
            pb[r4 + 8][g0 + 1] = p[0][3];
          }
          __syncwarp();
        }
      }
      // ---- next tile: wait for it and issue its score product now
      int nxt_blk = -1;
      bool nxt_touched = false;
      float acc2[NCH][kSc][4];
      if (j + 1 < pc.j1) {
        if (!prepare(j + 1, n + 1, nxt_blk, nxt_touched))
          ok = false;
        else if (nxt_blk >= 0)
          scores((n + 1) % SW, acc2);
      }
      if (cur_blk >= 0) {
        if constexpr (kPvMode == 2) {
          // ---- O^T += V^T P on the tensor cores, 8 columns per half: the
          // high 16-bit halves of the weights in one product, the low halves
          // in another; each V fragment serves both halves
          uint32_t bh[NCH][2], bl[NCH][2];
#pragma unroll
          for (int hf = 0; hf < NCH; ++hf) {
            bh[hf][0] = movmatrix_trans(pack_hi<kBf16>(p[hf][0], p[hf][1]));
            bh[hf][1] = movmatrix_trans(pack_hi<kBf16>(p[hf][2], p[hf][3]));
            bl[hf][0] = movmatrix_trans(pack_lo<kBf16>(p[hf][0], p[hf][1]));
            bl[hf][1] = movmatrix_trans(pack_lo<kBf16>(p[hf][2], p[hf][3]));
          }
          const uint32_t vs_addr = smem_addr(Vs);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(vs_addr + swz(v_tok, 2 * mt + v_cadd), a0, a1, a2, a3);
#pragma unroll
            for (int hf = 0; hf < NCH; ++hf) {
              mma16816<kBf16>(oc[hf][mt], a0, a1, a2, a3, bh[hf][0], bh[hf][1]);
              if constexpr (kLoApart)
                mma16816<kBf16>(oc2[mt], a0, a1, a2, a3, bl[hf][0], bl[hf][1]);
              else
                mma16816<kBf16>(oc[hf][mt], a0, a1, a2, a3, bl[hf][0], bl[hf][1]);
            }
          }
        } else if constexpr (kPvMode == 1) {
          // ---- O^T += V^T P on the tensor cores.  B operand: the weights as
          // a 16-token x 8-column matrix (columns 0-3: high 16-bit halves of
          // heads 0-3, columns 4-7: the low halves, so hi + lo carries p to
          // about 2^-17), transposed from the score fragment by movmatrix.
          const float x0 = __shfl_xor_sync(0xffffffffu, p[0][0], 2);
          const float x1 = __shfl_xor_sync(0xffffffffu, p[0][1], 2);
          const float x2 = __shfl_xor_sync(0xffffffffu, p[0][2], 2);
          const float x3 = __shfl_xor_sync(0xffffffffu, p[0][3], 2);
          const uint32_t w01 = c4 < 2 ? pack_hi<kBf16>(p[0][0], p[0][1]) : pack_lo<kBf16>(x0, x1);
          const uint32_t w23 = c4 < 2 ? pack_hi<kBf16>(p[0][2], p[0][3]) : pack_lo<kBf16>(x2, x3);
          const uint32_t b0 = movmatrix_trans(w01), b1 = movmatrix_trans(w23);
          const uint32_t vs_addr = smem_addr(Vs);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(vs_addr + swz(v_tok, 2 * mt + v_cadd), a0, a1, a2, a3);
            mma16816<kBf16>(oc[0][mt], a0, a1, a2, a3, b0, b1);
          }
        } else if (valid_tokens == kBlock) {  // ---- o += p V on the FMA pipes, full tile
          uint4 raw[kBlock / 2];
          float pp[kBlock / 2][PB];
#pragma unroll
          for (int k = 0; k < kBlock / 2; ++k) {
            const int t = 2 * k + r16;
            raw[k] = *reinterpret_cast<const uint4*>(Vs + swz(t, c16));
#pragma unroll
            for (int g4 = 0; g4 < PB; g4 += 4) {
              float4 q4 = *reinterpret_cast<const float4*>(&pb[t][g4]);
              pp[k][g4] = q4.x; pp[k][g4 + 1] = q4.y; pp[k][g4 + 2] = q4.z; pp[k][g4 + 3] = q4.w;
            }
          }
#pragma unroll
          for (int k = 0; k < kBlock / 2; ++k) {
            float2 vf[4];
            unpack8<kBf16>(raw[k], vf);
#pragma unroll
            for (int g = 0; g < (kMmaPv ? 1 : G); ++g) {
              const float2 p2 = make_float2(pp[k][g], pp[k][g]);
#pragma unroll
              for (int e = 0; e < 4; ++e) o[g][e] = __ffma2_rn(p2, vf[e], o[g][e]);
            }
          }
        } else {  // the sequence's last tile: skip the rows past its end
#pragma unroll
          for (int k = 0; k < kBlock / 2; ++k) {
            const int t = 2 * k + r16;
            if (t < valid_tokens) {
              uint4 raw = *reinterpret_cast<const uint4*>(Vs + swz(t, c16));
              float2 vf[4];
              unpack8<kBf16>(raw, vf);
              float pp[PB];
#pragma unroll
              for (int g4 = 0; g4 < PB; g4 += 4) {
                float4 q4 = *reinterpret_cast<const float4*>(&pb[t][g4]);
                pp[g4] = q4.x; pp[g4 + 1] = q4.y; pp[g4 + 2] = q4.z; pp[g4 + 3] = q4.w;
              }
#pragma unroll
              for (int g = 0; g < (kMmaPv ? 1 : G); ++g) {
                const float2 p2 = make_float2(pp[g], pp[g]);
#pragma unroll
                for (int e = 0; e < 4; ++e) o[g][e] = __ffma2_rn(p2, vf[e], o[g][e]);
              }
            }
          }
        }
      }
      __syncwarp();  // every lane is done with the stage and with pb
      if (cur_touched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(s);      // refill the stage just freed
      ++n;
      cur_blk = nxt_blk;
      cur_touched = nxt_touched;
#pragma unroll
      for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
        for (int c = 0; c < kSc; ++c)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[hf][c][e] = acc2[hf][c][e];
    }
    if (!ok) break;

    // ---- finish the piece: per-head m and l, then the output row or a
    // partial record
    float lsum[NCH][2];
#pragma unroll
    for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        lsum[hf][c] = l_run[hf][c];
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) lsum[hf][c] += __shfl_xor_sync(0xffffffffu, lsum[hf][c], msk);
      }
    // column g = 8hf + gg sits in lane gg / 2 of half hf
    float mg[G], lg[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mg[g] = __shfl_sync(0xffffffffu, m_run[g >> 3][g & 1], (g & 7) >> 1);
      lg[g] = __shfl_sync(0xffffffffu, lsum[g >> 3][g & 1], (g & 7) >> 1);
    }
    const long long row0 = (static_cast<long long>(pc.i) * P.Hq + pc.h * G) * kHeadDim;
    float* rec = P.ws + pc.rec * record_floats(G);
    if (kExt && P.lse && pc.final_out && lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g)
        P.lse[static_cast<long long>(pc.i) * P.Hq + pc.h * G + g] = lg[g] > 0.f ? mg[g] + __log2f(lg[g]) : -INFINITY;
    }
    if constexpr (kPvMode == 2) {
      // o = high + low products; lane c4 holds columns 8hf + 2c4, +1 at
      // dims 16mt+r4 (entries 0, 1) and 16mt+r4+8 (entries 2, 3)
      auto ov = [&](int hf, int mt, int j) {
        return oc[hf][mt][j] + (kLoApart ? oc2[mt][j] : 0.f);
      };
      if (!pc.final_out) {
        // a partial record in fragment order: per (hf, e, k) one 16-byte
        // store per lane, 512 contiguous bytes per warp
        float4* rec4 = reinterpret_cast<float4*>(rec);
#pragma unroll
        for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              rec4[((hf * 2 + e) * 4 + k) * 32 + lane] =
                  make_float4(ov(hf, 2 * k, e), ov(hf, 2 * k, 2 + e), ov(hf, 2 * k + 1, e), ov(hf, 2 * k + 1, 2 + e));
      }
#pragma unroll
      for (int hf = 0; hf < NCH; ++hf)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int g = 8 * hf + 2 * c4 + e;
          if (pc.final_out && g < G) {
            float lgg = lg[0];
#pragma unroll
            for (int gg = 1; gg < G; ++gg)
              if (g == gg) lgg = lg[gg];
            const float inv = lgg > 0.f ? 1.f / lgg : 0.f;
            const long long orow = io_at(pc.i, pc.h, g);
            if (orow >= 0) {
#pragma unroll
              for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                  store_out(P.out, orow + 16 * mt + r4 + 8 * hh, ov(hf, mt, 2 * hh + e) * inv, P.out_dtype);
            }
          }
        }
    } else if constexpr (kPvMode == 1) {
      // o = high + low columns; lanes c4 and c4^2 then hold the same sums:
      // lane c4 < 2 writes dims 16mt+r4, lane c4 >= 2 dims 16mt+r4+8, of
      // heads 2(c4&1) and 2(c4&1)+1
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) oc[0][mt][e] += __shfl_xor_sync(0xffffffffu, oc[0][mt][e], 2);
      const int hsel = (c4 & 1) * 2;
      const int dadd = c4 < 2 ? 0 : 8;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int g = hsel + e;
        if (g < G) {
          float lgg = lg[0], mgg = mg[0];
#pragma unroll
          for (int gg = 1; gg < G; ++gg)
            if (g == gg) {
              lgg = lg[gg];
              mgg = mg[gg];
            }
          (void)mgg;
          const float inv = lgg > 0.f ? 1.f / lgg : 0.f;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const float v = c4 < 2 ? oc[0][mt][e] : oc[0][mt][2 + e];
            const int d = 16 * mt + r4 + dadd;
            if (pc.final_out)
              store_out(P.out, row0 + g * kHeadDim + d, v * inv, P.out_dtype);
            else
              rec[g * kHeadDim + d] = v;
          }
        }
      }
    } else {
      // combine the token parities
#pragma unroll
      for (int g = 0; g < (kMmaPv ? 1 : G); ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[g][e].x += __shfl_xor_sync(0xffffffffu, o[g][e].x, 16);
          o[g][e].y += __shfl_xor_sync(0xffffffffu, o[g][e].y, 16);
        }
      if (lane < 16) {
#pragma unroll
        for (int g = 0; g < (kMmaPv ? 1 : G); ++g) {
          if (pc.final_out) {
            const float inv = lg[g] > 0.f ? 1.f / lg[g] : 0.f;
            float v[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[2 * e] = o[g][e].x * inv;
              v[2 * e + 1] = o[g][e].y * inv;
            }
            store_out8(P.out, row0 + g * kHeadDim + 8 * c16, v, P.out_dtype);
          } else {
            float4* dst = reinterpret_cast<float4*>(rec + g * kHeadDim + 8 * c16);
            dst[0] = make_float4(o[g][0].x, o[g][0].y, o[g][1].x, o[g][1].y);
            dst[1] = make_float4(o[g][2].x, o[g][2].y, o[g][3].x, o[g][3].y);
          }
        }
      }
    }
    if (!pc.final_out) {
      if constexpr (kPvMode == 2) {  // lane g writes column g's m and l
        float mv = mg[0], lv = lg[0];
#pragma unroll
        for (int gg = 1; gg < G; ++gg)
          if (lane == gg) {
            mv = mg[gg];
            lv = lg[gg];
          }
        if (lane < G) {
          rec[record_cols(G) * kHeadDim + lane] = mv;
          rec[record_cols(G) * kHeadDim + 64 + lane] = lv;
        }
      } else if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          rec[record_cols(G) * kHeadDim + g] = mg[g];
          rec[record_cols(G) * kHeadDim + 64 + g] = lg[g];
        }
      }
    }
    have_pc = cit.next(pc);
    if (have_pc) load_q();
  }

  // fused step: this grid completes only after the append grid (secondary
  // launch: after the kernel it depends on)
  if ((kFused || (kExt && (P.launch_flags & kLaunchSecondary))) && blockIdx.x == 0 && threadIdx.x == 0)
    asm volatile("griddepcontrol.wait;" ::: "memory");

  // --- drain: never leave a bulk copy in flight into this warp's ring -------
  if (!ok && lane == 0) {
    for (int k = n; k < n_issued; ++k) {
      const uint32_t bar = full0 + 8 * (k % SW);
      const uint32_t parity = static_cast<uint32_t>((k / SW) & 1);
      const long long t0 = global_ns();
      while (!mbar_try_wait(bar, parity) && global_ns() - t0 < P.wait_limit_ns) {
      }
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// The merge kernel: the log-sum-exp combination of the partial records of
// every segment that the decode kernel split (one warp per query head of a
// segment, records in their fixed order, so the result does not depend on
// timing):  M = max_p m_p;  out = sum_p 2^(m_p-M) o_p / sum_p 2^(m_p-M) l_p.
// It is launched as a programmatic dependent of the decode kernel: its
// set-up (the prefix over the lengths, which are inputs) overlaps the decode
// kernel's tail, and griddepcontrol.wait holds it until the decode kernel has
// completed and its records are visible.
// ---------------------------------------------------------------------------
constexpr int kMergeThreads = 128;
// record batch sizes of the merge loop, as a type (a generic lambda picks one)
template <int N>
struct RbTag {
  static constexpr int value = N;
};
// (16-column packed segments: short record lists and 3-4x the items, so
// batches of 4 and 64 registers, 8 CTAs per SM: every item in one wave)
template <int G, bool kExt>
__global__ void __launch_bounds__(kMergeThreads, (kExt && G > 8) ? 8 : 4) merge_kernel(const __grid_constant__ Params P) {
  extern __shared__ int mpfx[];  // [B + 1]
  block_prefix(P, mpfx, nullptr, false);
  const int lane = threadIdx.x & 31;
  const long long wpb = kMergeThreads / 32;
  const long long n_items = static_cast<long long>(P.B) * P.Hkv * G;
  // records of the extended kernel's 8-column tensor-core path are in fragment order
  constexpr bool kFrag = kExt && G > 4;
  constexpr int RB = kExt && G > 8 ? 4 : 16;  // records whose o loads are in flight together (4 for short lists)
  bool waited = false;
  for (long long it = blockIdx.x * wpb + (threadIdx.x >> 5); it < n_items; it += gridDim.x * wpb) {
    const int g = static_cast<int>(it % G);
    const long long sh = it / G;
    const int h = static_cast<int>(sh % P.Hkv);
    const int i = static_cast<int>(sh / P.Hkv);
    if (mpfx[i + 1] == mpfx[i]) continue;  // empty sequence: written by the decode kernel
    const long long at = kExt && P.ext_qbase ? packed_io_offset(P, P.ext_qbase[i], P.ext_ntok[i], h, g)
                                             : (static_cast<long long>(i) * P.Hq + h * G + g) * kHeadDim;
    if (at < 0) continue;  // a column that carries no query
    const SegmentRecords recs(P, mpfx, i, h);
    if (recs.count <= 1) continue;  // whole segment: written by the decode kernel
    if (!waited) {  // the index math above needs only the lengths
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
    }
    float M = -INFINITY, Ls = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < recs.count; c0 += 32) {
      const int cnt = recs.count - c0 < 32 ? recs.count - c0 : 32;
      const bool have = lane < cnt;
      const float* rl = P.ws + recs.at(P, c0 + (have ? lane : 0)) * record_floats(G);
      const float mv = __ldcg(rl + record_cols(G) * kHeadDim + g);
      const float lv = __ldcg(rl + record_cols(G) * kHeadDim + 64 + g);
      const float mk = have ? mv : -INFINITY;
      const float lk = have ? lv : 0.f;
      float wk = 0.f;
      auto batch = [&](auto tag) {
        constexpr int RBv = decltype(tag)::value;
        for (int b0 = 0; b0 < cnt; b0 += RBv) {
          float4 ob[RBv];
#pragma unroll
          for (int r = 0; r < RBv; ++r) {
            const int k = b0 + r < cnt ? b0 + r : 0;
            const float4* r4p = reinterpret_cast<const float4*>(P.ws + recs.at(P, c0 + k) * record_floats(G));
            ob[r] = __ldcg(r4p + (kFrag ? frag_record_index(g, lane) : g * (kHeadDim / 4) + lane));
          }
          if (b0 == 0) {  // this chunk's weights; rescale what came before
            float mx = mk;
#pragma unroll
            for (int msk = 1; msk < 32; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
            const float mn = fmaxf(M, mx);
            const float a = fast_exp2(M - mn);
            wk = fast_exp2(mk - mn);
            float lw = wk * lk;
#pragma unroll
            for (int msk = 1; msk < 32; msk <<= 1) lw += __shfl_xor_sync(0xffffffffu, lw, msk);
            Ls = Ls * a + lw;
            O.x *= a;
            O.y *= a;
            O.z *= a;
            O.w *= a;
            M = mn;
          }
#pragma unroll
          for (int r = 0; r < RBv; ++r) {
            const float w = __shfl_sync(0xffffffffu, wk, (b0 + r) & 31);
            if (b0 + r < cnt) {
              O.x = fmaf(w, ob[r].x, O.x);
              O.y = fmaf(w, ob[r].y, O.y);
              O.z = fmaf(w, ob[r].z, O.z);
              O.w = fmaf(w, ob[r].w, O.w);
            }
          }
        }
      };
      if (cnt <= 4)
        batch(RbTag<4>{});
      else
        batch(RbTag<RB>{});
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    if constexpr (kFrag) {  // this lane's dims are 32k + r + {0, 8, 16, 24}
      const long long d0 = at + 32 * (lane >> 3) + (lane & 7);
      store_out(P.out, d0, O.x * inv, P.out_dtype);
      store_out(P.out, d0 + 8, O.y * inv, P.out_dtype);
      store_out(P.out, d0 + 16, O.z * inv, P.out_dtype);
      store_out(P.out, d0 + 24, O.w * inv, P.out_dtype);
    } else {
      store_out4(P.out, at + 4 * lane, O.x * inv, O.y * inv, O.z * inv, O.w * inv, P.out_dtype);
    }
    if (P.lse && lane == 0)
      P.lse[static_cast<long long>(i) * P.Hq + h * G + g] = Ls > 0.f ? M + __log2f(Ls) : -INFINITY;
  }
  if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");  // completes after the decode grid
}

// ---------------------------------------------------------------------------
// Several new query tokens per sequence.  Sequence i's T_i new tokens are its
// last T_i positions; token t sees positions 0 .. L_i - T_i + t.  They are
// packed TC at a time (TC = 8 / G, or 16 / G in two column halves when the
// sequences average more than 8 columns of new tokens) into the columns of
// one extended-kernel segment: packed sequence v holds tokens t0 .. t0 +
// ntok - 1 of sequence i,
// its length is the last token's position + 1, column tt*G + g is token
// t0 + tt's query head g, and token t0 + tt sees ntok - 1 - tt positions
// fewer.  Every K/V tile of the prefix is read once per TC tokens.  The plan
// kernel writes the packed lengths and each packed sequence's first query
// row (its column blocks carry that row and the ones after it); the decode
// and merge kernels read q and write out at those rows, so nothing is copied
// into or out of a packed layout.
// ---------------------------------------------------------------------------
struct MultiPlan {
  const int32_t* q_start;   // [B + 1]
  const int32_t* seq_lens;  // [B]
  int B, n_q, TC, Bv, max_blocks;
  int32_t* lens_v;          // [Bv]
  int32_t* offs_v;          // [Bv]
  int32_t* ntok_v;          // [Bv]
  int32_t* qbase_v;         // [Bv]: query row of column block 0, or -1 (no query rows)
  long long* err;
};

// One CTA: packed sequences in sequence order (a block-wide scan of
// ceil(T_i / TC)), then the unused tail of the Bv slots.
__global__ void __launch_bounds__(1024) multi_plan_kernel(MultiPlan M) {
  __shared__ int warp_sum[32];
  __shared__ int carry_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int cap = M.max_blocks * kBlock;
  // the decode that reads the plan is launched as this grid's dependent and
  // waits for it to complete before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < M.B; base += blockDim.x) {
    const int i = base + tid;
    int T = 0, L = 0, V = 0;
    if (i < M.B) {
      T = M.q_start[i + 1] - M.q_start[i];
      L = M.seq_lens[i];
      V = T > 0 ? (T + M.TC - 1) / M.TC : 0;
      // q_start must not decrease and must run from 0 to n_q
      if (T < 0 || (i == 0 && M.q_start[0] != 0) || (i == M.B - 1 && M.q_start[M.B] != M.n_q))
        record_error(M.err, PA_ERR_DEVICE_CHECK, i);
    }
    int incl = V;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int w = lane < static_cast<int>(blockDim.x >> 5) ? warp_sum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int start = carry_s + (wid ? warp_sum[wid - 1] : 0) + incl - V;
    if (i < M.B && V > 0) {
      const bool bad = L < T || L > cap || start + V > M.Bv;
      if (bad) record_error(M.err, PA_ERR_DEVICE_CHECK, i);
      for (int k = 0; k < V && start + k < M.Bv; ++k) {
        const int v = start + k, t0 = k * M.TC;
        const int nt = T - t0 < M.TC ? T - t0 : M.TC;
        M.lens_v[v] = bad ? 0 : L - T + t0 + nt;
        M.offs_v[v] = i * M.max_blocks;
        M.ntok_v[v] = nt;
        // column block tt carries row r0 + tt (tt < nt)
        const int r0 = M.q_start[i] + t0;
        const bool rows_ok = r0 >= 0 && r0 + nt <= M.n_q;
        if (!rows_ok) record_error(M.err, PA_ERR_DEVICE_CHECK, i);
        M.qbase_v[v] = rows_ok ? r0 : -1;
      }
    }
    __syncthreads();
    if (tid == 0) carry_s += warp_sum[(blockDim.x >> 5) - 1];
    __syncthreads();
  }
  for (int v = carry_s + tid; v < M.Bv; v += blockDim.x) {
    M.lens_v[v] = 0;
    M.offs_v[v] = 0;
    M.ntok_v[v] = 1;
    M.qbase_v[v] = -1;
  }
}

// ---------------------------------------------------------------------------
// Shared-prefix (cascade) decode.  The members of group k share their first
// P_k blocks (the same physical blocks at the start of their tables).  The
// prefix pass attends all members' queries over those blocks in one segment
// per (group, kv head): member m's G query heads become columns m*G..m*G+G-1
// of a group of SM*G columns (SM = floor(8 / G) members at most), so each
// shared tile is read once for every member.  The suffix pass attends each
// sequence over its own blocks after the prefix.  Both passes return the
// normalised output and the log2-sum-exp; the combine kernel merges them.
// ---------------------------------------------------------------------------
struct CascadeArgs {
  const uint16_t* q;              // [B][Hq][128]
  const int32_t* seq_lens;        // [B]
  const int32_t* tables;          // [B][max_blocks]
  const int32_t* group_start;     // [n_groups + 1]
  const int32_t* members;         // [group_start[n_groups]]
  const int32_t* prefix_blocks;   // [n_groups]
  int B, Hq, Hkv, G, SM, n_groups, max_blocks;
  // workspace
  uint16_t* qv;                   // [n_groups][Hkv*SM*G][128]
  int32_t* lens_v;                // [n_groups]
  int32_t* offs_v;                // [n_groups]
  int32_t* lens_s;                // [B]
  int32_t* offs_s;                // [B]
  int32_t* slot_of;               // [B]: group * 8 + member slot, or -1
  long long* err;
};

// One CTA per (group, kv head): every CTA checks the group; those of kv head
// 0 write the member slots and the prefix lengths and offsets; each packs its
// kv head's queries of the prefix pass (zero past the group's members).
__global__ void cascade_prep_groups(CascadeArgs A) {
  __shared__ int s_bad;
  __shared__ int s_mem[PA_MAX_GROUP];  // the members (at most 8 / G of them)
  const int k = blockIdx.x;
  const int h = blockIdx.y;
  const int m0 = A.group_start[k], m1 = A.group_start[k + 1];
  const int S = m1 - m0;
  const int P = A.prefix_blocks[k];
  const int cap = A.max_blocks * kBlock;
  if (threadIdx.x == 0) s_bad = S < 1 || S > A.SM || P < 0 || P > A.max_blocks;
  __syncthreads();
  if (!s_bad && threadIdx.x < S) {  // one thread per member
    const int i = A.members[m0 + threadIdx.x];
    s_mem[threadIdx.x] = i;
    if (i < 0 || i >= A.B || A.seq_lens[i] < P * kBlock || A.seq_lens[i] > cap) s_bad = 1;
  }
  __syncthreads();
  if (!s_bad) {  // the shared blocks must be the first member's
    const long long first = static_cast<long long>(s_mem[0]) * A.max_blocks;
#pragma unroll 4
    for (int x = threadIdx.x; x < S * P; x += blockDim.x) {
      const int i = s_mem[x / P];
      if (A.tables[static_cast<long long>(i) * A.max_blocks + x % P] != A.tables[first + x % P]) s_bad = 1;
    }
  }
  __syncthreads();
  if (s_bad) {  // reported; its members are decoded without the group
    if (threadIdx.x == 0 && h == 0) {
      record_error(A.err, PA_ERR_DEVICE_CHECK, k);
      A.lens_v[k] = 0;
      A.offs_v[k] = 0;
    }
    return;
  }
  if (h == 0) {
    if (threadIdx.x == 0) {
      A.lens_v[k] = P * kBlock;
      A.offs_v[k] = s_mem[0] * A.max_blocks;
    }
    if (threadIdx.x < S) A.slot_of[s_mem[threadIdx.x]] = k * 8 + threadIdx.x;
  }
  // packed queries of kv head h: 16-byte vectors
  const int GC = A.SM * A.G;  // columns per kv head
  const int n_vec = GC * (kHeadDim / 8);
  const uint4* q = reinterpret_cast<const uint4*>(A.q);
  uint4* qv = reinterpret_cast<uint4*>(A.qv) + (static_cast<long long>(k) * A.Hkv + h) * n_vec;
  for (int x = threadIdx.x; x < n_vec; x += blockDim.x) {
    const int col = x / (kHeadDim / 8), m = col / A.G, g = col % A.G;
    const int w = x % (kHeadDim / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m < S) {
      const int i = s_mem[m];
      v = q[((static_cast<long long>(i) * A.Hq + h * A.G + g) * kHeadDim) / 8 + w];
    }
    qv[x] = v;
  }
}

// One thread per sequence: its suffix after its group's prefix (all of it
// when it is in no group).  Runs after cascade_prep_groups.
__global__ void cascade_prep_seqs(CascadeArgs A) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= A.B) return;
  int L = A.seq_lens[i];
  const int cap = A.max_blocks * kBlock;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int slot = A.slot_of[i];
  const int P = slot >= 0 ? A.prefix_blocks[slot >> 3] : 0;
  const int start = P * kBlock <= L ? P : 0;
  A.lens_s[i] = L - start * kBlock;
  A.offs_s[i] = i * A.max_blocks + start;
}

// One warp per (sequence, query head): merge the two passes' normalised
// outputs o1, o2 with log2-sum-exps e1, e2:
//   out = (2^e1 o1 + 2^e2 o2) / (2^e1 + 2^e2).
__global__ void cascade_combine(CascadeArgs A, const float* o_v, const float* lse_v, const float* o_s,
                                const float* lse_s, void* out, int out_dtype) {
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= static_cast<long long>(A.B) * A.Hq) return;
  const int i = static_cast<int>(wid / A.Hq), hq = static_cast<int>(wid % A.Hq);
  const float4 b = reinterpret_cast<const float4*>(o_s + wid * kHeadDim)[lane];
  float e2 = lse_s[wid];
  float4 r = b;
  const int slot = A.slot_of[i];
  if (slot >= 0) {
    const int k = slot >> 3, m = slot & 7;
    const int GC = A.SM * A.G;
    const int h = hq / A.G, g = hq % A.G;
    const long long row = static_cast<long long>(k) * A.Hkv * GC + h * GC + m * A.G + g;
    const float4 a = reinterpret_cast<const float4*>(o_v + row * kHeadDim)[lane];
    const float e1 = lse_v[row];
    const float M = fmaxf(e1, e2);
    if (M > -INFINITY) {
      const float w1 = fast_exp2(e1 - M), w2 = fast_exp2(e2 - M);
      const float inv = 1.f / (w1 + w2);
      r = make_float4((w1 * a.x + w2 * b.x) * inv, (w1 * a.y + w2 * b.y) * inv, (w1 * a.z + w2 * b.z) * inv,
                      (w1 * a.w + w2 * b.w) * inv);
    } else {
      r = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  store_out4(out, wid * kHeadDim + 4 * lane, r.x, r.y, r.z, r.w, out_dtype);
}

// Failure detection without a fault: the decode's bounded mbarrier wait on a
// barrier that nothing arrives at.  After limit_ns it records PA_ERR_TIMEOUT
// (detail: site 9) and returns; no copy is in flight, nothing traps.
__global__ void wait_selftest_kernel(long long limit_ns, long long* err) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_addr(&bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  wait_phase(smem_addr(&bar), 0u, &abort_flag, limit_ns, err, 9);
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

template <int G, bool kBf16, bool kFused, bool kExt>
static int occupancy_for(size_t bytes) {
  static std::mutex mu;
  static int cached_dev = -1;
  static size_t cached_bytes = 0;
  static int cached_occ = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if (dev == cached_dev && bytes == cached_bytes) return cached_occ;
  if (cudaFuncSetAttribute(decode_kernel<G, kBf16, kFused, kExt>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes<G>(kMaxSplitSeqs, true))) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<G, kBf16, kFused, kExt>,
                                                    Shape<G>::kThreads, bytes) != cudaSuccess)
    return 0;
  if (occ > kMaxCtasPerSm) occ = kMaxCtasPerSm;
  cached_dev = dev;
  cached_bytes = bytes;
  cached_occ = occ;
  return occ;
}

template <int G, bool kBf16, bool kFused, bool kExt>
static int launch_typed(Params& P, int device, cudaStream_t stream) {
  constexpr int NW = Shape<G>::NW;
  int B_smem = P.sched == SCHED_SEGMENT ? 0 : P.B;
  size_t bytes = smem_bytes<G>(B_smem, P.table_offs != nullptr);
  int occ = occupancy_for<G, kBf16, kFused, kExt>(bytes);
  if (occ <= 0) return PA_ERR_CUDA;
  long long slots = static_cast<long long>(sm_count(device)) * occ;
  long long grid;
  if (P.sched == SCHED_SEGMENT) {
    long long segs = static_cast<long long>(P.B) * P.Hkv;
    long long need = (segs + NW - 1) / NW;
    grid = need < slots ? need : slots;
  } else if (P.sched == SCHED_LEAN) {
    grid = slots;
  } else {
    long long parts = static_cast<long long>(P.B) * P.Hkv *
                      ((P.max_blocks + P.partition_blocks - 1) / P.partition_blocks);
    long long need = (parts + NW - 1) / NW;
    grid = need < slots ? need : slots;
  }
  if (grid < 1) grid = 1;
  P.lean_units = static_cast<int>(grid) * NW;
  const bool secondary = kExt && (P.launch_flags & (kLaunchSecondary | kLaunchAfterPlan));
  const bool with_decode = !(P.launch_flags & kLaunchMergeOnly);
  const bool with_merge = P.sched != SCHED_SEGMENT && !(P.launch_flags & kLaunchNoMerge);
  if (kFused && !with_decode) return PA_ERR_INVALID;
  const bool timed = 2 * static_cast<size_t>(g_prof_next) < g_prof_events.size();
  if (timed && cudaEventRecord(g_prof_events[2 * g_prof_next], stream) != cudaSuccess) return PA_ERR_CUDA;
  if (kFused) {
    // the cache write first; the decode is its programmatic dependent and
    // waits for it only before a tile that holds a new token
    const int rc = launch_append_tail(const_cast<uint16_t*>(P.k_pool), const_cast<uint16_t*>(P.v_pool), P.Hkv,
                                      P.num_blocks, P.err, device, P.k_new, P.v_new, P.tables, P.max_blocks,
                                      P.seq_lens, P.B, stream);
    if (rc != PA_OK) return rc;
  }
  if (with_decode && (kFused || secondary)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(Shape<G>::kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_kernel<G, kBf16, kFused, kExt>, P) != cudaSuccess) return PA_ERR_CUDA;
  } else if (with_decode) {
    decode_kernel<G, kBf16, kFused, kExt><<<static_cast<int>(grid), Shape<G>::kThreads, bytes, stream>>>(P);
  }
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  if (with_merge) {
    // the merge of split segments, as a programmatic dependent launch
    constexpr long long kWarpsPerCta = kMergeThreads / 32;
    long long items = static_cast<long long>(P.B) * P.Hkv * G;
    long long mgrid = (items + kWarpsPerCta - 1) / kWarpsPerCta;
    const long long mcap = static_cast<long long>(sm_count(device)) * 8;
    if (mgrid > mcap) mgrid = mcap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(mgrid));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = sizeof(int) * static_cast<size_t>(P.B + 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, merge_kernel<G, kExt>, P) != cudaSuccess) return PA_ERR_CUDA;
  }
  if (timed) {
    if (cudaEventRecord(g_prof_events[2 * g_prof_next + 1], stream) != cudaSuccess) return PA_ERR_CUDA;
    ++g_prof_next;
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <bool kBf16, bool kFused, bool kExt>
static int launch_g(int G, Params& P, int device, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_typed<1, kBf16, kFused, kExt>(P, device, stream);
    case 2: return launch_typed<2, kBf16, kFused, kExt>(P, device, stream);
    case 3: return launch_typed<3, kBf16, kFused, kExt>(P, device, stream);
    case 4: return launch_typed<4, kBf16, kFused, kExt>(P, device, stream);
    case 5: return launch_typed<5, kBf16, kFused, kExt>(P, device, stream);
    case 6: return launch_typed<6, kBf16, kFused, kExt>(P, device, stream);
    case 7: return launch_typed<7, kBf16, kFused, kExt>(P, device, stream);
    case 8: return launch_typed<8, kBf16, kFused, kExt>(P, device, stream);
    case kMaxPackedCols:  // packed tokens only (two column halves)
      if constexpr (kExt && !kFused) return launch_typed<kMaxPackedCols, kBf16, kFused, kExt>(P, device, stream);
      return PA_ERR_UNSUPPORTED;
    default: return PA_ERR_UNSUPPORTED;
  }
}

// Workspace layout: the partial records.
struct WorkspaceLayout {
  size_t records_bytes, total;
};

static bool workspace_layout(const pa_pool* p, int B, int Hq, int max_blocks, int partition_blocks,
                             WorkspaceLayout* out, int max_g = PA_MAX_GROUP) {
  if (!p || B <= 0 || Hq <= 0 || max_blocks <= 0 || partition_blocks < 0) return false;
  if (Hq % p->n_kv_heads) return false;
  int G = Hq / p->n_kv_heads;
  if (G > max_g) return false;
  size_t rec = sizeof(float) * record_floats(G);
  size_t n_rec;
  if (partition_blocks == 0)  // LEAN: two records per warp of the largest grid
    n_rec = 2 * static_cast<size_t>(sm_count(p->device)) * kMaxCtasPerSm * Shape<1>::NW;
  else
    n_rec = static_cast<size_t>(B) * p->n_kv_heads *
            ((max_blocks + partition_blocks - 1) / partition_blocks);
  out->records_bytes = rec * n_rec;
  out->total = out->records_bytes;
  return true;
}

static int decode_common(pa_pool_t p, const void* q, const void* k_new, const void* v_new,
                         const int32_t* tables, int max_blocks, const int32_t* seq_lens, int B,
                         int Hq, float scale, void* out, int out_dtype, int sched,
                         int partition_blocks, void* ws, size_t ws_bytes, void* stream,
                         const int32_t* table_offs = nullptr, float* lse = nullptr,
                         const int32_t* ext_ntok = nullptr, int ext_g = 0, int launch_flags = 0,
                         const int32_t* ext_qbase = nullptr, int ext_hq = 0) {
  if (!p || !q || !tables || !seq_lens || !out || B <= 0 || Hq <= 0 || max_blocks <= 0)
    return PA_ERR_INVALID;
  if (out_dtype != PA_FP16 && out_dtype != PA_BF16 && out_dtype != PA_FP32) return PA_ERR_INVALID;
  if (Hq % p->n_kv_heads) return PA_ERR_INVALID;
  const int G = Hq / p->n_kv_heads;
  // (more than 8 columns: packed query tokens only)
  const int max_g = ext_qbase ? kMaxPackedCols : PA_MAX_GROUP;
  if (G > max_g) return PA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15) return PA_ERR_INVALID;
  const bool fused = k_new != nullptr;
  if (fused && ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15))
    return PA_ERR_INVALID;
  if ((table_offs || lse) && (sched == SCHED_SEGMENT || fused)) return PA_ERR_INVALID;
  // packed tokens in q / out rows: ext_g columns each in the G, columns past the
  // last whole token empty (no log2-sum-exp out)
  if (ext_qbase && (!table_offs || !ext_ntok || lse || ext_g <= 0 || ext_g > G || ext_hq <= 0 ||
                    ext_hq % p->n_kv_heads || ext_hq / p->n_kv_heads != ext_g))
    return PA_ERR_INVALID;
  // (only the 8-column value path of groups above 4 writes packed rows)
  if (ext_qbase && G <= 4) return PA_ERR_UNSUPPORTED;
  if (!on_pool_device(p)) return PA_ERR_INVALID;  // the kernels run on the current device
  WorkspaceLayout lay{};
  if (sched != SCHED_SEGMENT) {
    if (B > kMaxSplitSeqs) return PA_ERR_UNSUPPORTED;
    if (!workspace_layout(p, B, Hq, max_blocks, partition_blocks, &lay, max_g)) return PA_ERR_INVALID;
    if (!ws || ws_bytes < lay.total || (reinterpret_cast<uintptr_t>(ws) & 15)) return PA_ERR_INVALID;
  }
  Params P{};
  P.tmap_kv = p->tmap_kv;
  P.q = static_cast<const uint16_t*>(q);
  P.k_pool = static_cast<const uint16_t*>(p->k);
  P.v_pool = static_cast<const uint16_t*>(p->v);
  P.k_new = static_cast<const uint16_t*>(k_new);
  P.v_new = static_cast<const uint16_t*>(v_new);
  P.tables = tables;
  P.table_offs = table_offs;
  P.lse = lse;
  P.ext_ntok = ext_ntok;
  P.ext_g = ext_g > 0 ? ext_g : 1;
  P.ext_qbase = ext_qbase;
  P.ext_hq = ext_hq;
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
  P.lean_units = 1;
  // (8-column packing keeps the plain cost: one token per sequence then splits
  // exactly like the plain decode, bit for bit)
  P.lean_cost = ext_qbase && G > 8 ? kLeanPieceCostPacked : kLeanPieceCost;
  P.wait_limit_ns = wait_limit_ns();
  P.launch_flags = launch_flags;
  cudaStream_t st = as_stream(stream);
  const bool bf16 = p->dtype == PA_BF16;
  {
    // table offsets (and, optionally, log2-sum-exp outputs) select the
    // extended kernel; the plain and fused kernels carry neither
    const bool ext = table_offs != nullptr;
    if (lse && !ext) return PA_ERR_INVALID;
    if (bf16) {
      if (ext) return launch_g<true, false, true>(G, P, p->device, st);
      return fused ? launch_g<true, true, false>(G, P, p->device, st) : launch_g<true, false, false>(G, P, p->device, st);
    }
    if (ext) return launch_g<false, false, true>(G, P, p->device, st);
    return fused ? launch_g<false, true, false>(G, P, p->device, st) : launch_g<false, false, false>(G, P, p->device, st);
  }
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

// Multi-token queries: workspace pieces, each 256-byte aligned.
struct MultiLayout {
  int TC, GP, Bv;  // tokens per packed sequence, kernel columns, packed sequences
  size_t lens_v, offs_v, ntok_v, qbase_v, rec, total;
};
static bool multi_layout(const pa_pool* p, int n_q, int B, int Hq, int max_blocks, MultiLayout* L) {
  if (!p || n_q <= 0 || B <= 0 || Hq <= 0 || max_blocks <= 0 || Hq % p->n_kv_heads) return false;
  // table rows are addressed by 32-bit element offsets
  if (static_cast<long long>(B) * max_blocks > 0x7fffffffll) return false;
  const int G = Hq / p->n_kv_heads;
  if (G > PA_MAX_GROUP) return false;
  // Sixteen columns (two halves sharing each tile) when the sequences carry
  // more than 8 columns of new tokens on average, else the 8 of one MMA
  // (whole tokens in both cases; columns past the last token stay empty).
  const bool wide = static_cast<long long>(n_q) * G > 8ll * B;
  L->TC = (wide ? kMaxPackedCols : PA_MAX_GROUP) / G;
  L->GP = wide ? kMaxPackedCols : G * L->TC;
  L->Bv = (n_q + L->TC - 1) / L->TC + B;  // every sequence's last pack may be partial
  WorkspaceLayout rw{};
  if (!workspace_layout(p, L->Bv, p->n_kv_heads * L->GP, max_blocks, 0, &rw, kMaxPackedCols)) return false;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  L->lens_v = take(sizeof(int32_t) * L->Bv);
  L->offs_v = take(sizeof(int32_t) * L->Bv);
  L->ntok_v = take(sizeof(int32_t) * L->Bv);
  L->qbase_v = take(sizeof(int32_t) * L->Bv);
  L->rec = take(rw.total);
  L->total = off;
  return true;
}

size_t pa_decode_multi_workspace_bytes(pa_pool_t p, int n_q, int num_seqs, int n_q_heads, int max_blocks_per_seq) {
  MultiLayout L{};
  return multi_layout(p, n_q, num_seqs, n_q_heads, max_blocks_per_seq, &L) ? L.total : 0;
}

int pa_decode_multi(pa_pool_t p, const void* q, const int32_t* q_start, int n_q,
                    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                    int num_seqs, int n_q_heads, float scale, void* out, int out_dtype,
                    void* workspace, size_t workspace_bytes, void* stream) {
  if (!p || !q || !out || !q_start || !seq_lens || !block_tables || num_seqs <= 0 || n_q <= 0 ||
      max_blocks_per_seq <= 0)
    return PA_ERR_INVALID;
  if (out_dtype != PA_FP16 && out_dtype != PA_BF16 && out_dtype != PA_FP32) return PA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15) return PA_ERR_INVALID;
  if (!on_pool_device(p)) return PA_ERR_INVALID;
  MultiLayout L{};
  if (!multi_layout(p, n_q, num_seqs, n_q_heads, max_blocks_per_seq, &L)) return PA_ERR_INVALID;
  if (num_seqs > kMaxSplitSeqs || L.Bv > kMaxSplitSeqs) return PA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return PA_ERR_INVALID;
  char* ws = static_cast<char*>(workspace);
  const int Hkv = p->n_kv_heads, G = n_q_heads / Hkv, GP = L.GP;
  MultiPlan M{};
  M.q_start = q_start;
  M.seq_lens = seq_lens;
  M.B = num_seqs;
  M.n_q = n_q;
  M.TC = L.TC;
  M.Bv = L.Bv;
  M.max_blocks = max_blocks_per_seq;
  M.lens_v = reinterpret_cast<int32_t*>(ws + L.lens_v);
  M.offs_v = reinterpret_cast<int32_t*>(ws + L.offs_v);
  M.ntok_v = reinterpret_cast<int32_t*>(ws + L.ntok_v);
  M.qbase_v = reinterpret_cast<int32_t*>(ws + L.qbase_v);
  M.err = p->err;
  cudaStream_t st = as_stream(stream);
  multi_plan_kernel<<<1, 1024, 0, st>>>(M);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  // the decode and its merge read q and write out at the plan's rows
  return decode_common(p, q, nullptr, nullptr, block_tables, max_blocks_per_seq, M.lens_v, L.Bv, Hkv * GP, scale,
                       out, out_dtype, SCHED_LEAN, 0, ws + L.rec, L.total - L.rec, stream, M.offs_v, nullptr,
                       M.ntok_v, G, kLaunchAfterPlan, M.qbase_v, n_q_heads);
}

// Shared-prefix decode: workspace pieces, each 256-byte aligned.
struct CascadeLayout {
  size_t qv, o_v, lse_v, lens_v, offs_v, o_s, lse_s, lens_s, offs_s, slot_of, rec, rec_v, total;
};
static bool cascade_layout(const pa_pool* p, int B, int Hq, int max_blocks, int n_groups, CascadeLayout* L) {
  if (!p || B <= 0 || Hq <= 0 || n_groups < 0 || max_blocks <= 0 || Hq % p->n_kv_heads) return false;
  // table rows are addressed by 32-bit element offsets
  if (static_cast<long long>(B) * max_blocks > 0x7fffffffll) return false;
  const int G = Hq / p->n_kv_heads;
  if (G > PA_MAX_GROUP) return false;
  const int GC = (PA_MAX_GROUP / G) * G;
  const size_t rows_v = static_cast<size_t>(n_groups) * p->n_kv_heads * GC;
  WorkspaceLayout ra{}, rb{};
  if (n_groups > 0 && !workspace_layout(p, n_groups, p->n_kv_heads * GC, max_blocks, 0, &ra)) return false;
  if (!workspace_layout(p, B, Hq, max_blocks, 0, &rb)) return false;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  L->qv = take(rows_v * kHeadDim * 2);
  L->o_v = take(rows_v * kHeadDim * 4);
  L->lse_v = take(rows_v * 4);
  L->lens_v = take(static_cast<size_t>(n_groups) * 4);
  L->offs_v = take(static_cast<size_t>(n_groups) * 4);
  L->o_s = take(static_cast<size_t>(B) * Hq * kHeadDim * 4);
  L->lse_s = take(static_cast<size_t>(B) * Hq * 4);
  L->lens_s = take(static_cast<size_t>(B) * 4);
  L->offs_s = take(static_cast<size_t>(B) * 4);
  L->slot_of = take(static_cast<size_t>(B) * 4);
  L->rec = take(rb.total);                    // the suffix pass's records
  L->rec_v = n_groups > 0 ? take(ra.total) : off;  // the prefix pass's (both passes run at once)
  L->total = off;
  return true;
}

size_t pa_decode_cascade_workspace_bytes(pa_pool_t p, int num_seqs, int n_q_heads, int max_blocks_per_seq,
                                         int n_groups) {
  CascadeLayout L{};
  return cascade_layout(p, num_seqs, n_q_heads, max_blocks_per_seq, n_groups, &L) ? L.total : 0;
}

int pa_decode_cascade(pa_pool_t p, const void* q, const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* seq_lens, int num_seqs, int n_q_heads, float scale,
                      const int32_t* group_start, const int32_t* members, const int32_t* prefix_blocks,
                      int n_groups, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                      void* stream) {
  if (!p || !q || !block_tables || !seq_lens || !out || num_seqs <= 0 || n_groups < 0 ||
      (n_groups > 0 && (!group_start || !members || !prefix_blocks)))
    return PA_ERR_INVALID;
  if (out_dtype != PA_FP16 && out_dtype != PA_BF16 && out_dtype != PA_FP32) return PA_ERR_INVALID;
  if (num_seqs > kMaxSplitSeqs || n_groups > kMaxSplitSeqs) return PA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15) return PA_ERR_INVALID;
  if (!on_pool_device(p)) return PA_ERR_INVALID;
  CascadeLayout L{};
  if (!cascade_layout(p, num_seqs, n_q_heads, max_blocks_per_seq, n_groups, &L)) return PA_ERR_INVALID;
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return PA_ERR_INVALID;
  char* ws = static_cast<char*>(workspace);
  const int G = n_q_heads / p->n_kv_heads;
  CascadeArgs A{};
  A.q = static_cast<const uint16_t*>(q);
  A.seq_lens = seq_lens;
  A.tables = block_tables;
  A.group_start = group_start;
  A.members = members;
  A.prefix_blocks = prefix_blocks;
  A.B = num_seqs;
  A.Hq = n_q_heads;
  A.Hkv = p->n_kv_heads;
  A.G = G;
  A.SM = PA_MAX_GROUP / G;
  A.n_groups = n_groups;
  A.max_blocks = max_blocks_per_seq;
  A.qv = reinterpret_cast<uint16_t*>(ws + L.qv);
  A.lens_v = reinterpret_cast<int32_t*>(ws + L.lens_v);
  A.offs_v = reinterpret_cast<int32_t*>(ws + L.offs_v);
  A.lens_s = reinterpret_cast<int32_t*>(ws + L.lens_s);
  A.offs_s = reinterpret_cast<int32_t*>(ws + L.offs_s);
  A.slot_of = reinterpret_cast<int32_t*>(ws + L.slot_of);
  A.err = p->err;
  cudaStream_t st = as_stream(stream);
  if (cudaMemsetAsync(A.slot_of, 0xff, sizeof(int32_t) * static_cast<size_t>(num_seqs), st) != cudaSuccess)
    return PA_ERR_CUDA;
  if (n_groups > 0) cascade_prep_groups<<<dim3(n_groups, p->n_kv_heads), 128, 0, st>>>(A);
  cascade_prep_seqs<<<(num_seqs + 255) / 256, 256, 0, st>>>(A);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  float* o_v = reinterpret_cast<float*>(ws + L.o_v);
  float* lse_v = reinterpret_cast<float*>(ws + L.lse_v);
  float* o_s = reinterpret_cast<float*>(ws + L.o_s);
  float* lse_s = reinterpret_cast<float*>(ws + L.lse_s);
  const size_t rec_s_bytes = L.rec_v - L.rec, rec_v_bytes = L.total - L.rec_v;
  // The suffix pass fills the GPU; the prefix pass is its programmatic
  // dependent and takes the SMs its tail frees.  Then the two merges and the
  // combine, in stream order.
  auto suffix = [&](int flags) {
    return decode_common(p, q, nullptr, nullptr, block_tables, max_blocks_per_seq, A.lens_s, num_seqs, n_q_heads,
                         scale, o_s, PA_FP32, SCHED_LEAN, 0, ws + L.rec, rec_s_bytes, stream, A.offs_s, lse_s,
                         nullptr, 0, flags);
  };
  auto prefix = [&](int flags) {
    return decode_common(p, A.qv, nullptr, nullptr, block_tables, max_blocks_per_seq, A.lens_v, n_groups,
                         p->n_kv_heads * A.SM * G, scale, o_v, PA_FP32, SCHED_LEAN, 0, ws + L.rec_v, rec_v_bytes,
                         stream, A.offs_v, lse_v, nullptr, 0, flags);
  };
  int rc;
  if (n_groups > 0) {
    if ((rc = suffix(kLaunchNoMerge)) != PA_OK) return rc;
    if ((rc = prefix(kLaunchSecondary | kLaunchNoMerge)) != PA_OK) return rc;
    if ((rc = prefix(kLaunchMergeOnly)) != PA_OK) return rc;
    if ((rc = suffix(kLaunchMergeOnly)) != PA_OK) return rc;
  } else if ((rc = suffix(0)) != PA_OK) {
    return rc;
  }
  const long long warps = static_cast<long long>(num_seqs) * n_q_heads;
  cascade_combine<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(A, o_v, lse_v, o_s, lse_s, out,
                                                                                   out_dtype);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_selftest_wait_timeout(pa_pool_t p, long long limit_ns, void* stream) {
  if (!p || limit_ns <= 0 || limit_ns > 1000000000ll || !on_pool_device(p)) return PA_ERR_INVALID;
  wait_selftest_kernel<<<1, 32, 0, as_stream(stream)>>>(limit_ns, p->err);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Split decode without allocation: the workspace is this file's static device
// array.  For callers that cannot allocate device memory when they decode.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace pa {

static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch on the current device (the host-side
// symbol is only a stand-in), looked up once per device and cached.  The
// cache assumes that the device's context lives as long as the process:
// after a cudaDeviceReset the library must not be used again.
static int static_scratch_on(int device, void** out) {
  static std::mutex mu;
  static std::vector<void*> addr;
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0) return PA_ERR_INVALID;
  if (static_cast<size_t>(device) >= addr.size()) addr.resize(device + 1, nullptr);
  if (!addr[device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return PA_ERR_CUDA;
    addr[device] = ptr;
  }
  *out = addr[device];
  return PA_OK;
}

}  // namespace pa

extern "C" int pa_decode_split_static(pa_pool_t p, const void* q, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                      int n_q_heads, float scale, void* out, int out_dtype,
                                      int partition_blocks, void* stream) {
  if (!p || partition_blocks < 0) return PA_ERR_INVALID;
  // the array looked up is the current device's: it must be the pool's
  if (!on_pool_device(p)) return PA_ERR_INVALID;
  WorkspaceLayout lay{};
  if (!workspace_layout(p, num_seqs, n_q_heads, max_blocks_per_seq, partition_blocks, &lay))
    return PA_ERR_INVALID;
  if (lay.total > static_cast<size_t>(PA_STATIC_SCRATCH_BYTES)) return PA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  int st = static_scratch_on(p->device, &scratch);
  if (st != PA_OK) return st;
  // nothing in the array needs clearing: every record is written before it is read
  return pa_decode_split(p, q, block_tables, max_blocks_per_seq, seq_lens, num_seqs, n_q_heads,
                         scale, out, out_dtype, partition_blocks, scratch,
                         static_cast<size_t>(PA_STATIC_SCRATCH_BYTES), stream);
}
