/*
 * pa.h - C ABI of the paged KV-cache decode library for one GB300 (sm_103a).
 *
 * What the library computes.  A KV cache keeps every earlier token's keys and
 * values so that a decode step only processes the one new token, and the
 * cached result is exact ("The KV Cache: How Transformers Avoid Recomputing
 * the Past", inference-serving tag page).  The cache lives in small fixed-size
 * blocks of 16 tokens that are handed out as a sequence grows; a per-sequence
 * table maps logical positions to physical blocks, and sequences that share a
 * prefix can share its blocks ("Serving", section 23.4 Paged Attention;
 * "Paged Attention: Managing the KV Cache Like Virtual Memory", teaser on the
 * inference-serving tag page, which also names copy-on-write sharing).  Decode
 * reads the whole cache for one query token per sequence, so it is bound by
 * memory traffic, not arithmetic ("Serving", section 23.2 Prefill and Decode).
 *
 * Conventions shared by every call:
 *  - Every call returns an int status (PA_OK or a negative PA_ERR_* code).
 *    Errors that the host can see (null pointer, bad size, unsupported shape,
 *    dtype mismatch) are returned before anything is launched, and nothing is
 *    written.  A failed launch returns PA_ERR_CUDA.
 *  - Device calls are asynchronous on `stream` (a cudaStream_t passed as
 *    void*; NULL is the legacy default stream).  "device" below means a
 *    pointer to memory of the GPU that owns the pool; "host" means CPU memory.
 *  - Ownership: the library owns only the pool's device memory (allocated in
 *    pa_pool_create, released in pa_pool_destroy) and the allocator's host
 *    state.  The caller owns every other buffer (q, k_new, v_new, out, tables,
 *    lengths, slot mappings, workspace); none is retained after a call
 *    returns.
 *  - Block size is 16 tokens and d_head is 128 (compile-time constants of the
 *    kernels); other values return PA_ERR_UNSUPPORTED.
 *  - Calls that launch kernels run them on the current device, which must be
 *    the device the pool was created on; a call made while another device
 *    is current returns PA_ERR_INVALID before anything is launched.
 *  - The library caches per-device state (SM counts, the static scratch
 *    array's address) for the life of the process: do not use it again
 *    after cudaDeviceReset.
 *  - Device-side bounds checks are always on: a block id outside
 *    [0, num_blocks) in a table or a slot outside [0, num_blocks*16) is never
 *    dereferenced.  The kernel skips it, records the first such event in the
 *    pool's device error word, and pa_check() reports it as
 *    PA_ERR_DEVICE_CHECK.  Every wait inside a kernel has an iteration limit;
 *    a wait that runs out records PA_ERR_TIMEOUT there instead of hanging.
 */
#ifndef PAGED_KV_CACHE_PA_H
#define PAGED_KV_CACHE_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  K/V pools, q, k_new and v_new are FP16 or BF16; the output
 * may also be FP32 (fp32 output isolates the kernel's arithmetic from the
 * final rounding to 16 bits). */
typedef enum { PA_FP16 = 0, PA_BF16 = 1, PA_FP32 = 2 } pa_dtype;

enum {
  PA_OK = 0,
  PA_ERR_INVALID = -1,      /* bad argument (null pointer, size <= 0, ...)   */
  PA_ERR_UNSUPPORTED = -2,  /* valid but not built (d_head != 128, ...)      */
  PA_ERR_OOM = -3,          /* device allocation or allocator free list empty */
  PA_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed           */
  PA_ERR_DEVICE_CHECK = -5, /* a kernel met an out-of-range block id or slot  */
  PA_ERR_TIMEOUT = -6,      /* a bounded in-kernel wait ran out               */
  PA_ERR_SCRATCH_LIMIT = -7 /* needs more than the library's static scratch   */
};

enum { PA_BLOCK_SIZE = 16, PA_HEAD_DIM = 128, PA_MAX_GROUP = 8 };

typedef struct pa_pool* pa_pool_t;

/* ---------------------------------------------------------------------------
 * Pool.  Two device arrays, K and V, each laid out [num_blocks][n_kv_heads]
 * [16][d_head] row-major, so one (block, kv head) tile is 16*128 elements =
 * 4 KiB contiguous and one whole block (all heads) is contiguous for a
 * copy-on-write copy.  Physical blocks of fixed size, per "Serving" 23.4.
 * ------------------------------------------------------------------------- */

/* Bytes of ONE pool array (K or V) for these sizes; host only, no GPU needed.
 * Returns 0 for invalid or unsupported sizes.  2*pa_pool_bytes(1,16,H,d,t)/16
 * is the per-token, per-layer KV size of the closed form in "Serving" 23.1:
 * 2 * n_kv_heads * d_head * n_bytes. */
size_t pa_pool_bytes(int num_blocks, int block_size, int n_kv_heads, int d_head,
                     int dtype);

/* Allocates K and V pools (cudaMalloc on the current device, zero-filled) and
 * the device error word.  dtype is PA_FP16 or PA_BF16.  *out receives the
 * handle.  Errors: INVALID (num_blocks <= 0, n_kv_heads <= 0, out null),
 * UNSUPPORTED (block_size != 16, d_head != 128, dtype not 16-bit, or
 * num_blocks * n_kv_heads * 16 >= 2^31 token rows: a 512 GiB array), OOM. */
int pa_pool_create(int num_blocks, int block_size, int n_kv_heads, int d_head,
                   int dtype, pa_pool_t* out);

/* Frees the pool's device memory after synchronising its device.  NULL is a
 * no-op returning PA_OK. */
int pa_pool_destroy(pa_pool_t pool);

/* Device addresses of the K and V arrays and the bytes of each (any output
 * pointer may be NULL).  The addresses stay owned by the pool. */
int pa_pool_info(pa_pool_t pool, void** k_pool, void** v_pool,
                 size_t* bytes_per_pool);

/* Shape of the pool (any output pointer may be NULL). */
int pa_pool_shape(pa_pool_t pool, int* num_blocks, int* n_kv_heads,
                  int* d_head, int* dtype);

/* ---------------------------------------------------------------------------
 * Cache write.  Writes the newest K/V of each token into its slot, the step
 * by which the cache grows a token at a time ("Serving" 23.4).
 *   k_new, v_new : device, [n_tok][n_kv_heads][128], pool dtype.
 *   slot_mapping : device int64 [n_tok]; slot = block*16 + offset; a negative
 *                  slot means "skip this row" (padding).
 * Rows with distinct slots are written bit for bit; two tokens naming the same
 * slot race (unspecified winner).  Out-of-range slots are skipped and
 * reported by pa_check.  n_tok == 0 is a no-op.
 * ------------------------------------------------------------------------- */
int pa_cache_append(pa_pool_t pool, const void* k_new, const void* v_new,
                    const int64_t* slot_mapping, int n_tok, void* stream);

/* ---------------------------------------------------------------------------
 * Decode attention over the paged cache ("Serving" 23.2 and 23.4).
 * For sequence i and query head h, with kv head g = h / (n_q_heads/n_kv_heads)
 * (contiguous grouped-query mapping) and L = seq_lens[i]:
 *   K_i[t] = Kpool[block_tables[i][t/16]][g][t%16],  t < L (same for V)
 *   out[i][h] = softmax(scale * K_i q[i][h]) V_i
 * computed with fp32 accumulation.  L == 0 gives an all-zero output row.
 *   q            : device, [num_seqs][n_q_heads][128], pool dtype.
 *   block_tables : device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  ceil(L/16) are never read.
 *   seq_lens     : device int32 [num_seqs]; 0 <= L <= 16*max_blocks_per_seq
 *                  (a larger L is clamped to that bound and reported by
 *                  pa_check).
 *   out          : device, [num_seqs][n_q_heads][128] of out_dtype.
 * n_q_heads must be a multiple of n_kv_heads.  Each CTA owns one (sequence,
 * kv head) pair and its whole query-head group, so every K/V tile is read
 * from HBM once per step.
 * ------------------------------------------------------------------------- */
int pa_decode(pa_pool_t pool, const void* q, const int32_t* block_tables,
              int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
              int n_q_heads, float scale, void* out, int out_dtype,
              void* stream);

/* Workspace bytes that pa_decode_split / pa_append_decode need for these
 * sizes on this pool's device (partition_blocks as passed to them; 0 = the
 * balanced automatic split).  Host only; returns 0 for invalid sizes. */
size_t pa_decode_workspace_bytes(pa_pool_t pool, int num_seqs, int n_q_heads,
                                 int max_blocks_per_seq, int partition_blocks);

/* Split-KV decode.  partition_blocks > 0: each sequence's logical blocks are
 * cut into partitions of partition_blocks blocks, and each (sequence, kv head,
 * partition) is one work unit.  partition_blocks == 0: the tiles of all
 * (sequence, kv head) pairs, laid end to end, are cut into equal ranges, one
 * per warp of a persistent grid sized to the GPU, so any length mix is
 * spread evenly; a pair cut by a range boundary becomes several units.  A unit
 * that does not cover its whole pair writes its running max m, sum l and
 * unnormalised output o in fp32 to the workspace; a second kernel, launched
 * on the same stream as a programmatic dependent of the first, merges each
 * cut pair's partial results by log-sum-exp in their fixed order:
 *   M = max_p m_p,  out = sum_p e^(m_p-M) o_p / sum_p e^(m_p-M) l_p.
 * The result equals pa_decode's up to rounding and does not depend on
 * timing.  Pairs covered by a single unit are written directly.  workspace:
 * device, at least pa_decode_workspace_bytes(...) bytes, 16-byte aligned,
 * caller-owned; its contents on entry do not matter.  Calls that share a
 * workspace must not overlap on the GPU.  num_seqs <= 4096 (the per-sequence
 * prefix lives in shared memory), else PA_ERR_UNSUPPORTED. */
int pa_decode_split(pa_pool_t pool, const void* q, const int32_t* block_tables,
                    int max_blocks_per_seq, const int32_t* seq_lens,
                    int num_seqs, int n_q_heads, float scale, void* out,
                    int out_dtype, int partition_blocks, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Fused append + split decode for one new token per sequence.  seq_lens
 * counts the new token (L >= 1); the new token sits at position L-1, whose
 * slot is block_tables[i][(L-1)/16]*16 + (L-1)%16.  A small kernel writes
 * k_new[i]/v_new[i] ([num_seqs][n_kv_heads][128]) to that slot; the decode is
 * launched as its programmatic dependent, streams every other tile at once
 * and waits for the write only before a tile that holds a new token.  The
 * result equals pa_cache_append followed by pa_decode_split.  Rows with
 * L == 0 write nothing and output zeros.  num_seqs <= 4096, else
 * PA_ERR_UNSUPPORTED.  Sequences that share a prefix are read once per
 * sharer here; a caller that wants the shared blocks read once appends with
 * pa_cache_append and decodes with pa_decode_cascade. */
int pa_append_decode(pa_pool_t pool, const void* q, const void* k_new,
                     const void* v_new, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* seq_lens,
                     int num_seqs, int n_q_heads, float scale, void* out,
                     int out_dtype, int partition_blocks, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Attention for several new query tokens per sequence: a chunk of a prompt
 * written onto the sequence's blocks, or drafted tokens checked in one pass
 * ("Serving", sections 23.2 Prefill and Decode and 23.5 Speculative
 * Decoding, over the blocks and tables of 23.4).  The new tokens' K/V must
 * already be in the pool (pa_cache_append); seq_lens[i] counts them.
 * q: device [n_q][n_q_heads][128]; sequence i's query rows are
 * q_start[i] .. q_start[i+1]-1 (device int32 [num_seqs+1], non-decreasing,
 * q_start[0] = 0, q_start[num_seqs] = n_q), its last T_i positions in order.
 * Row r = q_start[i] + t sits at position L_i - T_i + t and attends over
 * positions 0 .. L_i - T_i + t (causal within the new tokens):
 *   out[r][h] = softmax(scale * K[0..p] q[r][h]) V[0..p],  p = L_i - T_i + t.
 * out: device [n_q][n_q_heads][128] in out_dtype.  A sequence's new tokens
 * are packed 8/G at a time into the columns of one segment of the balanced
 * split (G = n_q_heads / n_kv_heads), each column masked to its token's causal
 * prefix, so every K/V tile is read once per 8/G new tokens.  A planning
 * kernel maps each packed column block to its query row; the decode (its
 * programmatic dependent) and the merge read q and write out through that
 * map.  workspace: device, >= pa_decode_multi_workspace_bytes(...) bytes,
 * 256-byte aligned (lengths, maps and the split's partial records).
 * ceil(n_q / (8/G)) + num_seqs <= 4096 (else PA_ERR_UNSUPPORTED);
 * num_seqs * max_blocks_per_seq < 2^31 (else PA_ERR_INVALID).  A
 * sequence with T_i > L_i, or a length out of range, records
 * PA_ERR_DEVICE_CHECK (pa_check) and outputs zeros.  A q_start that
 * decreases or does not run from 0 to n_q records PA_ERR_DEVICE_CHECK; rows
 * it leaves to no sequence are not written. */
size_t pa_decode_multi_workspace_bytes(pa_pool_t pool, int n_q, int num_seqs,
                                       int n_q_heads, int max_blocks_per_seq);
int pa_decode_multi(pa_pool_t pool, const void* q, const int32_t* q_start, int n_q,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* seq_lens, int num_seqs, int n_q_heads,
                    float scale, void* out, int out_dtype, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Shared-prefix (cascade) decode: pa_decode's result, with each group's
 * shared prefix read once for all of its members ("Serving" 23.4: sequences
 * that share a prefix share its blocks).  Group k's members are
 * members[group_start[k] .. group_start[k+1]-1] (device int32; 2 to
 * floor(8 / (n_q_heads / n_kv_heads)) sequences); they share their first
 * prefix_blocks[k] table entries (the same physical blocks), each full
 * (16 * prefix_blocks[k] <= every member's length).  One pass attends every
 * member's query heads over the shared blocks as one segment per (group, kv
 * head); a second attends each sequence over its blocks after its group's
 * prefix (all of them for a sequence in no group); a third merges the two by
 * log-sum-exp.  The first pass runs on the SMs that the second's tail frees
 * (a programmatic dependent launch), so the two passes overlap.  A group that breaks these rules is reported
 * (PA_ERR_DEVICE_CHECK) and its members are decoded without it.  q, out,
 * block_tables, seq_lens as for pa_decode; num_seqs and n_groups <= 4096;
 * num_seqs * max_blocks_per_seq < 2^31 (else PA_ERR_INVALID).
 * workspace: device, >= pa_decode_cascade_workspace_bytes(...), 256-byte
 * aligned. */
size_t pa_decode_cascade_workspace_bytes(pa_pool_t pool, int num_seqs, int n_q_heads,
                                         int max_blocks_per_seq, int n_groups);
int pa_decode_cascade(pa_pool_t pool, const void* q, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                      int n_q_heads, float scale, const int32_t* group_start,
                      const int32_t* members, const int32_t* prefix_blocks, int n_groups,
                      void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                      void* stream);

/* Split-KV decode that allocates nothing (the pages have no counterpart; this
 * is a deployment convenience).  Some callers cannot call cudaMalloc at the
 * time they decode: a serving loop whose device memory budget is fixed up
 * front, or a host that links this library without any allocator of its
 * own.  This call is
 * pa_decode_split with partition_blocks as there, but its workspace is a
 * static device array owned by the library instead of a caller buffer.
 *  - Limit: the array holds PA_STATIC_SCRATCH_BYTES (12 MiB); a call whose
 *    pa_decode_workspace_bytes(...) exceeds it returns PA_ERR_SCRATCH_LIMIT
 *    before launching anything.  num_seqs <= 4096, as for pa_decode_split.  With partition_blocks == 0 this fits every
 *    group size up to 8 on a 152-SM GPU; fixed partitions fit while
 *    num_seqs * n_kv_heads * ceil(max_blocks_per_seq / partition_blocks)
 *    records (each (G+1)*512 bytes) stay under the limit.
 *  - Every GPU that loads the library keeps the 12 MiB until the process
 *    exits.  The first call on a device looks the array's device address up
 *    (cudaGetSymbolAddress, with that device current) and caches it, so make
 *    the first call on each device before any stream capture.
 *  - All calls share the array and it keeps the last call's contents;
 *    nothing in it needs to start at zero.  Calls that overlap on the GPU
 *    (on two streams of one device) race on the array: serialise them.  A
 *    call made while another device than the pool's is current is refused
 *    (PA_ERR_INVALID), so a device's array is only used by its own pools.
 *  - No cudaMalloc, cudaFree or other allocating routine is called. */
enum { PA_STATIC_SCRATCH_BYTES = 12 << 20 };
int pa_decode_split_static(pa_pool_t pool, const void* q, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* seq_lens,
                           int num_seqs, int n_q_heads, float scale, void* out,
                           int out_dtype, int partition_blocks, void* stream);

/* Copy-on-write support: copies whole blocks (all kv heads, K and V) from
 * src[j] to dst[j], j < n, both device int32 arrays.  The destinations must be
 * distinct from each other and from every source.  Used when a sequence
 * appends into a block it shares with another ("Paged Attention" teaser:
 * sharing with copy-on-write). */
int pa_copy_blocks(pa_pool_t pool, const int32_t* src, const int32_t* dst,
                   int n, void* stream);

/* Kernel timing for benchmarks.  pa_profile_start(capacity) creates
 * `capacity` pairs of CUDA events on the current device; each later
 * pa_decode / pa_decode_split / pa_append_decode call (until `capacity` calls
 * have been recorded) records one pair on its stream, right before its first
 * kernel and right after its last (the append kernel of the fused step, the
 * decode kernel and the merge kernel).
 * pa_profile_stop(ms, cap) waits for the recorded pairs, writes up to cap
 * elapsed times in milliseconds to ms (host), releases the events and returns
 * how many pairs were recorded (or a negative status).  Process-wide, not
 * thread-safe; starting again discards an unfinished profile. */
int pa_profile_start(int capacity);
int pa_profile_stop(float* ms, int cap);

/* Failure-detection self-test (no counterpart on the pages): runs the
 * kernels' bounded mbarrier wait, on `stream`, on a barrier nothing arrives
 * at.  After limit_ns (0 < limit_ns <= 1e9) the wait gives up, records
 * PA_ERR_TIMEOUT in the pool's error word (detail 9, the wait site) and the
 * kernel returns; pa_check then reports it and the context stays usable.
 * Nothing traps or hangs. */
int pa_selftest_wait_timeout(pa_pool_t pool, long long limit_ns, void* stream);

/* Synchronises `stream`, reads and clears the pool's device error word.
 * Returns PA_OK, PA_ERR_DEVICE_CHECK or PA_ERR_TIMEOUT; *detail (may be NULL)
 * receives the offending block id / slot (or the wait site for a timeout). */
int pa_check(pa_pool_t pool, void* stream, int64_t* detail);

/* Static message for a status code. */
const char* pa_strerror(int code);

/* ---------------------------------------------------------------------------
 * Host block allocator (CPU only): free list, per-block reference counts,
 * prefix sharing by fork, and copy-on-write on append ("Serving" 23.4: blocks
 * allocated as a sequence grows, shared between sequences with a common
 * prefix; "Paged Attention" teaser: copy-on-write).
 *
 * Policy, fixed so that results are reproducible:
 *  - The free list is a FIFO queue.  It starts as free_order[0..num_blocks)
 *    (a permutation of the block ids; NULL means 0,1,2,...); allocation takes
 *    the front, a block whose count drops to 0 goes to the back.
 *  - Appending token number p (0-based) of a sequence: if p % 16 == 0 a new
 *    block is taken; otherwise, if the last block's count is > 1, it is
 *    copied on write: a new block is taken, the old block's count drops by
 *    one and the table points at the new block (the caller must then copy the
 *    old block's contents, e.g. with pa_copy_blocks).  slot = block*16 + p%16.
 *  - fork(parent, child): the child gets a copy of the parent's table and
 *    length; every block's count rises by one.
 *  - free(seq): counts drop in table order; blocks reaching 0 are queued.
 *  - Running out of blocks returns PA_ERR_OOM and changes nothing.
 * ------------------------------------------------------------------------- */
typedef struct pa_alloc* pa_alloc_t;

int pa_alloc_create(int num_blocks, int block_size, const int32_t* free_order,
                    pa_alloc_t* out);
int pa_alloc_destroy(pa_alloc_t a);
/* New empty sequence; INVALID if seq_id < 0 or already present. */
int pa_alloc_seq_add(pa_alloc_t a, int seq_id);
/* Child shares all of the parent's blocks; INVALID if the parent is missing or
 * the child exists. */
int pa_alloc_fork(pa_alloc_t a, int parent, int child);
/* Reserves the slot of the sequence's next token.  *slot receives it;
 * *cow_src/*cow_dst receive the copied block pair, or -1/-1 if no copy. */
int pa_alloc_append_slot(pa_alloc_t a, int seq, int64_t* slot,
                         int32_t* cow_src, int32_t* cow_dst);
/* n calls of pa_alloc_append_slot in one: slots[0..n) (may be NULL) receive
 * the slots; the at most one copy-on-write (it can only happen on the first
 * token) is reported in *cow_src/*cow_dst.  On OOM the tokens reserved before
 * the failure stay reserved and *n_done (may be NULL) says how many. */
int pa_alloc_extend(pa_alloc_t a, int seq, int n, int64_t* slots,
                    int32_t* cow_src, int32_t* cow_dst, int* n_done);
/* Releases the sequence's blocks (see policy) and forgets the sequence. */
int pa_alloc_seq_free(pa_alloc_t a, int seq);
/* Copies up to cap table entries into out; *n_blocks = the table's length. */
int pa_alloc_table(pa_alloc_t a, int seq, int32_t* out, int cap,
                   int* n_blocks);
/* Tokens held by the sequence, or a negative status. */
int pa_alloc_seq_len(pa_alloc_t a, int seq);
/* Reference count of a block (0 = free), or a negative status. */
int pa_alloc_refcount(pa_alloc_t a, int block);
/* Number of blocks on the free list. */
int pa_alloc_num_free(pa_alloc_t a);
/* Groups for pa_decode_cascade from host block tables: sequences whose
 * first blocks are the same, in order of first appearance, cut into groups
 * of at most max_members; a group's prefix is the run of table entries all
 * its members share, counting only blocks full in every member; groups of one
 * or with no shared full block are dropped.  Outputs (host, capacity
 * num_seqs + 1, num_seqs, num_seqs): group_start, members, prefix_blocks;
 * *n_groups receives the count. */
int pa_cascade_groups(const int32_t* tables, int num_seqs, int max_blocks,
                      const int32_t* seq_lens, int max_members, int32_t* group_start,
                      int32_t* members, int32_t* prefix_blocks, int* n_groups);

/* ---------------------------------------------------------------------------
 * Prefix caching by block hashes ("Paged Attention" teaser on the
 * inference-serving tag page: prefix caching by block hashes; the posts on
 * the pagedattention tag: blocks chained by hashes, so one changed character
 * early in a prompt voids every cached block after it).  Host only.
 *
 *  - A full block of a sequence whose tokens were all appended with their
 *    ids is hashed when its last token arrives:
 *      h_k = FNV-1a-64(h_{k-1} as 8 little-endian bytes ||
 *                      its 16 token ids as 4-byte little-endian integers),
 *    h_{-1} = 0 (FNV-1a: start 14695981039346656037; per byte: xor, then
 *    multiply by 1099511628211 mod 2^64).  A hash already indexed keeps its
 *    older block.  pa_alloc_append_slot (no id) stops hashing for that
 *    sequence.
 *  - The index keeps, per hash, the block, the parent hash and the 16 ids; a
 *    lookup accepts an entry only if all three match (a collision misses).
 *  - A block whose count drops to 0 joins the back of the free list and stays
 *    indexed; a lookup that hits it takes it back off the free list; taking a
 *    block from the front for a new allocation drops its index entry.
 * ------------------------------------------------------------------------- */
/* New sequence seq_id for a prompt of n_tokens ids (host array): shares the
 * longest chain of cached full blocks from the prompt's start (counts +1) and
 * stops at the first miss.  *n_cached (may be NULL) receives 16 x hits, the
 * tokens the sequence now holds; append the rest with pa_alloc_append_token.
 * INVALID if seq_id < 0 or exists, or tokens is NULL with n_tokens > 0. */
int pa_alloc_seq_add_cached(pa_alloc_t a, int seq_id, const int32_t* tokens,
                            int n_tokens, int* n_cached);
/* pa_alloc_append_slot that also records the token's id; completing a block
 * indexes it (see above). */
int pa_alloc_append_token(pa_alloc_t a, int seq, int32_t token, int64_t* slot,
                          int32_t* cow_src, int32_t* cow_dst);
/* 1 and *hash = the block's hash if the block is indexed, 0 if not, or a
 * negative status. */
int pa_alloc_block_hash(pa_alloc_t a, int block, uint64_t* hash);
/* Blocks looked up and hit by pa_alloc_seq_add_cached so far, and blocks now
 * indexed (each pointer may be NULL). */
int pa_alloc_prefix_stats(pa_alloc_t a, int64_t* queries, int64_t* hits,
                          int64_t* cached_blocks);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_CACHE_PA_H */
