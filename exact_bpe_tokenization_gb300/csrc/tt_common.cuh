// tt_common.cuh - device-side definitions shared by the kernels of the exact
// BPE tokenizer: sizes, tables, hashing, status reporting, block scans and
// decoupled look-back.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "tt_rules.cuh"

namespace tt {

// ------------------------------------------------------------ geometry
// Pre-tokenizer tiles: one CTA reads a 4096-byte window, 8 or 16 bytes (one
// vector load) per thread: 48 bytes before the tile (lookback and the
// shifted scan entry points), the 4016-byte tile, 32 bytes after it.
constexpr int WIN = 4096;
constexpr int HALO_L = 48;
constexpr int HALO_R = 32;
constexpr int TILE = WIN - HALO_L - HALO_R;  // 4016 = 16 * 251
constexpr int S1_SHIFT = 32;                 // mark-resolution scan enters at tile start - 32
constexpr int S2_SHIFT = 16;                 // forward scan enters at tile start - 16
static_assert(TILE % 16 == 0 && HALO_L % 16 == 0, "windows keep 16-byte alignment");

// BPE execution units by piece length (bytes)
constexpr int SMALL_MAX = 16;                // thread per piece, dense over all pieces
constexpr int MID_MAX = 256;                 // thread per piece, dense over the longer ones
                                             // (> MID_MAX: a block per piece)
constexpr int IDS_CHUNK = 512;               // pieces per chunk in the ID scatter
// capacity of one mid-length bucket, and the bucket of a piece length
constexpr int64_t list_cap(int64_t cap_bytes) { return cap_bytes / (SMALL_MAX + 1) + 2; }
TT_HD int mid_bucket(int64_t len) { return len > 128 ? 0 : len > 48 ? 1 : 2; }
TT_HD int mid_bucket_counter(int b) { return b == 0 ? 2 : b == 1 ? 7 : 8; }   // counters[] slot

// status codes (mirror include/toktier.h)
enum : int { ST_OK = 0, ST_INVALID_ARG = 1, ST_INVALID_UTF8 = 4, ST_CAPACITY = 5, ST_TIMEOUT = 8 };

struct DevStatus {
  int code;                       // first error recorded (0 = none)
  int pad;
  unsigned long long bad_request; // lowest rejected request index (~0 = none)
};

__device__ __forceinline__ void set_status(DevStatus *st, int code) { atomicCAS(&st->code, 0, code); }

// ------------------------------------------------------------ tables
// pair table entry (16 bytes): {left, right, rank, result}; empty: left = ~0
// whole-piece (vocabulary) table entry (16 bytes): the token's first
// VOCAB_INLINE bytes (little-endian words x, y, z, zero padded) and
// w = len << 20 | id; empty: w = 0 (no token is empty).  A probe of a piece
// of at most VOCAB_INLINE bytes reads one entry per slot and nothing else.
constexpr uint32_t PAIR_EMPTY = 0xFFFFFFFFu;
constexpr int MAX_VOCAB_BITS = 20;
constexpr int VOCAB_INLINE = 12;
constexpr int MAX_RANK_BITS = 24;

struct Tables {
  const uint16_t *cls1;       // code point >> 8 -> block index
  const uint8_t *cls2;        // block * 256 + (cp & 255) -> raw kind (K_*)
  const uint4 *pair_tab;       // {left, right, rank, result}
  uint32_t pair_mask;
  const int32_t *merge_result;
  const uint4 *vocab_tab;
  uint32_t vocab_mask;
  const uint8_t *vbytes;
  const int32_t *voff;
  const int32_t *byte_id;     // [256]
  const uint2 *ctx_tab;       // {ctx_key, lowest rank}: see ctx_key
  uint32_t ctx_mask;
  // the same for the byte tokens, indexed directly (a piece's first lookups):
  // bpair[b0 << 8 | b1] = {rank or -1, result} of the pair of byte tokens,
  // bctx[side << 16 | b << 8 | c] = the context table's entry for the byte
  // token b (INT_MAX: none)
  const int2 *bpair;
  const int32_t *bctx;
  int32_t max_tok_len;
  int32_t family;
  // added-token literals (n_lit == 0: none)
  const uint8_t *lit_bytes;
  const int32_t *lit_off;     // [n_lit + 1] into lit_bytes
  const int32_t *lit_order;   // literal indices by (first byte, length descending)
  const int32_t *lit_first;   // [257]: the lit_order range of each first byte
  int32_t n_lit;
};
constexpr int LIT_MAX_LEN = 255;       // bytes of one literal
constexpr int LIT_MAX_COUNT = 4095;    // literals (12-bit index)
enum : uint8_t { LIT_SEG = 1, LIT_INNER = 2 };   // per-byte marks of taken literals

TT_HD uint64_t mix64(uint64_t x) {
  x ^= x >> 33; x *= 0xff51afd7ed558ccdull;
  x ^= x >> 33; x *= 0xc4ceb9fe1a85ec53ull;
  x ^= x >> 33;
  return x;
}
// slot hash of a token pair: ids are below 2^20 and table masks below 2^32,
// so 32-bit multiply-xorshift mixing suffices (and costs a third of a 64-bit
// mix on the GPU)
TT_HD uint32_t pair_hash(uint32_t l, uint32_t r) {
  uint32_t h = l * 0x9E3779B1u ^ (r + 0x7F4A7C15u) * 0x85EBCA77u;
  h ^= h >> 16;
  h *= 0x7FEB352Du;
  h ^= h >> 15;
  return h;
}
TT_HD uint64_t pair_key(uint32_t l, uint32_t r) { return ((uint64_t)l << MAX_VOCAB_BITS) | r; }

// Context table of the out-of-order merges: for a token t and a byte c,
// side 0 holds the lowest rank of a merge (X, t) whose X ends with byte c
// (one that can take t from the left when c precedes it in the text), side
// 1 the lowest rank of a merge (t, Z) whose Z starts with byte c (one that
// can take t from the right when c follows it); no entry: no such merge.
constexpr uint32_t CTX_EMPTY = 0xFFFFFFFFu;
TT_HD uint32_t ctx_key(uint32_t t, uint32_t side, uint32_t c) { return (t << 9) | (side << 8) | c; }
TT_HD uint32_t ctx_hash(uint32_t k) {
  k *= 0x9E3779B1u;
  k ^= k >> 16;
  k *= 0x85EBCA77u;
  k ^= k >> 13;
  return k;
}

// hash of a byte string, 8 bytes at a time (little-endian words, zero padded)
struct ByteHash {
  uint64_t h;
  TT_HD void init(int len) { h = 0x9E3779B97F4A7C15ull ^ (uint64_t)len; }
  TT_HD void word(uint64_t w) { h = (h ^ w) * 0xff51afd7ed558ccdull; h ^= h >> 32; }
  TT_HD uint64_t fin() const { return mix64(h); }
};
TT_HD uint64_t hash_bytes(const uint8_t *b, int len) {
  ByteHash bh; bh.init(len);
  for (int i = 0; i < len; i += 8) {
    uint64_t w = 0;
    for (int k = 0; k < 8 && i + k < len; ++k) w |= (uint64_t)b[i + k] << (8 * k);
    bh.word(w);
  }
  return bh.fin();
}
// the whole-piece table entry of a token (len >= 1)
TT_HD void vocab_entry(const uint8_t *b, int len, int id, uint32_t out[4]) {
  out[0] = out[1] = out[2] = 0;
  for (int i = 0; i < len && i < VOCAB_INLINE; ++i) out[i / 4] |= (uint32_t)b[i] << (8 * (i % 4));
  out[3] = ((uint32_t)len << MAX_VOCAB_BITS) | (uint32_t)id;
}

#if defined(__CUDACC__)
// (rank, result) of the pair (l, r); rank -1 if (l, r) is not a merge
__device__ __forceinline__ int2 pair_lookup(const Tables &T, int l, int r) {
  uint32_t s = (uint32_t)pair_hash((uint32_t)l, (uint32_t)r) & T.pair_mask;
  for (;;) {
    const uint4 e = __ldg(&T.pair_tab[s]);
    if (e.x == PAIR_EMPTY) return make_int2(-1, -1);
    if (e.x == (uint32_t)l && e.y == (uint32_t)r) return make_int2((int)e.z, (int)e.w);
    s = (s + 1) & T.pair_mask;
  }
}
__device__ __forceinline__ int pair_rank(const Tables &T, int l, int r) { return pair_lookup(T, l, r).x; }

// 8 bytes starting at p, little-endian, bytes at or past `avail` zeroed
// (avail >= 1).  Reads only the 8-byte-aligned words that hold a byte of
// [p, p + min(avail, 8)); such a word never crosses a page, so no read can
// fault even at the very end of a buffer.
__device__ __forceinline__ uint64_t load8(const uint8_t *p, int avail) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint64_t *q = reinterpret_cast<const uint64_t *>(a & ~(uintptr_t)7);
  const int off = (int)(a & 7);
  uint64_t v = __ldg(q) >> (8 * off);
  if (off && avail > 8 - off) v |= __ldg(q + 1) << (64 - 8 * off);
  if (avail < 8) v &= (1ull << (8 * avail)) - 1;
  return v;
}


// ------------------------------------------------------------ memory order
__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// copy a trivially copyable struct through L2 (bypassing L1)
template <typename T>
__device__ __forceinline__ T ld_cg(const T *p) {
  static_assert(sizeof(T) % 4 == 0, "words");
  T out;
  uint32_t *o = reinterpret_cast<uint32_t *>(&out);
  const uint32_t *i = reinterpret_cast<const uint32_t *>(p);
#pragma unroll
  for (int k = 0; k < (int)(sizeof(T) / 4); ++k) o[k] = __ldcg(i + k);
  return out;
}

template <typename T>
__device__ __forceinline__ T shfl_up_t(T v, int d) {
  static_assert(sizeof(T) % 4 == 0, "words");
  uint32_t w[sizeof(T) / 4];
  memcpy(w, &v, sizeof(T));
#pragma unroll
  for (int k = 0; k < (int)(sizeof(T) / 4); ++k) w[k] = __shfl_up_sync(0xffffffffu, w[k], d);
  memcpy(&v, w, sizeof(T));
  return v;
}
template <typename T>
__device__ __forceinline__ T shfl_down_t(T v, int d) {
  uint32_t w[sizeof(T) / 4];
  memcpy(w, &v, sizeof(T));
#pragma unroll
  for (int k = 0; k < (int)(sizeof(T) / 4); ++k) w[k] = __shfl_down_sync(0xffffffffu, w[k], d);
  memcpy(&v, w, sizeof(T));
  return v;
}
template <typename T>
__device__ __forceinline__ T shfl_idx_t(T v, int src) {
  uint32_t w[sizeof(T) / 4];
  memcpy(w, &v, sizeof(T));
#pragma unroll
  for (int k = 0; k < (int)(sizeof(T) / 4); ++k) w[k] = __shfl_sync(0xffffffffu, w[k], src);
  memcpy(&v, w, sizeof(T));
  return v;
}

// Block-wide exclusive scan in thread order (NT threads, NT % 32 == 0).
// op(a, b) = "a then b".  Returns the exclusive prefix of this thread;
// *total receives the combination over all threads.  smem: NT/32 slots.
template <int NT, typename T, typename Op>
__device__ T block_exclusive_scan(T v, Op op, T identity, T *smem, T *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    T y = shfl_up_t(inc, d);
    if (lane >= d) inc = op(y, inc);
  }
  if (lane == 31) smem[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    T w = lane < NT / 32 ? smem[lane] : identity;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      T y = shfl_up_t(w, d);
      if (lane >= d) w = op(y, w);
    }
    if (lane < NT / 32) smem[lane] = w;       // inclusive over warps
  }
  __syncthreads();
  T warp_prefix = warp == 0 ? identity : smem[warp - 1];
  T excl_in_warp = shfl_up_t(inc, 1);
  if (lane == 0) excl_in_warp = identity;
  T r = op(warp_prefix, excl_in_warp);
  if (total) *total = smem[NT / 32 - 1];
  __syncthreads();
  return r;
}

// Block-wide exclusive suffix scan: the combination over threads AFTER this
// one, nearest first: op(near, far).  (Used with "first event" operators.)
template <int NT, typename T, typename Op>
__device__ T block_exclusive_suffix(T v, Op op, T identity, T *smem, T *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T inc = v;   // op over [me .. end of warp]
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    T y = shfl_down_t(inc, d);
    if (lane + d < 32) inc = op(inc, y);
  }
  if (lane == 0) smem[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    constexpr int NW = NT / 32;
    T w = lane < NW ? smem[lane] : identity;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      T y = shfl_down_t(w, d);
      if (lane + d < NW) w = op(w, y);
    }
    if (lane < NW) smem[lane] = w;            // suffix over warps, inclusive
  }
  __syncthreads();
  constexpr int NW = NT / 32;
  T warp_suffix = warp == NW - 1 ? identity : smem[warp + 1];
  T excl_in_warp = shfl_down_t(inc, 1);
  if (lane == 31) excl_in_warp = identity;
  T r = op(excl_in_warp, warp_suffix);
  if (total) *total = smem[0];
  __syncthreads();
  return r;
}

// Make a tile's aggregate (tile 0: its inclusive prefix) visible to its
// successors' look-back (one thread).
template <typename T>
__device__ __forceinline__ void lookback_publish(int tile, T local, T *agg, T *inc, int *flag) {
  if (tile == 0) {
    inc[0] = local;
    __threadfence();
    st_release(&flag[0], 2);
  } else {
    agg[tile] = local;
    __threadfence();
    st_release(&flag[tile], 1);
  }
}
// Decoupled look-back by one full warp (the warp that calls it; all 32 lanes
// must call).  Each step inspects the 32 nearest unread predecessors at once:
// a ballot finds the nearest one with an inclusive prefix, and the aggregates
// in between are combined by a warp reduction in tile order.  Returns the
// exclusive prefix on every lane; lane 0 publishes.  Tiles must be claimed
// in increasing order by running CTAs.  Every wait is bounded: after
// `spin_limit` polls the status records ST_TIMEOUT, *call_timeout is set (the
// later kernels of the call then withhold its outputs: a batch whose prefix
// is incomplete yields zero IDs, never approximate ones) and the walk stops
// with what it has, so no CTA can hang.  The prefix it then publishes is a
// partial sum of the predecessors' counts, never more than the true one, so
// indices derived from it stay inside the workspace.  With `published`, the
// tile's aggregate was already made visible by lookback_publish (so that the
// successors' look-back can start while this tile does other work).  With
// `withhold` (a test setting), the tile publishes nothing, so that its
// successors' waits run out.
template <typename T, typename Op>
__device__ T warp_lookback(int tile, T local, Op op, T identity, T *agg, T *inc, int *flag, DevStatus *st,
                           int *call_timeout, int spin_limit, bool published = false, bool withhold = false) {
  const int lane = threadIdx.x & 31;
  if (tile == 0) {
    if (lane == 0 && !published && !withhold) {
      inc[0] = local;
      __threadfence();
      st_release(&flag[0], 2);
    }
    __syncwarp();
    return identity;
  }
  if (lane == 0 && !published && !withhold) {
    agg[tile] = local;
    __threadfence();
    st_release(&flag[tile], 1);
  }
  T excl = identity;
  int top = tile - 1;                 // nearest predecessor not yet combined
  bool timed_out = false;
  for (;;) {
    const int t = top - lane;
    int f = t >= 0 ? ld_acquire(&flag[t]) : 2;
    int spins = 0;
    while (__any_sync(0xffffffffu, f == 0)) {
      if (++spins > spin_limit) { timed_out = true; break; }
      __nanosleep(64);
      if (f == 0) f = ld_acquire(&flag[t]);
    }
    if (timed_out) {
      if (lane == 0) {
        set_status(st, ST_TIMEOUT);
        atomicExch(call_timeout, 1);
      }
      break;
    }
    const unsigned incl = __ballot_sync(0xffffffffu, f == 2);
    const int first = incl ? __ffs(incl) - 1 : 32;   // nearest inclusive predecessor in this window
    T v = identity;
    if (t >= 0 && lane < first) v = ld_cg(&agg[t]);
    else if (t >= 0 && lane == first) v = ld_cg(&inc[t]);
    // combine in tile order: higher lanes are earlier tiles
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const T y = shfl_down_t(v, d);
      if (lane + d < 32) v = op(y, v);
    }
    v = shfl_idx_t(v, 0);
    excl = op(v, excl);
    if (first < 32) break;
    top -= 32;
  }
  if (lane == 0 && !withhold) {
    inc[tile] = op(excl, local);
    __threadfence();
    st_release(&flag[tile], 2);
  }
  __syncwarp();
  return excl;
}
#endif  // __CUDACC__

// Per-call arguments, read by every kernel from device memory (so that a
// captured graph can be replayed with new buffers).
struct CallArgs {
  const uint8_t *utf8;             // batch bytes (absolute)
  const int64_t *offs;             // [n + 1]
  int64_t n;                       // requests
  int32_t *out_ids;
  int64_t *out_id_offsets;         // [n + 1]
  int64_t *hook_starts;            // test hook outputs (NULL unless the hook runs)
  int64_t *hook_offsets;
  int32_t *out_spans;              // [2 * tokens]: (start, end) byte offsets from offs[0] per ID; NULL: none
  const uint8_t *utf8_src;         // the same bytes in page-locked host memory: the pre-pass reads them there
                                   // and copies each tile into utf8 (a buffer of the handle); NULL: none
  int64_t bound;                   // the caller's upper bound on the batch bytes (<= the workspace capacity):
                                   // a larger batch is refused on the device with ST_CAPACITY
};

#if defined(__CUDACC__)
// The batch's first byte offset and size, read from the per-call arguments.
// False when the batch is unsound (a negative offset or size) or larger than
// the bound the caller stated: every kernel then leaves the caller's buffers
// alone, except k_ids, which zeroes the ID offsets.
__device__ __forceinline__ bool batch_extent(const CallArgs &A, int64_t &base, int64_t &total) {
  base = __ldg(&A.offs[0]);
  total = __ldg(&A.offs[A.n]) - base;
  return !(total > A.bound || total < 0 || base < 0);
}
#endif

constexpr int CTR_TIMEOUT = 10;

// Per-stream workspace (device pointers; sizes fixed per capacity bucket).
struct Work {
  int64_t cap_bytes;               // largest batch this workspace holds
  int64_t cap_reqs;
  int32_t cap_tiles;
  int32_t spin_limit;              // polls before a look-back wait gives up (ST_TIMEOUT)
  int32_t withhold_tile;           // test setting: this pre-tokenizer tile never publishes (-1: none)
  // pre-pass summaries and carries
  int2 *s1_sum;                    // mark resolution: (last stretch start, last trigger)
  uint8_t *rq_sum;                 // [tiles][2]: first rq_ws / rq_up event
  // look-back state
  S2 *s2_agg, *s2_inc;
  int *s2_flag;
  int2 *cnt_agg, *cnt_inc;         // (pieces, last piece start * 2 + placeholder bit)
  int *cnt_flag;
  int *ids_agg, *ids_inc;          // per ID chunk: its ID count (summed by the BPE kernels), its first output
  int *counters;                   // [0] pretok tile ticket, [1] unused, [2] [7] [8] sizes of
                                   // the mid-length buckets 0..2, [3] pieces, [4] tokens, [5] bad
                                   // requests seen, [6] huge list size, [9] mid work ticket,
                                   // [CTR_TIMEOUT] a look-back wait of this call ran out
  // pieces and tokens
  int32_t *piece_start;            // [cap_bytes + 2], bit 31 = rejected-request placeholder
  int32_t *n_ids;                  // [cap_bytes + 1]
  int32_t *scratch;                // [cap_bytes] ids by byte position
  int32_t *tmp_a, *tmp_b, *tmp_c;  // [cap_bytes] long-piece work arrays
  int32_t *long_list;              // 3 buckets of LIST_CAP(cap_bytes) entries: pieces of
                                   // 129..256, 49..128 and 17..48 bytes
  int32_t *huge_list;              // [cap_bytes / (MID_MAX + 1) + 2] pieces > MID_MAX bytes
  uint8_t *bad;                    // [cap_reqs]
  int32_t *bad_pre;                // [cap_reqs + 1] (test hook)
  int32_t *req_piece;              // [cap_reqs + 1] first piece of each non-empty request
  int32_t *lit_cand;               // [cap_tiles * TILE] per tile, the positions (in the tile) of
                                   // literal candidates no earlier candidate reaches over
  int32_t *lit_cnt;                // [cap_tiles]
  uint8_t *lit_len;                // [cap_bytes + 8] longest literal starting at each byte (0: none)
  uint8_t *lit_flag;               // [cap_bytes + 8] LIT_SEG / LIT_INNER marks of taken literals
  DevStatus *status;
  CallArgs *args;
};

#if defined(__CUDACC__)
// A look-back wait of this call ran out: the kernels after the pre-tokenizer
// do no work and the call yields zero IDs for every request.
__device__ __forceinline__ bool call_timed_out(const Work &W) { return __ldcg(&W.counters[CTR_TIMEOUT]) != 0; }
#endif

}  // namespace tt
