// tt_bpe.cu - segmented byte-level BPE over the piece table and output
// compaction (TokTier: Exact Stateful CPU+GPU Tokenization for Agentic LLM
// Serving, §4.2 on BPE per piece and §4.3 on compacting the output).
//
// Every piece is encoded independently.  A piece whose bytes are a
// vocabulary entry is emitted as that one ID (the whole-piece shortcut).
// Otherwise merging proceeds in rounds: the lowest rank present among
// adjacent pairs names one pair, and every leftmost non-overlapping
// occurrence of it is merged in one sweep, together with every safe pair
// (one that no merge of lower rank can take a token from: see "safe pairs"
// below); only pairs next to a merge are looked up again.  With a
// well-ordered merge list (checked when the handle is created) the result
// equals merging the lowest-ranked leftmost pair one at a time.
//
// Execution units by piece length: a lane per piece of up to 16 bytes for
// the whole-piece probe, a miss merged by one lane (in batches, 32 queued
// misses side by side); a warp per piece of up to 256 bytes (in batches the
// pieces of 17..48 bytes four to a warp and of 49..128 bytes two to a warp;
// for a single request, one symbol a lane in registers up to 32 bytes, else
// a linked list in shared memory); a 512-thread block per longer piece (a
// linked list in shared memory up to 8 KiB, else global ping-pong buffers).
// IDs land in a byte-indexed scratch array, and each piece's ID count is
// also added into its 512-piece chunk's total; k_idscan (one CTA) scans the
// chunk totals, and k_ids scans each chunk's counts on its own, writes the
// final contiguous IDs and each request's ID offset.
#include <limits.h>

#include "tt_common.cuh"
#include "tt_kernels.h"

namespace tt {

#ifdef TT_TRACE
// ---------------------------------------------------------------- trace builds
// A library built with -DTT_TRACE (libtoktier_trace.so, never the product
// library) records one entry per ticket of the warp BPE kernel: the
// globaltimer (ns) at its start and end, its kind (0: a piece of 129..256
// bytes, 1: pieces of 49..128 bytes, 2: a chunk of short pieces with the
// misses merged during it, 3: pieces of 17..48 bytes, 4: a warp's last queued
// misses), its pieces, the longest of them and the most merge rounds the
// warp ran for one of them.  tt_trace_read (trace builds only) copies the
// records out and starts a new trace.
constexpr int TRACE_CAP = 1 << 20;
struct TraceRec {
  unsigned long long t0, t1;
  int kind, pieces, max_len, rounds;
};
__device__ TraceRec tt_trace_rec[TRACE_CAP];
__device__ int tt_trace_n;
__shared__ int tt_trace_rounds[BPE_WARP_THREADS / 32];
__device__ __forceinline__ unsigned long long trace_clock() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// a round of a warp-synchronous merge loop (counted once, by lane 0)
#define TT_TRACE_ROUND() \
  do { if ((threadIdx.x & 31) == 0) ++tt_trace_rounds[threadIdx.x >> 5]; } while (0)
// the rounds one lane took on its own
#define TT_TRACE_LANE_ROUNDS(r) atomicMax(&tt_trace_rounds[threadIdx.x >> 5], (r))
#else
#define TT_TRACE_ROUND() ((void)0)
#define TT_TRACE_LANE_ROUNDS(r) ((void)0)
#endif

// whole-piece vocabulary probe of len bytes at b (global memory): the hash
// of 8-byte words, then entries whose inline bytes and length match; only a
// token longer than VOCAB_INLINE bytes compares its remaining bytes in the
// token byte pool
__device__ __forceinline__ int vocab_probe(const Tables &T, const uint8_t *b, int len) {
  const uint64_t w0 = load8(b, len);
  const uint64_t w1 = len > 8 ? load8(b + 8, len - 8) : 0;
  ByteHash bh;
  bh.init(len);
  bh.word(w0);
  if (len > 8) bh.word(w1);
  for (int i = 16; i < len; i += 8) bh.word(load8(b + i, len - i));
  const uint32_t x = (uint32_t)w0, y = (uint32_t)(w0 >> 32), z = (uint32_t)w1;
  const uint32_t want_len = (uint32_t)len << MAX_VOCAB_BITS;
  uint32_t s = (uint32_t)bh.fin() & T.vocab_mask;
  for (;;) {
    const uint4 e = __ldg(&T.vocab_tab[s]);
    if (e.w == 0) return -1;
    if ((e.w & ~0xFFFFFu) == want_len && e.x == x && e.y == y && e.z == z) {
      const int id = (int)(e.w & 0xFFFFFu);
      if (len <= VOCAB_INLINE) return id;
      const uint8_t *v = T.vbytes + __ldg(&T.voff[id]);
      bool same = true;
      for (int i = VOCAB_INLINE; i < len && same; i += 8) same = load8(v + i, len - i) == load8(b + i, len - i);
      if (same) return id;
    }
    s = (s + 1) & T.vocab_mask;
  }
}

// the rest of a pair lookup whose first probe e (slot s) is already loaded
__device__ __forceinline__ int2 pair_finish(const Tables &T, uint4 e, uint32_t s, int l, int r) {
  for (;;) {
    if (e.x == PAIR_EMPTY) return make_int2(-1, -1);
    if (e.x == (uint32_t)l && e.y == (uint32_t)r) return make_int2((int)e.z, (int)e.w);
    s = (s + 1) & T.pair_mask;
    e = __ldg(&T.pair_tab[s]);
  }
}
__device__ __forceinline__ uint32_t pair_slot(const Tables &T, int l, int r) {
  return (uint32_t)pair_hash((uint32_t)l, (uint32_t)r) & T.pair_mask;
}

// ---------------------------------------------------------------- safe pairs
// Merges out of rank order, exact.  A pair x.y of rank q is safe when no
// merge of lower rank can take either token first: no merge (X, x) below q
// has X ending with the text byte before x, and no merge (y, Z) below q has
// Z starting with the byte after y (the context table).  Rank-ordered BPE
// then makes exactly this merge at rank q whatever it does elsewhere before,
// and every pair its result forms ranks above q (a merge's operands are made
// by lower ranks), so the pair can merge in any round.  A round merges the
// occurrences of the lowest rank r of all pairs (leftmost non-overlapping,
// as before) and every safe pair.  None of these overlap: two adjacent pairs
// are never both safe (each would need the other's rank to be the higher),
// and a safe pair of rank q >= r beside an occurrence of r would have a
// token that the merge of rank r can take.  A pair's key is 2 * rank + 1 if
// it is safe, 2 * rank if not, INT_MAX if it is no merge: the round minimum
// is the lowest rank's key.
__device__ __forceinline__ bool key_safe(int k) { return (k & 1) && k != INT_MAX; }

__device__ __forceinline__ uint32_t ctx_slot(const Tables &T, uint32_t key) { return ctx_hash(key) & T.ctx_mask; }
// the rest of a context lookup whose first probe e (slot s) is loaded:
// the lowest rank stored for key, INT_MAX if none
__device__ __forceinline__ int ctx_finish(const Tables &T, uint2 e, uint32_t s, uint32_t key) {
  for (;;) {
    if (e.x == key) return (int)e.y;
    if (e.x == CTX_EMPTY) return INT_MAX;
    s = (s + 1) & T.ctx_mask;
    e = __ldg(&T.ctx_tab[s]);
  }
}
// First probes of the pair (l, r) and of its two context entries, all in
// flight together; pb / nb: the text byte before l / after r, -1 at the
// piece's edge (nothing there can take the token).
struct PairProbe {
  uint4 e;
  uint2 el, er;
  uint32_t s, sl, sr;
};
__device__ __forceinline__ void probe_pair(const Tables &T, bool v, int l, int r, int pb, int nb, PairProbe &P) {
  P.s = pair_slot(T, l, r);
  P.sl = ctx_slot(T, ctx_key((uint32_t)l, 0, (uint32_t)pb & 255u));
  P.sr = ctx_slot(T, ctx_key((uint32_t)r, 1, (uint32_t)nb & 255u));
  P.e = v ? __ldg(&T.pair_tab[P.s]) : make_uint4(PAIR_EMPTY, 0, 0, 0);
  P.el = v && pb >= 0 ? __ldg(&T.ctx_tab[P.sl]) : make_uint2(CTX_EMPTY, 0);
  P.er = v && nb >= 0 ? __ldg(&T.ctx_tab[P.sr]) : make_uint2(CTX_EMPTY, 0);
}
// the pair's key (INT_MAX: no merge) and its merge result
__device__ __forceinline__ int probed_key(const Tables &T, const PairProbe &P, int l, int r, int pb, int nb,
                                          int &res) {
  const int2 pr = pair_finish(T, P.e, P.s, l, r);
  res = pr.y;
  if (pr.x < 0) return INT_MAX;
  const bool safe = (pb < 0 || ctx_finish(T, P.el, P.sl, ctx_key((uint32_t)l, 0, (uint32_t)pb)) > pr.x) &&
                    (nb < 0 || ctx_finish(T, P.er, P.sr, ctx_key((uint32_t)r, 1, (uint32_t)nb)) > pr.x);
  return 2 * pr.x + (safe ? 1 : 0);
}
// The key and result of the pair of byte tokens b0.b1 (the bytes at p and
// p + 1 of a piece), with the bytes pb before and nb after them (-1: the
// piece's edge), from the direct tables.
__device__ __forceinline__ int byte_pair_key(const Tables &T, int b0, int b1, int pb, int nb, int &res) {
  const int2 pr = __ldg(&T.bpair[b0 << 8 | b1]);
  const int cl = pb >= 0 ? __ldg(&T.bctx[b0 << 8 | pb]) : INT_MAX;
  const int cr = nb >= 0 ? __ldg(&T.bctx[65536 | b1 << 8 | nb]) : INT_MAX;
  res = pr.y;
  if (pr.x < 0) return INT_MAX;
  return 2 * pr.x + (cl > pr.x && cr > pr.x ? 1 : 0);
}
// the text byte at i of a piece of n bytes, -1 outside it
__device__ __forceinline__ int byte_at(const uint8_t *b, int i, int n) { return i >= 0 && i < n ? (int)__ldg(b + i) : -1; }

// Round merging of up to 32 / G pieces of at most G bytes at once, G lanes
// per piece and one symbol per lane: lane p of a group holds the symbol that
// starts at byte p (while alive), the rank and result of the pair it starts
// with the next alive lane.  Neighbours come from a ballot of alive lanes.
// A round: group min of the ranks (r); occurrences of r whose previous alive
// lane is not itself an occurrence take their merge result and unlink their
// right neighbour; leftover occurrences (inside runs of (a, a)) repeat with
// the same r; lanes whose pair changed look it up again.  All 32 lanes take
// part; a group with len 0 idles.  Writes the group's IDs to out[0..] and
// returns their count (on every lane of the group).
template <int G>
__device__ __forceinline__ int bpe_lanes(const Tables &T, const uint8_t *bytes, int len, int32_t *out) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr unsigned GM = G == 32 ? FULL : ((1u << G) - 1);
  const int lane = threadIdx.x & 31;
  const int p = lane % G, sh = lane - p;
  const unsigned below = (1u << p) - 1, above_me = ~((2u << p) - 1);
  bool alive = p < len;
  int tok = alive ? __ldg(&T.byte_id[__ldg(bytes + p)]) : -1;
  int rank = INT_MAX, res = 0;                 // the key of my pair (2 * rank + safe) and its result
  if (p + 1 < len)                            // a pair of byte tokens: the direct tables
    rank = byte_pair_key(T, __ldg(bytes + p), __ldg(bytes + p + 1), byte_at(bytes, p - 1, len),
                         byte_at(bytes, p + 2, len), res);
  for (int round = 0; round < G; ++round) {   // each round unlinks at least one symbol
    TT_TRACE_ROUND();
    int r = rank;
#pragma unroll
    for (int d = G / 2; d >= 1; d >>= 1) r = min(r, __shfl_xor_sync(FULL, r, d));
    if (__all_sync(FULL, r == INT_MAX)) break;
    for (int step = 0; step < G; ++step) {
      const unsigned am = (__ballot_sync(FULL, alive) >> sh) & GM;
      const unsigned lo = am & below;
      const int pvl = lo ? 31 - __clz(lo) : -1;
      const bool safe = alive && key_safe(rank);
      const bool hit = alive && !safe && rank == r && r != INT_MAX;
      const unsigned hm = (__ballot_sync(FULL, hit) >> sh) & GM;
      const bool sel = safe || (hit && !(pvl >= 0 && ((hm >> pvl) & 1u)));
      const unsigned sm = (__ballot_sync(FULL, sel) >> sh) & GM;
      const bool pending = hit && !sel;
      if (sel) tok = res;
      if (alive && pvl >= 0 && ((sm >> pvl) & 1u)) { alive = false; rank = INT_MAX; }
      const unsigned am2 = (__ballot_sync(FULL, alive) >> sh) & GM;
      const unsigned hi = am2 & above_me;
      const int nxl = hi ? __ffs(hi) - 1 : -1;
      const int tn = __shfl_sync(FULL, tok, sh + (nxl < 0 ? p : nxl));
      if (alive && (sel || (nxl >= 0 && ((sm >> nxl) & 1u)))) {
        if (nxl < 0) {
          rank = INT_MAX;
        } else {
          const int2 pr = pair_lookup(T, tok, tn);
          rank = pr.x < 0 ? INT_MAX : 2 * pr.x;
          res = pr.y;
        }
      }
      if (!__any_sync(FULL, pending)) break;
    }
  }
  const unsigned fm = (__ballot_sync(FULL, alive) >> sh) & GM;
  if (alive) out[__popc(fm & below)] = tok;
  return __popc(fm);
}

// ---------------------------------------------------------------- warp kernel
// Every piece of at most MID_MAX bytes, in one persistent kernel whose warps
// take tickets from one counter, the longest expected work first: the pieces
// of 49 .. MID_MAX bytes that k_pretok listed (a warp per piece), then chunks
// of 32 consecutive pieces, where each lane tries the whole-piece shortcut
// for its piece of at most SMALL_MAX bytes and the warp merges the misses two
// at a time, 16 lanes per piece, then the listed pieces of SMALL_MAX+1 .. 48
// bytes.  Longer pieces are left to k_bpe_long, which runs beside this
// kernel.
//
// A listed piece of at most 32 bytes runs bpe_lanes<32>; a longer one is a
// doubly linked list over fixed positions in shared memory (lane l owns
// positions l, l + 32, ...), each alive position holding its token and the
// rank and result of the pair it starts.  A round: warp min of the ranks
// (r); every occurrence of r whose predecessor is not itself an occurrence
// merges in place (its right neighbour is unlinked) and looks up the two
// pairs it touches.  Occurrences left over -- only inside runs of a pair
// (a, a) -- repeat that step with the same r, which takes every other member
// of a run from its left end: the leftmost non-overlapping set.  Pairs made
// by a merge rank above r (well-ordered list), so they never join a run.
constexpr int WARP_KERNEL_WARPS = BPE_WARP_THREADS / 32;

// workspaces above this size (batches; the single request stays below) pair
// the pieces of 49..128 bytes
constexpr int64_t PAIR_MIN_CAP_BYTES = 4ll << 20;
constexpr int GROUP2 = 4;   // pieces of 17..48 bytes a warp when grouped (8 lanes x 6 positions each)
constexpr int SMALL_CHUNK = 32;   // pieces per small-piece ticket (IDS_CHUNK is a multiple)
static_assert(IDS_CHUNK % SMALL_CHUNK == 0, "a small-piece ticket lies in one ID chunk");

// A piece's ID count, also added into the total of its ID chunk (IDS_CHUNK
// pieces), which the ID scatter's chunk scan reads.
__device__ __forceinline__ void put_count(const Work &W, int k, int c) {
  W.n_ids[k] = c;
  if (c) atomicAdd(&W.ids_agg[k / IDS_CHUNK], c);
}

// ---------------------------------------------------------------- short misses
// A short piece that is no token is merged by one lane on its own: the
// pieces of a warp's short-piece chunks that miss the whole-piece table
// queue up in the warp's MissQueue, and every 32 of them are merged side by
// side, one per lane.  A lane holds its piece as a compact array of packed
// words -- key of the pair the position starts << 40 | that pair's merge
// result << 20 | token, with RANK_NIL for no pair or no merge -- in the
// warp's shared arrays, word i of lane l at v[32 * i + l] (conflict-free).
// Keys as in the linked lists (2 * rank + safe), the safe bit found only for
// the first pairs, from the direct tables (for pieces this short, context
// probes at every lookup cost more than the rounds they save).  A round: the
// lowest key r over the array; one pass that merges every leftmost
// non-overlapping occurrence of r and every safe pair, and compacts; then
// lookups of the pairs next to a merge, four first probes in flight at a
// time.
constexpr uint32_t RANK_NIL = 0xFFFFFFu;   // no rank: 2^24 - 1 is above every rank
constexpr int MISS_QUEUE = 2 * 32;          // < 32 left over plus one chunk's 32
struct MissQueue {
  int32_t piece[MISS_QUEUE], start[MISS_QUEUE];
  uint8_t len[MISS_QUEUE];
};
__device__ __forceinline__ uint64_t pack_pos(uint32_t rank, uint32_t res, uint32_t tok) {
  return ((uint64_t)rank << 40) | ((uint64_t)res << 20) | tok;
}
__device__ __forceinline__ uint32_t pos_rank(uint64_t w) { return (uint32_t)(w >> 40); }
__device__ __forceinline__ uint32_t pos_res(uint64_t w) { return (uint32_t)(w >> 20) & 0xFFFFFu; }
__device__ __forceinline__ uint32_t pos_tok(uint64_t w) { return (uint32_t)w & 0xFFFFFu; }

// the rank and result of the pairs (i, i + 1) for the set bits i of need
__device__ __forceinline__ void seq_lookups(const Tables &T, uint64_t *v, uint32_t need) {
  const int lane = threadIdx.x & 31;
  while (need) {
    int at[4];
    uint32_t sl[4], l[4], r[4];
    uint4 e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      at[q] = need ? __ffs(need) - 1 : -1;
      need &= need - 1;
      l[q] = r[q] = 0;
      sl[q] = 0;
      e[q] = make_uint4(PAIR_EMPTY, 0, 0, 0);
      if (at[q] >= 0) {
        l[q] = pos_tok(v[32 * at[q] + lane]);
        r[q] = pos_tok(v[32 * (at[q] + 1) + lane]);
        sl[q] = pair_slot(T, (int)l[q], (int)r[q]);
        e[q] = __ldg(&T.pair_tab[sl[q]]);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (at[q] >= 0) {
        const int2 pr = pair_finish(T, e[q], sl[q], (int)l[q], (int)r[q]);
        v[32 * at[q] + lane] = pr.x < 0 ? pack_pos(RANK_NIL, 0, l[q]) : pack_pos(2u * (uint32_t)pr.x, (uint32_t)pr.y, l[q]);
      }
    }
  }
}

// BPE of the n <= SMALL_MAX bytes at b by this lane alone: writes the IDs to
// out and returns their count.
__device__ __forceinline__ int seq_bpe(const Tables &T, const uint8_t *b, int n, uint64_t *v, int32_t *out) {
  const int lane = threadIdx.x & 31;
  // the first pairs are pairs of byte tokens (the direct tables, keys with
  // the safe bit); later lookups leave it clear
  int bp = -1, b0 = __ldg(b), b1 = n > 1 ? __ldg(b + 1) : -1;
  for (int i = 0; i < n; ++i) {
    const int b2 = i + 2 < n ? __ldg(b + i + 2) : -1;
    int rs = 0;
    const int key = b1 >= 0 ? byte_pair_key(T, b0, b1, bp, b2, rs) : INT_MAX;
    const uint32_t t = (uint32_t)__ldg(&T.byte_id[b0]);
    v[32 * i + lane] = key == INT_MAX ? pack_pos(RANK_NIL, 0, t) : pack_pos((uint32_t)key, (uint32_t)rs, t);
    bp = b0; b0 = b1; b1 = b2;
  }
  int m = n;
  int rounds = 0;
  for (int round = 0; round < n; ++round) {   // each round merges at least one pair
    uint32_t r = RANK_NIL;
    for (int i = 0; i + 1 < m; ++i) r = min(r, pos_rank(v[32 * i + lane]));
    if (r == RANK_NIL) break;
    ++rounds;
    // merge every leftmost non-overlapping occurrence of r, compacting; the
    // pairs a merge touches are looked up again
    int w = 0;
    uint32_t need = 0;
    for (int i = 0; i < m; ++w) {
      const uint64_t x = v[32 * i + lane];
      const uint32_t k = pos_rank(x);
      if (i + 1 < m && (k == r || ((k & 1) && k != RANK_NIL))) {
        v[32 * w + lane] = pack_pos(RANK_NIL, 0, pos_res(x));
        need |= (1u << w) | (w ? 1u << (w - 1) : 0u);
        i += 2;
      } else {
        v[32 * w + lane] = x;
        i += 1;
      }
    }
    m = w;
    seq_lookups(T, v, need & ((1u << (m - 1)) - 1));   // no pair starts at the last position
  }
  TT_TRACE_LANE_ROUNDS(rounds);
  (void)rounds;
  for (int i = 0; i < m; ++i) out[i] = (int32_t)pos_tok(v[32 * i + lane]);
  return m;
}

// Merge the first cnt (<= 32) queued misses, one per lane.
__device__ __forceinline__ void run_misses(const Tables &T, const Work &W, const uint8_t *g, const MissQueue &Q,
                                           int cnt, uint64_t *v) {
  const int lane = threadIdx.x & 31;
  if (lane < cnt) {
    const int k = Q.piece[lane], s = Q.start[lane];
    const int c = seq_bpe(T, g + s, Q.len[lane], v, W.scratch + s);
    W.n_ids[k] = c;
    atomicAdd(&W.ids_agg[k / IDS_CHUNK], c);
  }
  __syncwarp();
}

// R chunks of 32 consecutive pieces from kb on: each lane tries the
// whole-piece shortcut for its piece of at most SMALL_MAX bytes (longer ones
// are listed by k_pretok) and the misses join the warp's queue; 32 queued
// misses are merged as soon as they are there.  QUEUE: the rest stay queued
// (batches: full warps); else they are merged at the end of the ticket (a
// single request, whose latency a queue's leftovers at the end of the
// kernel would lengthen).  qn: the queue's length (warp-uniform).
template <bool QUEUE>
__device__ __forceinline__ void small_chunk(const Tables &T, const Work &W, const uint8_t *g, int64_t total, int np,
                                            int kb, int R, MissQueue &Q, int &qn, uint64_t *v) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < R; ++r) {
    const int k = kb + 32 * r + lane;
    int32_t s = 0;
    int len = 0;
    bool miss = false;
    int mine = 0;                               // IDs this lane wrote counts for
    if (k < np) {
      s = __ldcg(&W.piece_start[k]);
      if (s < 0) {
        W.n_ids[k] = 0;                                                // rejected request
      } else {
        const int32_t e = __ldcg(&W.piece_start[k + 1]) & 0x7FFFFFFF;
        len = e - s;
        if (len <= 0 || e > total) {
          W.n_ids[k] = 0;
          set_status(W.status, ST_INVALID_ARG);
        } else if (len <= SMALL_MAX) {
          const int id = len <= T.max_tok_len ? vocab_probe(T, g + s, len) : -1;
          if (id >= 0) {
            W.scratch[s] = id;
            W.n_ids[k] = 1;
            mine = 1;
          } else {
            miss = true;
          }
        }
      }
    }
    // the hits' counts, all in one ID chunk
#pragma unroll
    for (int d = 16; d; d >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, d);
    if (lane == 0 && mine) atomicAdd(&W.ids_agg[kb / IDS_CHUNK], mine);
    const unsigned mm = __ballot_sync(0xffffffffu, miss);
    if (miss) {
      const int at = qn + __popc(mm & ((1u << lane) - 1));
      Q.piece[at] = k;
      Q.start[at] = s;
      Q.len[at] = (uint8_t)len;
    }
    qn += __popc(mm);
    __syncwarp();
    if (qn >= 32) {
      run_misses(T, W, g, Q, 32, v);
      const bool mv = lane < qn - 32;           // move the rest to the front
      int rk = 0, rs = 0, rl = 0;
      if (mv) { rk = Q.piece[32 + lane]; rs = Q.start[32 + lane]; rl = Q.len[32 + lane]; }
      __syncwarp();
      if (mv) { Q.piece[lane] = rk; Q.start[lane] = rs; Q.len[lane] = (uint8_t)rl; }
      __syncwarp();
      qn -= 32;
    }
  }
  if (!QUEUE && qn) {
    run_misses(T, W, g, Q, qn, v);
    qn = 0;
  }
}

// After a merge at position p of a linked list over a piece of n bytes at b:
// the keys and results of the pairs (a, p) and (p, c) beside it, all their
// probes in flight together.  CTX: test safety (else the keys say "not
// safe", which is always exact).
template <bool CTX = true>
__device__ __forceinline__ void relink_lookups(const Tables &T, const uint8_t *b, int n, int p, const int32_t *tok,
                                               int32_t *rank, int32_t *res, const int16_t *nx, const int16_t *pv) {
  const int a = pv[p], c = nx[p];
  const int tp = tok[p];
  const int ta = a >= 0 ? tok[a] : 0, tc = c < n ? tok[c] : 0;
  if (!CTX) {
    const uint32_t sa = pair_slot(T, ta, tp), sc = pair_slot(T, tp, tc);
    const uint4 ea = a >= 0 ? __ldg(&T.pair_tab[sa]) : make_uint4(PAIR_EMPTY, 0, 0, 0);
    const uint4 ec = c < n ? __ldg(&T.pair_tab[sc]) : make_uint4(PAIR_EMPTY, 0, 0, 0);
    if (a >= 0) {
      const int2 pr = pair_finish(T, ea, sa, ta, tp);
      rank[a] = pr.x < 0 ? INT_MAX : 2 * pr.x;
      res[a] = pr.y;
    }
    if (c < n) {
      const int2 pr = pair_finish(T, ec, sc, tp, tc);
      rank[p] = pr.x < 0 ? INT_MAX : 2 * pr.x;
      res[p] = pr.y;
    }
    return;
  }
  const int e = c < n ? nx[c] : n;
  const int pba = a >= 0 ? byte_at(b, a - 1, n) : -1, nba = byte_at(b, c, n);   // around (a, p)
  const int pbc = byte_at(b, p - 1, n), nbc = c < n ? byte_at(b, e, n) : -1;      // around (p, c)
  PairProbe Pa, Pc;
  probe_pair(T, a >= 0, ta, tp, pba, nba, Pa);
  probe_pair(T, c < n, tp, tc, pbc, nbc, Pc);
  int rs;
  if (a >= 0) {
    rank[a] = probed_key(T, Pa, ta, tp, pba, nba, rs);
    res[a] = rs;
  }
  if (c < n) {
    rank[p] = probed_key(T, Pc, tp, tc, pbc, nbc, rs);
    res[p] = rs;
  }
}

// The linked-list rounds of one piece of n bytes (32 < n <= 32 * NS) in the
// warp's shared arrays, NS positions per lane (lane l owns l, l + 32, ...);
// writes the IDs to out and returns their count.  The ranks of a lane's own
// positions are read once per step into registers.
template <int NS>
__device__ __forceinline__ int list_rounds(const Tables &T, const uint8_t *b, int n, int32_t *out, int32_t *tok,
                                           int32_t *rank, int32_t *res, int16_t *nx, int16_t *pv) {
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1;
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int p = lane + 32 * k;
    tok[p] = p < n ? __ldg(&T.byte_id[__ldg(b + p)]) : -1;
    rank[p] = INT_MAX;
    nx[p] = (int16_t)(p + 1);
    pv[p] = (int16_t)(p - 1);
  }
  __syncwarp();
  // initial pair lookups (pairs of byte tokens: the direct tables)
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int p = lane + 32 * k;
    if (p + 1 < n) {
      int rs;
      rank[p] = byte_pair_key(T, __ldg(b + p), __ldg(b + p + 1), byte_at(b, p - 1, n), byte_at(b, p + 2, n), rs);
      res[p] = rs;
    }
  }
  __syncwarp();
  for (int round = 0; round < n; ++round) {   // each round unlinks at least one symbol
    TT_TRACE_ROUND();
    int rr[NS];
    int lm = INT_MAX;
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      rr[k] = rank[lane + 32 * k];
      lm = min(lm, rr[k]);
    }
    const int r = __reduce_min_sync(0xffffffffu, lm);
    if (r == INT_MAX) break;
    for (int step = 0; step < n; ++step) {
      if (step > 0) {                         // ranks changed in the previous step
#pragma unroll
        for (int k = 0; k < NS; ++k) rr[k] = rank[lane + 32 * k];
      }
      uint32_t sel = 0;
      bool left = false;
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        if (key_safe(rr[k])) {
          sel |= 1u << k;
        } else if (rr[k] == r) {
          const int q = pv[lane + 32 * k];
          if (q < 0 || rank[q] != r) sel |= 1u << k;
          else left = true;
        }
      }
      __syncwarp();
      for (uint32_t m = sel; m; m &= m - 1) {
        const int p = lane + 32 * (__ffs(m) - 1);
        const int q = nx[p], nq = nx[q];
        tok[p] = res[p];
        tok[q] = -1;
        rank[q] = INT_MAX;
        rank[p] = INT_MAX;
        nx[p] = (int16_t)nq;
        if (nq < n) pv[nq] = (int16_t)p;
      }
      __syncwarp();
      for (uint32_t m = sel; m; m &= m - 1) {
        const int p = lane + 32 * (__ffs(m) - 1);
        relink_lookups(T, b, n, p, tok, rank, res, nx, pv);
      }
      __syncwarp();
      if (!__any_sync(0xffffffffu, left)) break;
    }
  }
  // surviving tokens in position order
  int cnt = 0;
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int t = tok[lane + 32 * k];
    const unsigned bal = __ballot_sync(0xffffffffu, t >= 0);
    if (t >= 0) out[cnt + __popc(bal & lt_mask)] = t;
    cnt += __popc(bal);
  }
  __syncwarp();
  return cnt;
}

// 32 / G pieces side by side, G lanes each (group q of the warp takes piece
// q; lane l of a group owns positions l, l + G, ...), each group on its own
// share of the warp's arrays.  Rounds run in lockstep: each group takes its
// own lowest rank (an xor butterfly over its lanes) and merges as list_rounds
// does; a group with nothing left idles until the others are done.  Each
// group passes its own piece (n = 0: none) and gets its IDs' count.  For
// batches, where warps are the scarce resource: a round's instructions serve
// several pieces.
// NS: positions per lane (pieces of at most G * NS bytes).  CTX: the
// lookups after a merge test safety (groups of 16 lanes); the groups of 8
// lanes (pieces of 17..48 bytes, four a warp) find it for their first pairs
// only, which measured faster for them (burst k_bpe_warp 0.468 -> 0.447 ms,
// o200k-style batch 1.59 -> 1.56 ms) and slower for the groups of 16 (0.468
// -> 0.526 ms).
constexpr int PAIR_MAX = MID_MAX / 2;
template <int G, int NS, bool CTX = (G >= 16)>
__device__ __forceinline__ int group_rounds(const Tables &T, const uint8_t *b, int n, int32_t *out, int32_t *tok,
                                            int32_t *rank, int32_t *res, int16_t *nx, int16_t *pv) {
  static_assert(G * NS <= MID_MAX * G / 32, "a group's share of the arrays");
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int SHARE = MID_MAX * G / 32;
  const int lane = threadIdx.x & 31, hl = lane % G;
  const unsigned lt_mask = (1u << hl) - 1;
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int p = hl + G * k;
    tok[p] = p < n ? __ldg(&T.byte_id[__ldg(b + p)]) : -1;
    rank[p] = INT_MAX;
    nx[p] = (int16_t)(p + 1);
    pv[p] = (int16_t)(p - 1);
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < NS; ++k) {              // initial lookups (pairs of byte tokens: the direct tables)
    const int p = hl + G * k;
    if (p + 1 < n) {
      int rs;
      rank[p] = byte_pair_key(T, __ldg(b + p), __ldg(b + p + 1), byte_at(b, p - 1, n), byte_at(b, p + 2, n), rs);
      res[p] = rs;
    }
  }
  __syncwarp();
  for (int round = 0; round < SHARE; ++round) {      // a group with pairs unlinks at least one symbol a round
    TT_TRACE_ROUND();
    int rr[NS];
    int r = INT_MAX;
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      rr[k] = rank[hl + G * k];
      r = min(r, rr[k]);
    }
#pragma unroll
    for (int d = G / 2; d >= 1; d >>= 1) r = min(r, __shfl_xor_sync(FULL, r, d));   // my group's lowest rank
    if (__all_sync(FULL, r == INT_MAX)) break;
    for (int step = 0; step < SHARE; ++step) {      // (a bound the same on every lane: the loop holds warp votes)
      if (step > 0) {
#pragma unroll
        for (int k = 0; k < NS; ++k) rr[k] = rank[hl + G * k];
      }
      uint32_t sel = 0;
      bool left = false;
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        if (key_safe(rr[k])) {
          sel |= 1u << k;
        } else if (r != INT_MAX && rr[k] == r) {
          const int q = pv[hl + G * k];
          if (q < 0 || rank[q] != r) sel |= 1u << k;
          else left = true;
        }
      }
      __syncwarp();
      for (uint32_t m = sel; m; m &= m - 1) {
        const int p = hl + G * (__ffs(m) - 1);
        const int q = nx[p], nq = nx[q];
        tok[p] = res[p];
        tok[q] = -1;
        rank[q] = INT_MAX;
        rank[p] = INT_MAX;
        nx[p] = (int16_t)nq;
        if (nq < n) pv[nq] = (int16_t)p;
      }
      __syncwarp();
      for (uint32_t m = sel; m; m &= m - 1) {
        const int p = hl + G * (__ffs(m) - 1);
        relink_lookups<CTX>(T, b, n, p, tok, rank, res, nx, pv);
      }
      __syncwarp();
      if (!__any_sync(FULL, left)) break;
    }
  }
  // surviving tokens of my group in position order
  int cnt = 0;
  const int sh = lane - hl;
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int t = tok[hl + G * k];
    const unsigned bal = (__ballot_sync(FULL, t >= 0) >> sh) & (G == 32 ? FULL : (1u << G) - 1);
    if (t >= 0) out[cnt + __popc(bal & lt_mask)] = t;
    cnt += __popc(bal);
  }
  __syncwarp();
  return cnt;
}

// 32 / G listed pieces of at most G * NS bytes on one warp -- entries
// first .. first + 32 / G - 1 of a list of n_list pieces (past n_list: none): each
// group probes its piece whole, then the misses merge side by side.
template <int G, int NS>
__device__ __forceinline__ void mid_group(const Tables &T, const Work &W, const uint8_t *g, const int32_t *list,
                                          int first, int n_list, int32_t *tok, int32_t *rank, int32_t *res,
                                          int16_t *nx, int16_t *pv) {
  const int lane = threadIdx.x & 31, grp = lane / G, gl = lane % G;
  const int pc = first + grp < n_list ? __ldcg(&list[first + grp]) : -1;
  int32_t s = 0;
  int n = 0;
  if (pc >= 0) {
    s = __ldcg(&W.piece_start[pc]);
    n = (__ldcg(&W.piece_start[pc + 1]) & 0x7FFFFFFF) - s;
  }
  const uint8_t *b = g + s;
  int id = -1;
  if (gl == 0 && n > 0 && n <= T.max_tok_len) id = vocab_probe(T, b, n);
  id = __shfl_sync(0xffffffffu, id, lane - gl);
  if (id >= 0) {
    if (gl == 0) { W.scratch[s] = id; put_count(W, pc, 1); }
    n = 0;                                    // this group idles
  }
  const int off = grp * (MID_MAX * G / 32);
  const int cnt = group_rounds<G, NS>(T, b, n, W.scratch + s, tok + off, rank + off, res + off, nx + off, pv + off);
  if (gl == 0 && n > 0) put_count(W, pc, cnt);
  __syncwarp();
}

__device__ __forceinline__ void mid_piece(const Tables &T, const Work &W, const uint8_t *g, int pc, int32_t *tok,
                                          int32_t *rank, int32_t *res, int16_t *nx, int16_t *pv) {
  const int lane = threadIdx.x & 31;
  const int32_t s = __ldcg(&W.piece_start[pc]);
  const int32_t e = __ldcg(&W.piece_start[pc + 1]) & 0x7FFFFFFF;
  const int n = e - s;
  const uint8_t *b = g + s;
  if (n <= T.max_tok_len) {
    int id = 0;
    if (lane == 0) id = vocab_probe(T, b, n);
    id = __shfl_sync(0xffffffffu, id, 0);
    if (id >= 0) {
      if (lane == 0) { W.scratch[s] = id; put_count(W, pc, 1); }
      return;
    }
  }
  if (n <= 32) {                              // one symbol per lane, state in registers
    const int cnt = bpe_lanes<32>(T, b, n, W.scratch + s);
    if (lane == 0) put_count(W, pc, cnt);
    return;
  }
  int cnt;
  switch ((n + 31) >> 5) {                    // 2 .. MID_MAX / 32 positions per lane
    case 2: cnt = list_rounds<2>(T, b, n, W.scratch + s, tok, rank, res, nx, pv); break;
    case 3: cnt = list_rounds<3>(T, b, n, W.scratch + s, tok, rank, res, nx, pv); break;
    case 4: cnt = list_rounds<4>(T, b, n, W.scratch + s, tok, rank, res, nx, pv); break;
    case 5: cnt = list_rounds<5>(T, b, n, W.scratch + s, tok, rank, res, nx, pv); break;
    case 6: cnt = list_rounds<6>(T, b, n, W.scratch + s, tok, rank, res, nx, pv); break;
    case 7: cnt = list_rounds<7>(T, b, n, W.scratch + s, tok, rank, res, nx, pv); break;
    default: cnt = list_rounds<8>(T, b, n, W.scratch + s, tok, rank, res, nx, pv); break;
  }
  if (lane == 0) put_count(W, pc, cnt);
  __syncwarp();
}

// PAIRS: which listed pieces go two to a warp: 0 none (a single request,
// whose longest merge chains set its latency: pairing even the short pieces
// measured slower there), 1 those of 17..48 bytes, 2 those of 17..48 and of
// 49..128 bytes (batches).
// Each warp's merge arrays (a listed piece of up to MID_MAX bytes: token,
// -1 once unlinked; rank of (p, next), INT_MAX if none; its merge result;
// the list links), which also hold the packed words of 32 short misses.
struct __align__(16) WarpArrays {
  int32_t tok[MID_MAX], rank[MID_MAX], res[MID_MAX];
  int16_t nx[MID_MAX], pv[MID_MAX];
};
static_assert(sizeof(WarpArrays) >= 32 * SMALL_MAX * sizeof(uint64_t), "room for 32 short misses");

template <int PAIRS>
__global__ void __launch_bounds__(BPE_WARP_THREADS, BPE_WARP_CTAS_PER_SM) k_bpe_warp(Tables T, Work W) {
  __shared__ WarpArrays wa[WARP_KERNEL_WARPS];
  __shared__ MissQueue mq[WARP_KERNEL_WARPS];
  const CallArgs A = *W.args;
  if (A.n <= 0) return;
  int64_t base, total;
  if (!batch_extent(A, base, total) || call_timed_out(W)) return;
  const int np = __ldcg(&W.counters[3]);
  const int c0 = __ldcg(&W.counters[mid_bucket_counter(0)]), c1 = __ldcg(&W.counters[mid_bucket_counter(1)]);
  const int c2 = __ldcg(&W.counters[mid_bucket_counter(2)]);
  // ticket order, the longest work a ticket first: listed pieces of
  // 129..256 and 49..128 bytes, listed pieces of 17..48 bytes, then the
  // chunks of short pieces (the shortest tickets, which even out the end of
  // the kernel).  In batches the pieces of 49..128 bytes go two to a ticket
  // and those of 17..48 bytes GROUP2 to a ticket.
  const int tb1 = PAIRS >= 2 ? (c1 + 1) / 2 : c1, tb2 = PAIRS >= 1 ? (c2 + GROUP2 - 1) / GROUP2 : c2;
  // a single request with more chunks of short pieces than the grid has
  // warps takes two chunks a ticket (their misses merged together: fuller
  // lanes, 1M-char request 0.087 -> 0.078 ms); a smaller one keeps one
  // chunk a ticket for more tickets in flight
  const int R = PAIRS == 0 && (int64_t)np > (int64_t)SMALL_CHUNK * gridDim.x * (blockDim.x / 32) ? 2 : 1;
  const int CH = SMALL_CHUNK * R;
  const int t1 = c0 + tb1, t2 = t1 + tb2, nwork = t2 + (np + CH - 1) / CH;
  const int64_t lcap = list_cap(W.cap_bytes);
  const uint8_t *g = A.utf8 + base;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t *s_tok = wa[warp].tok, *s_rank = wa[warp].rank, *s_res = wa[warp].res;
  int16_t *s_nx = wa[warp].nx, *s_pv = wa[warp].pv;
  uint64_t *v = reinterpret_cast<uint64_t *>(&wa[warp]);
  int qn = 0;                                   // queued short misses (warp-uniform)
  for (;;) {
    int gi = 0;
    if (lane == 0) gi = atomicAdd(&W.counters[9], 1);
    gi = __shfl_sync(0xffffffffu, gi, 0);
    if (gi >= nwork) break;
#ifdef TT_TRACE
    if (lane == 0) tt_trace_rounds[warp] = 0;
    __syncwarp();
    const unsigned long long tr0 = trace_clock();
#endif
    if (PAIRS >= 2 && gi >= c0 && gi < t1) {     // pieces of 49..128 bytes, two a ticket
      mid_group<16, PAIR_MAX / 16>(T, W, g, W.long_list + lcap, 2 * (gi - c0), c1, s_tok, s_rank, s_res, s_nx,
                                   s_pv);
    } else if (PAIRS >= 1 && gi >= t1 && gi < t2) {   // pieces of 17..48 bytes, GROUP2 a ticket
      mid_group<32 / GROUP2, (48 * GROUP2 + 31) / 32>(T, W, g, W.long_list + 2 * lcap, GROUP2 * (gi - t1), c2,
                                                      s_tok, s_rank, s_res, s_nx, s_pv);
    } else if (gi < t2) {
      const int64_t slot = gi < c0 ? gi : gi < t1 ? lcap + (gi - c0) : 2 * lcap + (gi - t1);
      mid_piece(T, W, g, __ldcg(&W.long_list[slot]), s_tok, s_rank, s_res, s_nx, s_pv);
    } else {
      small_chunk<PAIRS >= 1>(T, W, g, total, np, (gi - t2) * CH, R, mq[warp], qn, v);
    }
#ifdef TT_TRACE
    __syncwarp();
    if (lane == 0) {
      // the ticket's list entries (kinds 0, 1, 3) or chunk (kind 2)
      const int kind = gi < c0 ? 0 : gi < t1 ? 1 : gi < t2 ? 3 : 2;
      int first = 0, cnt = 1;
      const int32_t *list = W.long_list;
      if (kind == 0) first = gi;
      if (kind == 1) { list += lcap; first = PAIRS >= 2 ? 2 * (gi - c0) : gi - c0; cnt = min(PAIRS >= 2 ? 2 : 1, c1 - first); }
      if (kind == 3) { list += 2 * lcap; first = PAIRS >= 1 ? GROUP2 * (gi - t1) : gi - t1; cnt = min(PAIRS >= 1 ? GROUP2 : 1, c2 - first); }
      int max_len = 0;
      if (kind == 2) {
        cnt = min(CH, np - (gi - t2) * CH);
        max_len = SMALL_MAX;
      } else {
        for (int q = 0; q < cnt; ++q) {
          const int pc = __ldcg(&list[first + q]);
          max_len = max(max_len, (__ldcg(&W.piece_start[pc + 1]) & 0x7FFFFFFF) - __ldcg(&W.piece_start[pc]));
        }
      }
      const int at = atomicAdd(&tt_trace_n, 1);
      if (at < TRACE_CAP) tt_trace_rec[at] = TraceRec{tr0, trace_clock(), kind, cnt, max_len, tt_trace_rounds[warp]};
    }
#endif
  }
#ifdef TT_TRACE
  if (lane == 0) tt_trace_rounds[warp] = 0;
  __syncwarp();
  const unsigned long long tr1 = trace_clock();
#endif
  if (qn) run_misses(T, W, g, mq[warp], qn, v);   // the warp's last queued misses
#ifdef TT_TRACE
  __syncwarp();
  if (lane == 0 && qn) {
    const int at = atomicAdd(&tt_trace_n, 1);
    if (at < TRACE_CAP) tt_trace_rec[at] = TraceRec{tr1, trace_clock(), 4, qn, SMALL_MAX, tt_trace_rounds[warp]};
  }
#endif
}

#ifdef TT_TRACE
// Trace builds only: copy up to cap records (struct TraceRec, 32 bytes each)
// of the traced kernels since the last call into out, return how many there
// were, and start a new trace.
extern "C" int tt_trace_read(void *out, int cap) {
  int n = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(&n, tt_trace_n, sizeof(int)) != cudaSuccess) return -1;
  const int k = n < cap ? n : cap;
  if (k > 0 && cudaMemcpyFromSymbol(out, tt_trace_rec, (size_t)k * sizeof(TraceRec)) != cudaSuccess) return -1;
  const int zero = 0;
  if (cudaMemcpyToSymbol(tt_trace_n, &zero, sizeof(int)) != cudaSuccess) return -1;
  return n;
}
#endif

// ---------------------------------------------------------------- long
// Block per piece.  Thread t owns a contiguous segment of the current token
// array; a round is: block min of the ranks, a block max-scan that carries
// "where the current run of hits started" across segments (a run of equal
// pairs (a, a) is merged at even offsets: the leftmost non-overlapping
// selection), a block sum-scan of kept tokens, and a write of the new tokens
// (merge flag in bit 31) and of the old rank of every untouched pair into the
// other buffer; after a barrier the pairs next to a merge are looked up.
// A one-entry cache per thread absorbs the repeated lookups of long runs.
__device__ __forceinline__ int cached_rank(const Tables &T, int l, int r, int &cl, int &cr, int &cv) {
  if (l == cl && r == cr) return cv;
  cl = l; cr = r; cv = pair_rank(T, l, r);
  return cv;
}

// Pieces of up to LONG_SMEM_MAX bytes run the warp kernel's linked-list
// rounds with the whole block: the list lives in dynamic shared memory
// (thread t owns positions t, t + NT, ...), the round minimum is a block
// reduction, and each merge step costs three barriers and one lookup; safe
// pairs merge in any round, as in the warp rounds.
constexpr int LONG_SMEM_MAX = 8192;
constexpr size_t LONG_SMEM_BYTES = (size_t)LONG_SMEM_MAX * (4 + 4 + 4 + 2 + 2);
static_assert(LONG_SMEM_MAX / BPE_LONG_THREADS <= 32, "slot mask is 32 bits");

__device__ void bpe_block_list(const Tables &T, const Work &W, const uint8_t *b, int n, int32_t *out, int piece,
                               unsigned char *dsm, int *red) {
  constexpr int NT = BPE_LONG_THREADS;
  const int tid = threadIdx.x, lane = tid & 31;
  int32_t *tok = reinterpret_cast<int32_t *>(dsm);
  int32_t *rank = tok + LONG_SMEM_MAX;
  int32_t *res = rank + LONG_SMEM_MAX;
  int16_t *nx = reinterpret_cast<int16_t *>(res + LONG_SMEM_MAX);
  int16_t *pv = nx + LONG_SMEM_MAX;
  const int nslot = (n + NT - 1) / NT;
  for (int k = 0; k < nslot; ++k) {
    const int p = tid + NT * k;
    tok[p] = p < n ? __ldg(&T.byte_id[__ldg(b + p)]) : -1;
    rank[p] = INT_MAX;
    nx[p] = (int16_t)(p + 1);
    pv[p] = (int16_t)(p - 1);
  }
  __syncthreads();
  for (int k = 0; k < nslot; ++k) {            // first lookups: pairs of byte tokens, the direct tables
    const int p = tid + NT * k;
    if (p + 1 < n) {
      int rs;
      rank[p] = byte_pair_key(T, __ldg(b + p), __ldg(b + p + 1), byte_at(b, p - 1, n), byte_at(b, p + 2, n), rs);
      res[p] = rs;
    }
  }
  __syncthreads();
  for (int round = 0; round < n; ++round) {       // each round unlinks at least one symbol
    int lm = INT_MAX;
    for (int k = 0; k < nslot; ++k) lm = min(lm, rank[tid + NT * k]);
    lm = __reduce_min_sync(0xffffffffu, lm);
    if (lane == 0) red[tid >> 5] = lm;
    __syncthreads();
    const int r = __reduce_min_sync(0xffffffffu, lane < NT / 32 ? red[lane] : INT_MAX);
    if (r == INT_MAX) break;
    for (int step = 0; step < n; ++step) {
      uint32_t sel = 0;
      bool pending = false;
      for (int k = 0; k < nslot; ++k) {
        const int p = tid + NT * k;
        const int key = rank[p];
        if (key_safe(key)) {
          sel |= 1u << k;
        } else if (key == r) {
          const int q = pv[p];
          if (q < 0 || rank[q] != r) sel |= 1u << k;
          else pending = true;
        }
      }
      __syncthreads();
      for (uint32_t m = sel; m; m &= m - 1) {
        const int p = tid + NT * (__ffs(m) - 1);
        const int q = nx[p], nq = nx[q];
        tok[p] = res[p];
        tok[q] = -1;
        rank[q] = INT_MAX;
        rank[p] = INT_MAX;
        nx[p] = (int16_t)nq;
        if (nq < n) pv[nq] = (int16_t)p;
      }
      __syncthreads();
      for (uint32_t m = sel; m; m &= m - 1) relink_lookups(T, b, n, tid + NT * (__ffs(m) - 1), tok, rank, res, nx, pv);
      if (!__syncthreads_or(pending)) break;
    }
  }
  __syncthreads();   // every thread has read red[] before it is reused below
  // surviving tokens in position order: thread t compacts positions [t*seg, (t+1)*seg)
  const int seg = (n + NT - 1) / NT;
  const int lo = min(tid * seg, n), hi = min(lo + seg, n);
  int cnt = 0;
  for (int p = lo; p < hi; ++p) cnt += tok[p] >= 0;
  int tot;
  int w = block_exclusive_scan<NT>(cnt, [](int x, int y) { return x + y; }, 0, red, &tot);
  for (int p = lo; p < hi; ++p)
    if (tok[p] >= 0) out[w++] = tok[p];
  if (tid == 0) put_count(W, piece, tot);
  __syncthreads();
}

__global__ void __launch_bounds__(BPE_LONG_THREADS, 1) k_bpe_long(Tables T, Work W) {
  constexpr int NT = BPE_LONG_THREADS;
  constexpr int32_t MERGED = (int32_t)0x80000000;
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ int red[NT / 32];
  __shared__ int s_whole;
  const CallArgs A = *W.args;
  const int tid = threadIdx.x;
  if (A.n <= 0) return;
  int64_t base, total;
  if (!batch_extent(A, base, total) || call_timed_out(W)) return;
  const int nh = __ldcg(&W.counters[6]);
  const uint8_t *g = A.utf8 + base;
  auto plus = [](int a, int b) { return a + b; };
  auto mx = [](int a, int b) { return a > b ? a : b; };
  auto mn = [](int a, int b) { return a < b ? a : b; };
  int cl = -1, cr = -1, cv = -1;
  for (int li = blockIdx.x; li < nh; li += gridDim.x) {
    const int k = __ldcg(&W.huge_list[li]);
    const int32_t s = __ldcg(&W.piece_start[k]);
    const int32_t e = __ldcg(&W.piece_start[k + 1]) & 0x7FFFFFFF;
    const int len = e - s;
    const uint8_t *b = g + s;
    if (len <= T.max_tok_len) {
      if (tid == 0) s_whole = vocab_probe(T, b, len);
      __syncthreads();
      const int whole = s_whole;
      __syncthreads();
      if (whole >= 0) {
        if (tid == 0) { W.scratch[s] = whole; put_count(W, k, 1); }
        continue;
      }
    }
    if (len <= LONG_SMEM_MAX) {
      bpe_block_list(T, W, b, len, W.scratch + s, k, dsm, red);
      continue;
    }
    int32_t *cur = W.scratch + s, *nxt = W.tmp_b + s;
    int32_t *rcur = W.tmp_a + s, *rnxt = W.tmp_c + s;
    int n = len;
    for (int i = tid; i < n; i += NT) cur[i] = __ldg(&T.byte_id[__ldg(b + i)]);
    __syncthreads();
    for (int i = tid; i + 1 < n; i += NT) rcur[i] = cached_rank(T, cur[i], cur[i + 1], cl, cr, cv);
    __syncthreads();
    for (;;) {
      const int seg = (n + NT - 1) / NT;
      const int lo = min(tid * seg, n), hi = min(lo + seg, n);
      int lm = INT_MAX;
      for (int i = lo; i < hi && i + 1 < n; ++i)
        if (rcur[i] >= 0 && rcur[i] < lm) lm = rcur[i];
      int r;
      block_exclusive_scan<NT>(lm, mn, INT_MAX, red, &r);
      if (r == INT_MAX) break;
      const int res = __ldg(&T.merge_result[r]);
      // position after the last non-hit of my segment (-1 if all hits)
      int after_nh = -1;
      for (int i = lo; i < hi; ++i)
        if (!(i + 1 < n && rcur[i] == r)) after_nh = i + 1;
      int run_in = block_exclusive_scan<NT>(after_nh, mx, -1, red, (int *)nullptr);
      if (run_in < 0) run_in = 0;
      // was the element before my segment selected?
      bool prev_sel = false;
      if (lo > 0 && lo < n) {
        const bool h = rcur[lo - 1] == r;          // lo - 1 + 1 < n holds
        prev_sel = h && ((lo - 1 - run_in) % 2 == 0);
      }
      // count kept tokens
      int keep = 0;
      {
        int run = run_in;
        bool ps = prev_sel;
        for (int i = lo; i < hi; ++i) {
          const bool h = i + 1 < n && rcur[i] == r;
          if (!h) run = i + 1;
          const bool sel = h && ((i - run) % 2 == 0);
          if (!ps) ++keep;
          ps = sel;
        }
      }
      int n_new;
      const int wbase = block_exclusive_scan<NT>(keep, plus, 0, red, &n_new);
      // write new tokens (merge flag in bit 31) and candidate ranks
      {
        int run = run_in, w = wbase;
        bool ps = prev_sel;
        for (int i = lo; i < hi; ++i) {
          const bool h = i + 1 < n && rcur[i] == r;
          if (!h) run = i + 1;
          const bool sel = h && ((i - run) % 2 == 0);
          if (!ps) {
            nxt[w] = sel ? (res | MERGED) : cur[i];
            // the old pair (i, i+1) survives unless i or i+1 merges
            rnxt[w] = (i + 1 < n) ? rcur[i] : -1;
            ++w;
          }
          ps = sel;
        }
      }
      __syncthreads();
      // ranks of the new pairs next to a merge
      {
        const int nlo = wbase, nhi = wbase + keep;
        for (int j = nlo; j < nhi; ++j) {
          if (j + 1 >= n_new) { rnxt[j] = -1; continue; }
          const int a = nxt[j], bb = nxt[j + 1];
          if ((a | bb) & MERGED) rnxt[j] = cached_rank(T, a & 0x7FFFFFFF, bb & 0x7FFFFFFF, cl, cr, cv);
        }
      }
      __syncthreads();
      for (int j = wbase; j < wbase + keep; ++j) nxt[j] &= 0x7FFFFFFF;
      __syncthreads();
      int32_t *t1 = cur; cur = nxt; nxt = t1;
      int32_t *t2 = rcur; rcur = rnxt; rnxt = t2;
      n = n_new;
    }
    if (cur != W.scratch + s) {
      for (int i = tid; i < n; i += NT) W.scratch[s + i] = cur[i];
    }
    if (tid == 0) put_count(W, k, n);
    __syncthreads();
  }
}

// ---------------------------------------------------------------- ids
// The first piece of request r (recorded by the pre-tokenizer), or np for a
// request with no piece (empty at the batch end) and for r = n.  It never
// decreases with r; `bad` reports an entry outside the piece table.
__device__ __forceinline__ int request_piece(const CallArgs &A, const Work &W, int64_t base, int64_t total, int np,
                                             int64_t r, bool *bad) {
  if (r >= A.n || __ldg(&A.offs[r]) - base >= total) return np;
  const int k = __ldcg(&W.req_piece[r]);
  if (k < 0 || k >= np) { *bad = true; return np; }
  return k;
}
// The first request r in [0, n] whose first piece is >= p (p <= np), by one
// warp: 32 probes per step, so a handful of steps for any batch.
__device__ int64_t first_request_from(const CallArgs &A, const Work &W, int64_t base, int64_t total, int np, int p) {
  const int lane = threadIdx.x & 31;
  int64_t lo = 0, hi = A.n;   // the answer lies in [lo, hi]; request_piece(n) = np >= p
  bool bad = false;
  while (lo < hi) {
    const int64_t step = (hi - lo + 31) / 32;
    const int64_t r = lo + (int64_t)lane * step;
    const bool ge = r < hi && request_piece(A, W, base, total, np, r, &bad) >= p;
    const unsigned m = __ballot_sync(0xffffffffu, ge);
    if (m) {
      const int f = __ffs(m) - 1;
      hi = lo + (int64_t)f * step;
      if (f) lo += (int64_t)(f - 1) * step + 1;
    } else {
      lo += ((hi - 1 - lo) / step) * step + 1;   // past the last probe below hi
    }
  }
  return lo;
}

// Exclusive scan of the ID chunks' totals (summed by the BPE kernels as they
// write each piece's count) into each chunk's first output, and the batch's
// ID count.  One CTA: each thread sums a contiguous run of chunks (loads in
// flight together), one block scan, then the run's prefixes.
__global__ void __launch_bounds__(1024) k_idscan(Work W) {
  __shared__ int red[32];
  const CallArgs A = *W.args;
  const int tid = threadIdx.x;
  int np = 0;
  if (A.n > 0) {
    int64_t base, total;
    if (batch_extent(A, base, total) && !call_timed_out(W)) np = __ldcg(&W.counters[3]);
  }
  const int nchunks = (np + IDS_CHUNK - 1) / IDS_CHUNK;
  const int per = (nchunks + 1023) / 1024;
  const int lo = min(tid * per, nchunks), hi = min(lo + per, nchunks);
  int sum = 0;
#pragma unroll 8
  for (int c = lo; c < hi; ++c) sum += __ldcg(&W.ids_agg[c]);
  int tot;
  int ex = block_exclusive_scan<1024>(sum, [](int a, int b) { return a + b; }, 0, red, &tot);
  for (int c = lo; c < hi; ++c) {
    const int v = __ldcg(&W.ids_agg[c]);
    W.ids_inc[c] = ex;
    ex += v;
  }
  if (tid == 0) W.counters[4] = tot;
}

__global__ void __launch_bounds__(IDS_THREADS) k_ids(Tables T, Work W) {
  constexpr int PER = IDS_CHUNK / IDS_THREADS;
  __shared__ int s_off[IDS_CHUNK + 1];   // chunk-local output offset of each piece
  __shared__ int s_st[IDS_CHUNK];        // its start byte (its IDs sit at scratch[start ...])
  __shared__ int red[IDS_THREADS / 32];
  __shared__ int2 s_red2[IDS_THREADS / 32];
  __shared__ int64_t s_rlo, s_rhi;       // requests whose first piece is in the chunk
  const CallArgs A = *W.args;
  const int tid = threadIdx.x;
  if (A.n <= 0) return;
  int64_t base, total;
  const bool sound = batch_extent(A, base, total) && !call_timed_out(W);
  const int np = sound ? __ldcg(&W.counters[3]) : 0;
  const int nchunks = (np + IDS_CHUNK - 1) / IDS_CHUNK;
  if (nchunks == 0) {   // no pieces (an empty, unsound or timed-out batch): every request has no IDs
    for (int64_t r = (int64_t)blockIdx.x * IDS_THREADS + tid; r <= A.n; r += (int64_t)gridDim.x * IDS_THREADS)
      A.out_id_offsets[r] = 0;
    return;
  }
  // chunks are independent: each one's first output comes from the chunk scan
  for (int t = blockIdx.x; t < nchunks; t += gridDim.x) {
    const int cb = __ldcg(&W.ids_inc[t]);
    const int k0 = t * IDS_CHUNK;
    const int nloc = min(IDS_CHUNK, np - k0);
    int cnt[PER], st[PER];
    int sum = 0;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int q = tid * PER + m;
      cnt[m] = 0;
      st[m] = 0;
      if (q < nloc) {
        cnt[m] = __ldcg(&W.n_ids[k0 + q]);
        st[m] = __ldcg(&W.piece_start[k0 + q]) & 0x7FFFFFFF;
        if (cnt[m] < 0 || (int64_t)st[m] + cnt[m] > total) {   // never for a sound piece table
          set_status(W.status, ST_INVALID_ARG);
          cnt[m] = 0;
        }
      }
      sum += cnt[m];
    }
    int chunk_total;
    const int ex = block_exclusive_scan<IDS_THREADS>(sum, [](int a, int b) { return a + b; }, 0, red, &chunk_total);
    // (warps 0 and 1 find the chunk's requests; the counts the chunk scan
    // summed must be the ones read here)
    if (tid < 32) {
      const int64_t r = first_request_from(A, W, base, total, np, k0);
      if (tid == 0) s_rlo = r;
    } else if (tid < 64) {
      const int64_t r = t == nchunks - 1 ? A.n + 1 : first_request_from(A, W, base, total, np, k0 + nloc);
      if (tid == 32) s_rhi = r;
    } else if (tid == 64 && __ldcg(&W.ids_agg[t]) != chunk_total) {
      set_status(W.status, ST_INVALID_ARG);
    }
    __syncthreads();
    int off = ex;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int q = tid * PER + m;
      s_off[q] = off;
      s_st[q] = st[m];
      off += cnt[m];
    }
    if (tid == 0) s_off[IDS_CHUNK] = chunk_total;
    __syncthreads();
    // per-request ID offsets: a request starts at its first piece's offset
    // (the last chunk also writes those past its last piece: the batch's token
    // count for empty requests at the end and for the end offset n)
    for (int64_t r = s_rlo + tid; r < s_rhi; r += IDS_THREADS) {
      bool bad = false;
      const int k = request_piece(A, W, base, total, np, r, &bad);
      if (bad) set_status(W.status, ST_INVALID_ARG);
      A.out_id_offsets[r] = cb + ((k >= k0 && k < k0 + nloc) ? s_off[k - k0] : chunk_total);
    }
    // output-parallel copy: output o of the chunk belongs to the last piece
    // whose offset is <= o (pieces with no IDs share their successor's offset)
    auto piece_of = [&](int o) {
      int lo = 0, hi = nloc - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= o) lo = mid;
        else hi = mid - 1;
      }
      return lo;
    };
    if ((int64_t)cb + chunk_total > total) {
      if (tid == 0) set_status(W.status, ST_INVALID_ARG);
    } else if (!A.out_spans) {
      // four outputs a thread at a time: their searches and loads overlap
      constexpr int U = 4;
      for (int ob = 0; ob < chunk_total; ob += U * IDS_THREADS) {
        int src[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int o = ob + u * IDS_THREADS + tid;
          src[u] = -1;
          if (o < chunk_total) {
            const int q = piece_of(o);
            src[u] = s_st[q] + (o - s_off[q]);
          }
        }
        int id[U];
#pragma unroll
        for (int u = 0; u < U; ++u) id[u] = src[u] >= 0 ? __ldcg(&W.scratch[src[u]]) : 0;
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (src[u] >= 0) A.out_ids[cb + ob + u * IDS_THREADS + tid] = id[u];
      }
    } else {
      // with byte spans: the IDs of a piece cover its bytes in order, so an
      // ID starts where the lengths of the piece's earlier IDs end -- a scan
      // of token lengths segmented by piece, IDS_THREADS outputs at a time,
      // the open piece's byte count carried from one step to the next
      auto seg = [](int2 a, int2 b) { return make_int2(a.x | b.x, b.x ? b.y : a.y + b.y); };
      int carry = 0;
      for (int ob = 0; ob < chunk_total; ob += IDS_THREADS) {
        const int o = ob + tid;
        int q = 0, len = 0;
        bool head = false;
        if (o < chunk_total) {
          q = piece_of(o);
          const int id = __ldcg(&W.scratch[s_st[q] + (o - s_off[q])]);
          A.out_ids[cb + o] = id;
          len = __ldg(&T.voff[id + 1]) - __ldg(&T.voff[id]);
          head = o == s_off[q];
        }
        int2 step;
        const int2 ex = block_exclusive_scan<IDS_THREADS>(make_int2(head, len), seg, make_int2(0, 0), s_red2,
                                                          &step);
        if (o < chunk_total) {
          const int before = head ? 0 : ex.y + (ex.x ? 0 : carry);   // bytes of my piece before me
          const int start = s_st[q] + before;
          A.out_spans[2 * ((int64_t)cb + o)] = start;
          A.out_spans[2 * ((int64_t)cb + o) + 1] = start + len;
        }
        carry = step.x ? step.y : carry + step.y;
      }
    }
    __syncthreads();
  }
}

// first piece whose start (flag bit cleared) is >= pos, in [0, np]
__device__ __forceinline__ int lower_bound_piece(const int32_t *ps, int np, int64_t pos) {
  int lo = 0, hi = np;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)(__ldcg(&ps[mid]) & 0x7FFFFFFF) < pos) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------- test hook
__global__ void __launch_bounds__(1024) k_hook_pre(Work W) {
  __shared__ int red[32];
  __shared__ int carry;
  const CallArgs A = *W.args;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int64_t c = 0; c <= A.n; c += 1024) {
    const int64_t r = c + threadIdx.x;
    const int v = r < A.n ? W.bad[r] : 0;
    int tot;
    const int ex = block_exclusive_scan<1024>(v, [](int a, int b) { return a + b; }, 0, red, &tot);
    if (r <= A.n) W.bad_pre[r] = carry + ex;
    __syncthreads();
    if (threadIdx.x == 0) carry += tot;
    __syncthreads();
  }
}

__global__ void k_hook_pieces(Work W) {
  const CallArgs A = *W.args;
  if (A.n <= 0) return;
  int64_t base, total;
  if (!batch_extent(A, base, total) || call_timed_out(W)) return;
  const int np = __ldcg(&W.counters[3]);
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < np; k += gridDim.x * blockDim.x) {
    const int32_t s = __ldcg(&W.piece_start[k]);
    if (s < 0) continue;
    int64_t lo = 0, hi = A.n + 1;     // last r with offs[r] <= base + s
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (__ldg(&A.offs[mid]) < base + s + 1) lo = mid + 1; else hi = mid;
    }
    const int64_t r = lo - 1;
    A.hook_starts[k - W.bad_pre[r]] = base + s;
  }
}

__global__ void k_hook_offsets(Work W) {
  const CallArgs A = *W.args;
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (A.n <= 0 || r > A.n) return;
  int64_t base, total;
  if (!batch_extent(A, base, total) || call_timed_out(W)) { A.hook_offsets[r] = 0; return; }
  const int np = __ldcg(&W.counters[3]);
  const int k = lower_bound_piece(W.piece_start, np, __ldg(&A.offs[r]) - base);
  A.hook_offsets[r] = k - W.bad_pre[r];
}

void launch_bpe_warp(const Tables &T, const Work &W, int grid, cudaStream_t s) {
  if (W.cap_bytes > PAIR_MIN_CAP_BYTES) k_bpe_warp<2><<<grid, BPE_WARP_THREADS, 0, s>>>(T, W);
  else k_bpe_warp<0><<<grid, BPE_WARP_THREADS, 0, s>>>(T, W);
}
void launch_bpe_long(const Tables &T, const Work &W, int grid, cudaStream_t s) {
  k_bpe_long<<<grid, BPE_LONG_THREADS, LONG_SMEM_BYTES, s>>>(T, W);
}
void launch_idscan(const Work &W, cudaStream_t s) { k_idscan<<<1, 1024, 0, s>>>(W); }
void launch_ids(const Tables &T, const Work &W, int grid, cudaStream_t s) { k_ids<<<grid, IDS_THREADS, 0, s>>>(T, W); }
void launch_hook_pre(const Work &W, cudaStream_t s) { k_hook_pre<<<1, 1024, 0, s>>>(W); }
void launch_hook_pieces(const Work &W, int grid, cudaStream_t s) { k_hook_pieces<<<grid, 256, 0, s>>>(W); }
void launch_hook_offsets(const Work &W, int grid, cudaStream_t s) { k_hook_offsets<<<grid, 256, 0, s>>>(W); }

cudaError_t bpe_configure() {
  return cudaFuncSetAttribute(k_bpe_long, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LONG_SMEM_BYTES);
}

}  // namespace tt
