// tt_pretok.cu - parallel pre-tokenizer: UTF-8 decode, character classes,
// run aggregates by prefix scans, the piece-start predicate and piece
// compaction (TokTier: Exact Stateful CPU+GPU Tokenization for Agentic LLM
// Serving, §4.1 run decomposition, §4.3 multi-document batching: runs are cut
// at document boundaries and counts stay in device memory).
//
// Two kernels per batch:
//   k_prepass   one CTA per 4016-byte tile, independent: validates UTF-8
//               (per request), and summarises each tile for the two scans
//               whose carries are found ahead of their use, from the bytes
//               alone: the reverse "first event after" queries (one warp
//               from the tile start) and o200k mark resolution (the last
//               stretch start and trigger, on a tiling shifted 32 bytes left:
//               one warp back from the tile end); it resets the look-back
//               flags and ID chunk totals of its tile, and copies page-locked
//               host input into the device batch when asked to.
//   k_pretok    one CTA per tile, tiles claimed in order: the two carries
//               from the other tiles' summaries (one warp each, 32 summaries
//               a step), effective classes (deepseek-style: segment starts),
//               the forward scan (number-run count, blank-run start, o200k
//               contraction chain and case state) with decoupled look-back
//               on a tiling shifted 16 bytes left, its aggregate published
//               before the reverse queries, the predicate, and compaction of
//               piece starts with a second decoupled look-back.
#include <limits.h>

#include "tt_common.cuh"
#include "tt_kernels.h"

namespace tt {

// A window char's attributes in one word: the window index of its lead byte
// (12 bits), its code point if ASCII else 0x80 (8), raw kind (5), effective
// kind (4), and whether it starts a request or a segment (1).
__device__ __forceinline__ uint32_t ci_pack(int lead, uint32_t cp8, uint32_t raw, bool rs) {
  return (uint32_t)lead | (cp8 << 12) | (raw << 20) | ((uint32_t)rs << 29);
}
__device__ __forceinline__ int ci_lead(uint32_t c) { return (int)(c & 0xFFFu); }
__device__ __forceinline__ uint32_t ci_cp8(uint32_t c) { return (c >> 12) & 0xFFu; }
__device__ __forceinline__ uint8_t ci_raw(uint32_t c) { return (uint8_t)((c >> 20) & 0x1Fu); }
__device__ __forceinline__ uint8_t ci_eff(uint32_t c) { return (uint8_t)((c >> 25) & 0xFu); }
__device__ __forceinline__ bool ci_rs(uint32_t c) { return (c >> 29) & 1u; }
static_assert(WIN <= 4096, "lead index is 12 bits");

template <int NT>   // threads per window
struct WinSmem {
  uint8_t bytes[WIN + 8];
  uint8_t rsb[WIN + 8];      // byte starts a request
  uint32_t ci[WIN];          // per char: ci_pack
  int cbase[NT + 1];         // chars of thread t: [cbase[t], cbase[t+1])
  uint8_t ascii[128];
  int r0, r1;
  int nch;
  __device__ __forceinline__ int lead(int j) const { return ci_lead(ci[j]); }
  __device__ __forceinline__ uint32_t cp8(int j) const { return ci_cp8(ci[j]); }
  __device__ __forceinline__ uint8_t raw(int j) const { return ci_raw(ci[j]); }
  __device__ __forceinline__ uint8_t eff(int j) const { return ci_eff(ci[j]); }
  __device__ __forceinline__ bool rs(int j) const { return ci_rs(ci[j]); }
  // (only the char's own thread writes these; neighbours may read the word
  // meanwhile, and the bits they read do not change)
  __device__ __forceinline__ void set_eff(int j, uint8_t e) { ci[j] = (ci[j] & ~(0xFu << 25)) | ((uint32_t)e << 25); }
  __device__ __forceinline__ void set_rs(int j) { ci[j] |= 1u << 29; }
};

// The prepass's view of a window: bytes, request starts and the ASCII classes.
struct ByteWin {
  alignas(16) uint8_t bytes[WIN + 8];
  uint8_t rsb[WIN + 8];
  uint8_t ascii[128];
  int r0, r1;
};

// The first index i in [0, n) with a[i] >= v (n if none), a ascending, by
// one whole warp: each step splits the interval into 32 parts and one load a
// lane finds the part holding the answer (two steps for up to 1,024
// requests, instead of one dependent load per halving).
__device__ __forceinline__ int64_t warp_lower_bound64(const int64_t *a, int64_t n, int64_t v) {
  const int lane = threadIdx.x & 31;
  int64_t lo = 0, hi = n;                   // the answer lies in [lo, hi]
  while (lo < hi) {
    const int64_t step = (hi - lo + 31) / 32;
    const int64_t idx = lo + (int64_t)(lane + 1) * step - 1;   // last index of part lane
    const bool less = idx < hi && __ldg(&a[idx]) < v;
    const int k = __popc(__ballot_sync(0xffffffffu, less));     // parts wholly below v (a prefix)
    lo += (int64_t)k * step;                // every index below is < v
    hi = min(hi, lo + step - 1);            // part k's last index (if tested) is >= v
  }
  return lo;
}

__device__ __forceinline__ int64_t lower_bound64(const int64_t *a, int64_t n, int64_t v) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    int64_t mid = (lo + hi) >> 1;
    if (__ldg(&a[mid]) < v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

template <class WS>
__device__ __forceinline__ uint8_t kind_of(const Tables &T, const WS &S, uint32_t cp) {
  if (cp < 128) return S.ascii[cp];
  return __ldg(&T.cls2[(uint32_t)__ldg(&T.cls1[cp >> 8]) * 256u + (cp & 255u)]);
}

// Code point of the char whose lead byte is window byte i (a char start):
// U+FFFD for a malformed or truncated sequence, or one that runs into the
// next request.
template <class WS>
__device__ __forceinline__ uint32_t decode_at(const WS &S, int64_t ws, int64_t total, int i) {
  const uint8_t b0 = S.bytes[i];
  int len;
  uint32_t cp;
  if (b0 < 0x80) return b0;
  if (b0 >= 0xC0 && b0 < 0xE0) { len = 2; cp = b0 & 0x1F; }
  else if (b0 >= 0xE0 && b0 < 0xF0) { len = 3; cp = b0 & 0x0F; }
  else if (b0 >= 0xF0 && b0 < 0xF8) { len = 4; cp = b0 & 0x07; }
  else return 0xFFFD;
  for (int q = 1; q < len; ++q) {
    if (i + q >= WIN || ws + i + q >= total || S.rsb[i + q] || (S.bytes[i + q] & 0xC0) != 0x80) return 0xFFFD;
    cp = (cp << 6) | (S.bytes[i + q] & 0x3F);
  }
  return cp < 0x110000u ? cp : 0xFFFD;
}

// Load the bytes of the window [ws, ws + WIN) and mark request starts.  All
// threads participate.  src: where to read the batch (NULL: A.utf8).
// WARP_SEARCH: warps 0 and 1 find the window's request range (the pre-pass,
// whose tiles wait on it); else thread 0 bisects (the pre-tokenizer, whose
// batch variant keeps its register count lower that way).
template <int NT, class WS, bool WARP_SEARCH = false>
__device__ void load_bytes(const Tables &T, const CallArgs &A, int64_t base, int64_t total, int64_t ws, WS &S,
                           const uint8_t *src = nullptr) {
  constexpr int PT_BYTES = WIN / NT;
  const int tid = threadIdx.x;
  const uint8_t *g = (src ? src : A.utf8) + base;
  const int64_t x0 = ws + PT_BYTES * tid;
  uint8_t *dst = &S.bytes[PT_BYTES * tid];
  if (x0 >= 0 && x0 + PT_BYTES <= total && ((reinterpret_cast<uintptr_t>(g + x0) & (PT_BYTES - 1)) == 0)) {
    if constexpr (PT_BYTES == 16) *reinterpret_cast<uint4 *>(dst) = __ldg(reinterpret_cast<const uint4 *>(g + x0));
    else *reinterpret_cast<uint2 *>(dst) = __ldg(reinterpret_cast<const uint2 *>(g + x0));
  } else {
#pragma unroll
    for (int k = 0; k < PT_BYTES; ++k) {
      const int64_t x = x0 + k;
      dst[k] = (x >= 0 && x < total) ? __ldg(g + x) : 0;
    }
  }
#pragma unroll
  for (int k = 0; k < PT_BYTES; ++k) S.rsb[PT_BYTES * tid + k] = 0;
  if (tid < 8) { S.bytes[WIN + tid] = 0; S.rsb[WIN + tid] = 0; }
  if (tid < 128) S.ascii[tid] = __ldg(&T.cls2[(uint32_t)__ldg(&T.cls1[0]) * 256u + tid]);
  const int64_t wlo = ws < 0 ? 0 : ws;
  const int64_t whi = ws + WIN < total ? ws + WIN : total;
  if constexpr (WARP_SEARCH) {
    if (tid < 64) {
      const int r = (int)warp_lower_bound64(A.offs, A.n, base + (tid < 32 ? wlo : whi));
      if (tid == 0) S.r0 = r;
      if (tid == 32) S.r1 = r;
    }
  } else if (tid == 0) {
    S.r0 = (int)lower_bound64(A.offs, A.n, base + wlo);
    S.r1 = (int)lower_bound64(A.offs, A.n, base + whi);
  }
  __syncthreads();
  for (int r = S.r0 + tid; r < S.r1; r += NT) {
    const int64_t x = __ldg(&A.offs[r]) - base - ws;
    if (x >= 0 && x < WIN && __ldg(&A.offs[r]) - base < total) S.rsb[x] = 1;
  }
  __syncthreads();
}

// Load the window [ws, ws + WIN) of the batch, mark request starts, find
// char starts, decode and classify.  All threads participate.
// lit: the batch's added-token marks (LIT_SEG / LIT_INNER per byte), or
// NULL when the handle has no literals.
template <int NT>
__device__ void load_window(const Tables &T, const CallArgs &A, int64_t base, int64_t total, int64_t ws,
                            WinSmem<NT> &S, int *scan_tmp, const uint8_t *lit) {
  constexpr int PT_BYTES = WIN / NT;
  const int tid = threadIdx.x;
  load_bytes<NT>(T, A, base, total, ws, S);
  // char starts among my PT_BYTES bytes
  uint32_t smask = 0;
#pragma unroll
  for (int k = 0; k < PT_BYTES; ++k) {
    const int i = PT_BYTES * tid + k;
    const int64_t x = ws + i;
    if (x < 0 || x >= total) continue;
    const uint8_t b = S.bytes[i];
    if ((b & 0xC0) != 0x80 || S.rsb[i]) smask |= 1u << k;
  }
  const int cnt = __popc(smask);
  int tot;
  const int cb = block_exclusive_scan<NT>(cnt, [](int a, int b) { return a + b; }, 0, scan_tmp, &tot);
  S.cbase[tid] = cb;
  if (tid == NT - 1) { S.cbase[NT] = tot; S.nch = tot; }
  int j = cb;
  for (uint32_t m = smask; m; m &= m - 1) {
    const int k = __ffs(m) - 1;
    const int i = PT_BYTES * tid + k;
    const uint32_t cp = decode_at(S, ws, total, i);
    const uint8_t mark = lit ? __ldg(lit + ws + i) : 0;
    S.ci[j] = ci_pack(i, cp < 128 ? cp : 0x80u, mark == LIT_INNER ? (uint32_t)K_LIT : kind_of(T, S, cp),
                      S.rsb[i] || mark == LIT_SEG);
    ++j;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- k_prepass
template <int NT>
__global__ void __launch_bounds__(NT) k_prepass(Tables T, Work W) {
  constexpr int PT_BYTES = WIN / NT;
  __shared__ ByteWin S;
  const CallArgs A = *W.args;
  const int tid = threadIdx.x;
  if (A.n <= 0) return;
  int64_t base, total;
  if (!batch_extent(A, base, total)) {
    if (blockIdx.x == 0 && tid == 0) set_status(W.status, total > A.bound ? ST_CAPACITY : ST_INVALID_ARG);
    return;
  }
  // offsets must be non-decreasing
  for (int64_t r = (int64_t)blockIdx.x * NT + tid; r < A.n; r += (int64_t)gridDim.x * NT)
    if (__ldg(&A.offs[r]) > __ldg(&A.offs[r + 1])) set_status(W.status, ST_INVALID_ARG);
  const int ntiles = (int)((total + TILE - 1) / TILE);
  const int t = blockIdx.x;
  if (t >= ntiles) return;
  const int64_t ts = (int64_t)t * TILE, te = ts + TILE < total ? ts + TILE : total;
  const int64_t ws = ts - HALO_L;
  // reset what the later kernels accumulate into: this tile's look-back
  // flags, and the ID totals of the 512-piece chunks whose index times 512
  // falls in the tile (over all tiles: every chunk the batch's pieces can fill)
  if (tid == 0) { W.s2_flag[t] = 0; W.cnt_flag[t] = 0; }
  for (int64_t c = (ts + IDS_CHUNK - 1) / IDS_CHUNK + tid; c < (te + IDS_CHUNK - 1) / IDS_CHUNK; c += NT)
    W.ids_agg[c] = 0;
  // bytes and request starts suffice: the few chars the summaries look at
  // are decoded where they are met
  load_bytes<NT, ByteWin, true>(T, A, base, total, ws, S, A.utf8_src);
  // this thread's bytes as words, and which of them lie in the tile
  uint32_t wd[PT_BYTES / 4];
#pragma unroll
  for (int q = 0; q < PT_BYTES / 4; ++q) wd[q] = reinterpret_cast<const uint32_t *>(&S.bytes[PT_BYTES * tid])[q];
  const int64_t x0 = ws + PT_BYTES * tid;
  const bool whole = x0 >= ts && x0 + PT_BYTES <= te;
  uint32_t in_tile = whole ? (1u << PT_BYTES) - 1 : 0;
  if (!whole)
    for (int k = 0; k < PT_BYTES; ++k) in_tile |= (uint32_t)(x0 + k >= ts && x0 + k < te) << k;
  if (A.utf8_src) {                           // the later kernels read the device copy of the tile
    uint8_t *dst = const_cast<uint8_t *>(A.utf8) + base + x0;
    if (whole && (reinterpret_cast<uintptr_t>(dst) & 3) == 0) {
#pragma unroll
      for (int q = 0; q < PT_BYTES / 4; ++q) reinterpret_cast<uint32_t *>(dst)[q] = wd[q];
    } else {
      for (int k = 0; k < PT_BYTES; ++k)
        if ((in_tile >> k) & 1) dst[k] = S.bytes[PT_BYTES * tid + k];
    }
  }

  // --- UTF-8 validation of the tile's bytes (RFC 3629, per request).  Each
  // thread checks, in one pass over its bytes, the sequences that start among
  // them: continuation bytes at its start that a lead before them claims are
  // passed over (that lead's thread checks them), and a sequence open at its
  // last byte is completed by reading on (at most three bytes).  A request
  // is rejected for a lead whose sequence is malformed, cut by a request
  // start or by the batch end, and for a continuation byte no lead claims or
  // a byte no sequence starts with -- as a byte-by-byte check would find.
  // Threads with only ASCII bytes in the tile have nothing to check.
  uint32_t hi = 0;
#pragma unroll
  for (int q = 0; q < PT_BYTES / 4; ++q) hi |= top_bits4(wd[q]) << (4 * q);
  if (hi & in_tile) {
    auto reject = [&](int i) {               // the request holding window byte i
      const int64_t r = lower_bound64(A.offs, A.n + 1, base + ws + i + 1) - 1;
      if (r >= 0 && r < A.n) {
        W.bad[r] = 1;
        atomicMin(&W.status->bad_request, (unsigned long long)r);
        set_status(W.status, ST_INVALID_UTF8);
        atomicExch(&W.counters[5], 1);
      }
    };
    const int f = PT_BYTES * tid + (__ffs(in_tile) - 1);      // my first byte in the tile
    const int e = PT_BYTES * tid + (32 - __clz(in_tile));     // past my last one
    int p = f;
    {
      // the nearest non-continuation byte before f (at most 3 back, not
      // across a request start or the batch start) and the bytes from f on
      // that it claims, if it is a lead
      int reach = 0;
      for (int d = 1; d <= 3; ++d) {
        const int q = f - d;
        if (ws + q < 0) break;
        const uint8_t bq = S.bytes[q];
        if ((bq & 0xC0) == 0x80) {
          if (S.rsb[q]) break;
          continue;
        }
        reach = ((bq >= 0xC2 && bq <= 0xDF) ? 2 : (bq >= 0xE0 && bq <= 0xEF) ? 3 : (bq >= 0xF0 && bq <= 0xF4) ? 4 : 1) - d;
        break;
      }
      for (; reach > 0 && p < e && (S.bytes[p] & 0xC0) == 0x80 && !S.rsb[p]; --reach) ++p;
    }
    int need = 0, lead = -1;                 // continuation bytes the open sequence still needs, its lead
    uint32_t lo = 0x80, top = 0xBF;          // the range of its next byte
    for (; p < e || need > 0; ++p) {
      const uint32_t b = S.bytes[p];
      if (need > 0) {
        if (!S.rsb[p] && ws + p < total && b >= lo && b <= top) {
          --need;
          lo = 0x80;
          top = 0xBF;
          continue;
        }
        reject(lead);                        // malformed, or cut by a request start or the batch end
        need = 0;
        if (p >= e) break;                   // (past my bytes: another thread checks this one)
      }
      if (b < 0x80) continue;
      lead = p;
      if (b >= 0xC2 && b <= 0xDF) {
        need = 1;
        lo = 0x80;
        top = 0xBF;
      } else if (b >= 0xE0 && b <= 0xEF) {
        need = 2;
        lo = b == 0xE0 ? 0xA0 : 0x80;        // no overlong three-byte form
        top = b == 0xED ? 0x9F : 0xBF;       // no surrogate
      } else if (b >= 0xF0 && b <= 0xF4) {
        need = 3;
        lo = b == 0xF0 ? 0x90 : 0x80;        // no overlong four-byte form
        top = b == 0xF4 ? 0x8F : 0xBF;       // nothing past U+10FFFF
      } else {
        reject(p);                           // a continuation no lead claims, or C0, C1, F5..FF
      }
    }
  }

  const uint8_t *lit = T.n_lit ? W.lit_flag : nullptr;
  // the char starting at window byte i: request-or-segment start, raw kind, code point
  auto char_at = [&](int i, bool &rs, uint8_t &raw, uint32_t &cp) {
    cp = decode_at(S, ws, total, i);
    const uint8_t mark = lit ? __ldg(lit + ws + i) : 0;
    rs = S.rsb[i] != 0 || mark == LIT_SEG;
    raw = mark == LIT_INNER ? (uint8_t)K_LIT : kind_of(T, S, cp);
  };
  auto is_start = [&](int64_t x) { return x >= 0 && x < total && ((S.bytes[x - ws] & 0xC0) != 0x80 || S.rsb[x - ws]); };
  const int lane = tid & 31;
  if (tid < 32) {
    // --- reverse-query summary: the first rq_ws (and, o200k, rq_up) event
    // among the tile's chars, 32 bytes a step (usually one step)
    const bool want_up = T.family == FAM_O200K;
    int evw = 0xFF, evu = want_up ? 0xFF : 0x00;
    for (int64_t x0 = ts; x0 < te && (evw == 0xFF || evu == 0xFF); x0 += 32) {
      const int64_t x = x0 + lane;
      int ew = 0xFF, eu = 0xFF;
      if (x < te && is_start(x)) {
        bool rs;
        uint8_t raw;
        uint32_t cp;
        char_at((int)(x - ws), rs, raw, cp);
        ew = rq_ws_event(T.family, rs, raw, cp < 128 ? cp : 0x80u);
        eu = rq_up_event(rs, raw);
      }
      const unsigned mw = __ballot_sync(0xffffffffu, ew != 0xFF);
      const unsigned mu = __ballot_sync(0xffffffffu, eu != 0xFF);
      if (evw == 0xFF && mw) evw = __shfl_sync(0xffffffffu, ew, __ffs(mw) - 1);
      if (evu == 0xFF && mu) evu = __shfl_sync(0xffffffffu, eu, __ffs(mu) - 1);
    }
    if (lane == 0) { W.rq_sum[2 * t] = (uint8_t)evw; W.rq_sum[2 * t + 1] = want_up ? (uint8_t)evu : (uint8_t)0xFF; }
  } else if (tid < 64 && T.family == FAM_O200K) {
    // --- mark-resolution summary over the chars in [ts - 32, te - 32): the
    // last stretch start x and the last trigger y, scanning back from the end
    // 32 bytes a step until a stretch start is met.  A trigger before x is
    // reported as none: every use compares the latest trigger with the latest
    // stretch start, and x is at least as late as any earlier one.
    const int64_t lo = ts - S1_SHIFT > 0 ? ts - S1_SHIFT : 0, hi = te - S1_SHIFT;
    int xs = -1, ys = -1;
    for (int64_t x1 = hi; x1 > lo && xs < 0; x1 -= 32) {
      const int64_t x = x1 - 32 + lane;
      bool rstart = false, trig = false;
      if (x >= lo && x < hi && is_start(x)) {
        bool rs0;
        uint8_t raw0;
        uint32_t cp0;
        char_at((int)(x - ws), rs0, raw0, cp0);
        uint8_t rp = K_NONE, rn = K_NONE;
        uint32_t cpp = 0;
        if (!rs0) {                               // the previous char: at most 3 bytes back
          int64_t px = x - 1;
          while (px > x - 4 && px > 0 && !is_start(px)) --px;
          bool rsp;
          uint32_t cpv;
          char_at((int)(px - ws), rsp, rp, cpv);
          cpp = cpv < 128 ? cpv : 0x80u;
        }
        int64_t nx = x + 1;                       // the next char: at most 4 bytes on
        while (nx < x + 4 && nx < total && !is_start(nx)) ++nx;
        if (nx < total && is_start(nx)) {
          bool rsn;
          uint32_t cpn;
          uint8_t rawn;
          char_at((int)(nx - ws), rsn, rawn, cpn);
          if (!rsn) rn = rawn;
        }
        rstart = region_start(raw0, rp);
        trig = trigger(raw0, rp, cpp, rn);
      }
      const unsigned mr = __ballot_sync(0xffffffffu, rstart), mt = __ballot_sync(0xffffffffu, trig);
      if (mr) {
        const int fl = 31 - __clz(mr);
        xs = (int)(x1 - 32 + fl);
        const unsigned at_or_after = mt & ~((1u << fl) - 1);
        if (ys < 0 && at_or_after) ys = (int)(x1 - 32 + 31 - __clz(at_or_after));
      } else if (ys < 0 && mt) {
        ys = (int)(x1 - 32 + 31 - __clz(mt));
      }
    }
    if (lane == 0) W.s1_sum[t] = make_int2(xs, ys);
  }
}

// ---------------------------------------------------------------- tile carries
// A tile's carries come from the pre-pass summaries of the other tiles, found
// by one warp 32 summaries a step (usually one step: nearly every tile holds
// both kinds of event).

// Summary of tile u for the reverse queries (low byte rq_ws, high byte
// rq_up; 0xFF: none in the tile), 0xFFFF past the batch.
__device__ __forceinline__ int rq_summary(const Work &W, int u, int ntiles) {
  return u < ntiles ? (int)__ldcg(reinterpret_cast<const uint16_t *>(W.rq_sum) + u) : 0xFFFF;
}

// The reverse-query carry of tile t: per byte, the first event in the tiles
// after t, R_END past the batch (without rq_up events, as in cl100k- and
// deepseek-style, always R_END).  v: this lane's rq_summary of tile
// t + 1 + lane, loaded ahead.
__device__ int rq_carry_of(const Work &W, int t, int ntiles, bool want_up, int v) {
  const int lane = threadIdx.x & 31;
  int lo = 0xFF, hi = want_up ? 0xFF : (int)R_END;
  for (int u0 = t + 1;; u0 += 32) {
    const unsigned ml = __ballot_sync(0xffffffffu, (v & 0xFF) != 0xFF);
    const unsigned mh = __ballot_sync(0xffffffffu, (v >> 8) != 0xFF);
    if (lo == 0xFF && ml) lo = __shfl_sync(0xffffffffu, v & 0xFF, __ffs(ml) - 1);
    if (hi == 0xFF && mh) hi = __shfl_sync(0xffffffffu, v >> 8, __ffs(mh) - 1);
    if ((lo != 0xFF && hi != 0xFF) || u0 + 32 >= ntiles) break;
    v = rq_summary(W, u0 + 32 + lane, ntiles);
  }
  return (lo == 0xFF ? (int)R_END : lo) | ((hi == 0xFF ? (int)R_END : hi) << 8);
}

// The mark-resolution carry of tile t (o200k): the latest stretch start and
// the latest trigger in the tiles before t, -1 for none.  Summary positions
// grow with the tile index, so the latest is the nearest tile's.  v: this
// lane's summary of tile t - 1 - lane, loaded ahead.
__device__ int2 s1_carry_of(const Work &W, int t, int2 v) {
  const int lane = threadIdx.x & 31;
  int x = -1, y = -1;
  bool fx = false, fy = false;
  for (int u0 = t - 1;; u0 -= 32) {
    const unsigned mx = __ballot_sync(0xffffffffu, v.x >= 0), my = __ballot_sync(0xffffffffu, v.y >= 0);
    if (!fx && mx) { x = __shfl_sync(0xffffffffu, v.x, __ffs(mx) - 1); fx = true; }
    if (!fy && my) { y = __shfl_sync(0xffffffffu, v.y, __ffs(my) - 1); fy = true; }
    if ((fx && fy) || u0 < 32) break;
    const int u = u0 - 32 - lane;
    v = u >= 0 ? __ldcg(&W.s1_sum[u]) : make_int2(-1, -1);
  }
  return make_int2(x, y);
}

// ---------------------------------------------------------------- k_pretok
template <int NT>
struct PretokSmem {
  WinSmem<NT> w;
  uint8_t chain[WIN];
  uint16_t dagg[NT][3];  // scan values of chars whose predicate waits for the barrier
  S2 s2_tmp[NT / 32];        // (holds the family's scan state: S2, or the smaller S2L)
  int2 i2_tmp[NT / 32];
  int i_tmp[NT / 32];
  S2 s2_prefix;              // (likewise)
  int2 s1c;                  // mark-resolution carry (o200k)
  int rqc;                   // reverse-query carry
  int tile;
  int piece_base;
  int prev_last;
};

template <class WS>
__device__ __forceinline__ Nbr make_nbr(const WS &S, const uint8_t *chain, int j) {
  Nbr b;
  uint8_t e[5];
  uint32_t c[5];
  bool inside = true;
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int x = j - k;
    if (k > 0 && (x < 0 || S.rs(x + 1))) inside = false;
    e[k] = inside ? S.eff(x) : K_NONE;
    c[k] = inside ? S.cp8(x) : 0;
  }
  b.e0 = e[0]; b.e1 = e[1]; b.e2 = e[2]; b.e3 = e[3]; b.e4 = e[4];
  b.c0 = c[0]; b.c1 = c[1]; b.c2 = c[2]; b.c3 = c[3]; b.c4 = c[4];
  const bool in1 = j + 1 < S.nch && !S.rs(j + 1);
  const bool in2 = in1 && j + 2 < S.nch && !S.rs(j + 2);
  b.en1 = in1 ? S.eff(j + 1) : K_NONE;
  b.en2 = in2 ? S.eff(j + 2) : K_NONE;
  b.cn1 = in1 ? S.cp8(j + 1) : 0;
  b.cn2 = in2 ? S.cp8(j + 2) : 0;
  b.rs = S.rs(j) != 0;
  if (chain) {
    b.l1 = j >= 1 ? chain[j - 1] != 0 : true;
    b.l2 = j >= 2 ? chain[j - 2] != 0 : true;
    b.l3 = j >= 3 ? chain[j - 3] != 0 : true;
  } else {
    b.l1 = b.l2 = b.l3 = true;
  }
  return b;
}

// A char's neighbourhood slid along a thread's contiguous chars: each step
// shifts the lookback registers and loads only what enters the window.
struct Slider {
  static constexpr uint32_t NO_CHAR = 1u << 29;   // past the window's chars: reads as a request start
  Nbr b;
  int32_t pos, p1, p2;   // byte positions of j, j+1, j+2
  uint32_t w1, w2;       // char words of j+1, j+2 (one shared-memory load a step)
  template <class WS>
  __device__ __forceinline__ void start(const WS &S, int64_t ws, int j) {
    b = make_nbr(S, nullptr, j);
    w1 = j + 1 < S.nch ? S.ci[j + 1] : NO_CHAR;
    w2 = j + 2 < S.nch ? S.ci[j + 2] : NO_CHAR;
    pos = (int32_t)(ws + S.lead(j));
    p1 = j + 1 < S.nch ? (int32_t)(ws + ci_lead(w1)) : pos + 1;
    p2 = j + 2 < S.nch ? (int32_t)(ws + ci_lead(w2)) : pos + 2;
  }
  template <class WS>
  __device__ __forceinline__ void step(const WS &S, int64_t ws, int j) {   // from j - 1 to j
    const uint32_t w0 = w1;
    w1 = w2;
    w2 = j + 2 < S.nch ? S.ci[j + 2] : NO_CHAR;
    const bool rsj = ci_rs(w0);
    if (rsj) {
      b.e1 = b.e2 = b.e3 = b.e4 = K_NONE;
      b.c1 = b.c2 = b.c3 = b.c4 = 0;
      b.e0 = ci_eff(w0);
      b.c0 = ci_cp8(w0);
    } else {
      b.e4 = b.e3; b.e3 = b.e2; b.e2 = b.e1; b.e1 = b.e0; b.e0 = b.en1;
      b.c4 = b.c3; b.c3 = b.c2; b.c2 = b.c1; b.c1 = b.c0; b.c0 = b.cn1;
    }
    b.rs = rsj;
    const bool in1 = !ci_rs(w1);
    const bool in2 = in1 && !ci_rs(w2);
    if (!rsj) { b.en1 = in1 ? b.en2 : K_NONE; b.cn1 = in1 ? b.cn2 : 0; }   // old j+2 is new j+1
    else { b.en1 = in1 ? ci_eff(w1) : K_NONE; b.cn1 = in1 ? ci_cp8(w1) : 0; }
    b.en2 = in2 ? ci_eff(w2) : K_NONE;
    b.cn2 = in2 ? ci_cp8(w2) : 0;
    pos = p1;
    p1 = p2;
    p2 = j + 2 < S.nch ? (int32_t)(ws + ci_lead(w2)) : pos + 2;
  }
};

// The forward-scan state of a family: the 12-byte S2L for the families
// without a case rule, the full S2 for the o200k-style one.
template <int FAM> struct ScanOf { using T = S2L; };
template <> struct ScanOf<FAM_O200K> { using T = S2; };
__device__ __forceinline__ S2 st_identity(const S2 *) { return s2_identity(); }
__device__ __forceinline__ S2L st_identity(const S2L *) { return s2l_identity(); }
__device__ __forceinline__ S2 st_combine(const S2 &a, const S2 &b) { return s2_combine(a, b); }
__device__ __forceinline__ S2L st_combine(const S2L &a, const S2L &b) { return s2l_combine(a, b); }

// The reverse queries of char j of the tile (pos in [ts, te)), asked only
// where a rule reads them: the first rq_ws event (low byte, if want_ws) and
// rq_up event (high byte, if want_up) among the tile's chars after j, else
// the tile's carry (the first event in the tiles after it).
template <class WS>
__device__ __forceinline__ int rq_after(int fam, const WS &S, int64_t ws, int64_t te, int j, int carry, bool want_ws,
                                        bool want_up) {
  int lo = want_ws ? 0xFF : 0, hi = want_up ? 0xFF : 0;   // 0xFF: still searching
  for (int k = j + 1; k < S.nch && (lo == 0xFF || hi == 0xFF); ++k) {
    const uint32_t c = S.ci[k];
    if (ws + ci_lead(c) >= te) break;
    if (lo == 0xFF) {
      const uint8_t e = rq_ws_event(fam, ci_rs(c), ci_raw(c), ci_cp8(c));
      if (e != 0xFF) lo = e;
    }
    if (hi == 0xFF) {
      const uint8_t e = rq_up_event(ci_rs(c), ci_raw(c));
      if (e != 0xFF) hi = e;
    }
  }
  if (lo == 0xFF) lo = carry & 0xFF;
  if (hi == 0xFF) hi = (carry >> 8) & 0xFF;
  return lo | (hi << 8);
}

template <int FAM, int NT>
__global__ void __launch_bounds__(NT, NT == 512 ? 3 : 5) k_pretok(Tables T, Work W) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PretokSmem<NT> &P = *reinterpret_cast<PretokSmem<NT> *>(smem_raw);
  WinSmem<NT> &S = P.w;
  const CallArgs A = *W.args;
  const int tid = threadIdx.x;
  if (A.n <= 0) return;
  int64_t base, total;
  if (!batch_extent(A, base, total)) return;
  const int ntiles = (int)((total + TILE - 1) / TILE);
  if (tid == 0) P.tile = atomicAdd(&W.counters[0], 1);
  __syncthreads();
  const int t = P.tile;
  if (t >= ntiles) return;
  constexpr int fam = FAM;
  const int64_t ts = (int64_t)t * TILE, te = ts + TILE < total ? ts + TILE : total;
  const int64_t ws = ts - HALO_L;
  // the first steps of the carry searches load while the window does
  const int wid = tid >> 5, lane = tid & 31;
  int rq_v = 0;
  int2 s1_v = make_int2(-1, -1);
  if (wid == 0) rq_v = rq_summary(W, t + 1 + lane, ntiles);
  if (fam == FAM_O200K && wid == 1 && t - 1 - lane >= 0) s1_v = __ldcg(&W.s1_sum[t - 1 - lane]);
  load_window(T, A, base, total, ws, S, P.i_tmp, T.n_lit ? W.lit_flag : nullptr);
  const int c0 = S.cbase[tid], c1 = S.cbase[tid + 1];
  // (read after the barriers of the scans below)
  if (wid == 0) {
    const int c = rq_carry_of(W, t, ntiles, fam == FAM_O200K, rq_v);
    if (lane == 0) P.rqc = c;
  }
  if (fam == FAM_O200K && wid == 1) {
    const int2 c = s1_carry_of(W, t, s1_v);
    if (lane == 0) P.s1c = c;
  }

  // --- effective kinds (o200k: resolve marks with a max-scan entering at ts - 32)
  if (fam == FAM_O200K) {
    // (each pass slides the previous, own and next words along the thread's
    // chars: one shared-memory load a char)
    constexpr uint32_t PAST = 1u << 29;      // past the window's chars: reads as a request start
    int2 v = make_int2(-1, -1);
    if (c0 < c1) {
      uint32_t wp = c0 > 0 ? S.ci[c0 - 1] : 0, w0 = S.ci[c0];
      for (int j = c0; j < c1; ++j) {
        const uint32_t wn = j + 1 < S.nch ? S.ci[j + 1] : PAST;
        const int64_t pos = ws + ci_lead(w0);
        if (pos >= ts - S1_SHIFT) {
          const bool in_prev = !ci_rs(w0) && j > 0;
          const uint8_t rp = in_prev ? ci_raw(wp) : K_NONE;
          const uint32_t cpp = in_prev ? ci_cp8(wp) : 0;
          const uint8_t rn = !ci_rs(wn) ? ci_raw(wn) : K_NONE;
          if (region_start(ci_raw(w0), rp)) v.x = (int)pos;
          if (trigger(ci_raw(w0), rp, cpp, rn)) v.y = (int)pos;
        }
        wp = w0;
        w0 = wn;
      }
    }
    auto mx = [](int2 a, int2 b) { return make_int2(max(a.x, b.x), max(a.y, b.y)); };
    int2 ex = block_exclusive_scan<NT>(v, mx, make_int2(-1, -1), P.i2_tmp, (int2 *)nullptr);
    int2 run = mx(P.s1c, ex);
    if (c0 < c1) {
      uint32_t wp = c0 > 0 ? S.ci[c0 - 1] : 0, w0 = S.ci[c0];
      for (int j = c0; j < c1; ++j) {
        const uint32_t wn = j + 1 < S.nch ? S.ci[j + 1] : PAST;
        const int64_t pos = ws + ci_lead(w0);
        const uint8_t r0 = ci_raw(w0);
        bool mark_other = false;
        if (pos >= ts - S1_SHIFT) {
          const bool in_prev = !ci_rs(w0) && j > 0;
          const uint8_t rp = in_prev ? ci_raw(wp) : K_NONE;
          const uint32_t cpp = in_prev ? ci_cp8(wp) : 0;
          const uint8_t rn = !ci_rs(wn) ? ci_raw(wn) : K_NONE;
          if (region_start(r0, rp)) run.x = (int)pos;
          if (trigger(r0, rp, cpp, rn)) run.y = (int)pos;
          mark_other = r0 == K_MARK && run.x >= 0 && run.y >= run.x;
        }
        S.ci[j] = (w0 & ~(0xFu << 25)) | ((uint32_t)effective(fam, r0, mark_other) << 25);
        wp = w0;
        w0 = wn;
      }
    }
  } else {
    for (int j = c0; j < c1; ++j) {
      S.set_eff(j, effective(fam, S.raw(j), false));
      // deepseek-style: segment starts of the first two splitters act as
      // request starts (j = 0 has no predecessor in the window; it lies in
      // the left halo, further back than any rule or scan looks)
      if (fam == FAM_DEEPSEEK && j > 0 && ds_segment_start(S.raw(j - 1), S.raw(j))) S.set_rs(j);
    }
  }
  __syncthreads();

  // --- forward scan (scan 2) over chars with pos in [ts - 16, te); the
  // published aggregate covers the shifted tile [ts - 16, te - 16)
  using ST = typename ScanOf<FAM>::T;
  ST *st_tmp = reinterpret_cast<ST *>(P.s2_tmp);
  ST *st_agg = reinterpret_cast<ST *>(W.s2_agg), *st_inc = reinterpret_cast<ST *>(W.s2_inc);
  const ST st_id = st_identity((const ST *)nullptr);
  const int64_t s2_lo = ts - S2_SHIFT, s2_pub_hi = t == ntiles - 1 ? INT64_MAX : te - S2_SHIFT;
  int jlo = c0, jhi = c1;                       // my chars with pos in [s2_lo, te)
  while (jlo < jhi && ws + S.lead(jlo) < s2_lo) ++jlo;
  while (jhi > jlo && ws + S.lead(jhi - 1) >= te) --jhi;
  ST agg_all = st_id, agg_pub = st_id;
  bool pub_done = false;
  if constexpr (FAM == FAM_O200K) {
    if (jlo < jhi) {
      Slider w;
      w.start(S, ws, jlo);
      for (int j = jlo;;) {
        if (!pub_done && w.pos >= s2_pub_hi) { agg_pub = agg_all; pub_done = true; }
        if (!s2_trivial(fam, w.b)) agg_all = s2_combine(agg_all, s2_element(fam, w.b, w.pos, w.p1, w.p2));
        if (++j >= jhi) break;
        w.step(S, ws, j);
      }
    }
  } else {
    // only digits and blanks contribute, and their elements read nothing
    // but their own kind, code point and position and their predecessor's kind
    for (int j = jlo; j < jhi; ++j) {
      const uint32_t c = S.ci[j];
      const int32_t pos = (int32_t)(ws + ci_lead(c));
      if (!pub_done && pos >= s2_pub_hi) { agg_pub = agg_all; pub_done = true; }
      const uint8_t e0 = ci_eff(c);
      if (e0 == K_NUM || e0 == K_WS) {
        const uint8_t e1 = (ci_rs(c) || j == 0) ? (uint8_t)K_NONE : ci_eff(S.ci[j - 1]);
        agg_all = s2l_combine(agg_all, s2l_element(e0, e1, ci_cp8(c), pos));
      }
    }
  }
  if (!pub_done) agg_pub = agg_all;
  auto comb = [](const ST &a, const ST &b) { return st_combine(a, b); };
  ST tile_pub;
  block_exclusive_scan<NT>(agg_pub, comb, st_id, st_tmp, &tile_pub);
  // publish now: the successors' look-back runs while this tile scans its
  // own chars
  if (tid == 0 && t != W.withhold_tile) lookback_publish(t, tile_pub, st_agg, st_inc, W.s2_flag);
  const ST my_ex = block_exclusive_scan<NT>(agg_all, comb, st_id, st_tmp, (ST *)nullptr);
  if (tid < 32) {
    const ST pre = warp_lookback(t, tile_pub, comb, st_id, st_agg, st_inc, W.s2_flag, W.status,
                                 &W.counters[CTR_TIMEOUT], W.spin_limit, true, t == W.withhold_tile);
    if (tid == 0) *reinterpret_cast<ST *>(&P.s2_prefix) = pre;
  }
  __syncthreads();
  ST before = st_combine(*reinterpret_cast<const ST *>(&P.s2_prefix), my_ex);

  // --- walk: per-char scan values and the predicate.  o200k chars whose
  // contraction lookback reaches the previous thread's chars wait for the
  // barrier (their chain states are written by that thread in this walk).
  // The reverse queries (is a later CR/LF in this blank run; is the rest of
  // this letter run upper case) are answered only for the chars whose rule
  // reads them.
  uint32_t starts = 0, placeholder = 0, deferred = 0;   // bit (j - c0) for my chars (<= PT_BYTES)
  const bool filter = __ldcg(&W.counters[5]) != 0;
  auto decide = [&](int j, const Nbr &nb, const Aggs &a, int64_t pos) {
    bool st = piece_start(fam, nb, a);
    if (st && filter) {
      const int64_t r = lower_bound64(A.offs, A.n + 1, base + pos + 1) - 1;
      if (r >= 0 && r < A.n && W.bad[r]) {
        if (S.rsb[S.lead(j)]) placeholder |= 1u << (j - c0);   // the request's start, not a literal's
        else st = false;
      }
    }
    if (st) starts |= 1u << (j - c0);
  };
  // cl100k-style tiles of 16 bytes a thread (batches): inside a letter run or
  // a run of "other" chars no rule starts a piece (a letter run's only inner
  // starts follow an apostrophe two or three chars back), and such chars add
  // nothing to the scan; they are passed over reading their own and their
  // predecessor's words, and every other char builds its neighbourhood where
  // it stands.  Elsewhere the neighbourhood slides along the thread's chars:
  // on text with short runs (glued kana/CJK text) or 8 bytes a thread, the
  // lanes of a warp rarely all pass over the same step, and rebuilding a
  // neighbourhood costs more than sliding it.
  constexpr bool RUN_SKIP = FAM == FAM_CL100K && NT == 256;
  if constexpr (FAM == FAM_O200K) {
    for (int j = c0; j < jlo; ++j) P.chain[j] = 1;
    for (int j = jhi; j < c1; ++j) P.chain[j] = 1;
  } else if constexpr (RUN_SKIP) {
    for (int j = jlo; j < jhi; ++j) {
      const uint32_t c = S.ci[j];
      const uint8_t e0 = ci_eff(c);
      const bool rs = ci_rs(c);
      uint8_t e1 = K_NONE;
      uint32_t c1 = 0;
      if (!rs && j > 0) {
        const uint32_t w1 = S.ci[j - 1];
        e1 = ci_eff(w1);
        c1 = ci_cp8(w1);
      }
      if (!rs && j > 0 && (is_letter(e0) || e0 == K_OTHER)) {
        if (e0 == K_OTHER ? e1 == K_OTHER
                          : (is_letter(e1) && !(j >= 2 && ci_cp8(S.ci[j - 2]) == '\'') &&
                             !(j >= 3 && ci_cp8(S.ci[j - 3]) == '\'')))
          continue;
      }
      // the near fields suffice except for a letter after an "other" char or a letter
      Nbr nb;
      if (needs_far_nbr(e0, e1)) {
        nb = make_nbr(S, nullptr, j);
      } else {
        nb.e0 = e0; nb.c0 = ci_cp8(c); nb.rs = rs; nb.e1 = e1; nb.c1 = c1;
        nb.e2 = nb.e3 = nb.e4 = K_NONE; nb.c2 = nb.c3 = nb.c4 = 0;
        nb.en1 = nb.en2 = K_NONE; nb.cn1 = nb.cn2 = 0;
        nb.l1 = nb.l2 = nb.l3 = true;
        if (j + 1 < S.nch) {
          const uint32_t w = S.ci[j + 1];
          if (!ci_rs(w)) { nb.en1 = ci_eff(w); nb.cn1 = ci_cp8(w); }
        }
      }
      const int32_t pos = (int32_t)(ws + ci_lead(c));
      Aggs a{};
      if (e0 == K_NUM || e0 == K_WS) {
        const S2L after = s2l_combine(before, s2l_element(e0, nb.e1, nb.c0, pos));
        s2l_values(before, after, pos, a);
        before = after;
      }
      if (pos >= ts) {
        if (e0 == K_WS && is_crlf(nb.c1)) a.rq_ws = (uint8_t)(rq_after(fam, S, ws, te, j, P.rqc, true, false) & 0x3);
        decide(j, nb, a, pos);
      }
    }
  }
  if constexpr (FAM != FAM_O200K && !RUN_SKIP) {
    // the other tiles of the families without a case rule: the near fields
    // (own, predecessor's, successor's word) slide along the thread's chars
    // with the code points two and three back; a letter after a letter
    // starts nothing unless an apostrophe is two or three back, and a letter
    // after an "other" char or an apostrophe builds the rest
    if (jlo < jhi) {
      uint32_t w0 = S.ci[jlo];
      uint32_t wp = jlo > 0 ? S.ci[jlo - 1] : 0;
      uint32_t cp2 = jlo > 1 ? ci_cp8(S.ci[jlo - 2]) : 0, cp3 = jlo > 2 ? ci_cp8(S.ci[jlo - 3]) : 0;
      for (int j = jlo; j < jhi; ++j) {
        const uint32_t wn = j + 1 < S.nch ? S.ci[j + 1] : (1u << 29);   // past the window: a request start
        const bool rs = ci_rs(w0);
        Nbr nb;
        nb.e0 = ci_eff(w0); nb.c0 = ci_cp8(w0); nb.rs = rs;
        const bool in_p = !rs && j > 0, in_n = !ci_rs(wn);
        nb.e1 = in_p ? ci_eff(wp) : (uint8_t)K_NONE;
        nb.c1 = in_p ? ci_cp8(wp) : 0;
        nb.en1 = in_n ? ci_eff(wn) : (uint8_t)K_NONE;
        nb.cn1 = in_n ? ci_cp8(wn) : 0;
        nb.e2 = nb.e3 = nb.e4 = K_NONE; nb.c2 = nb.c3 = nb.c4 = 0;
        nb.en2 = K_NONE; nb.cn2 = 0;
        nb.l1 = nb.l2 = nb.l3 = true;
        const int32_t pos = (int32_t)(ws + ci_lead(w0));
        Aggs a{};
        if (nb.e0 == K_NUM || nb.e0 == K_WS) {   // the only chars whose rules read scan values
          const S2L after = s2l_combine(before, s2l_element(nb.e0, nb.e1, nb.c0, pos));
          s2l_values(before, after, pos, a);
          before = after;
        }
        const bool inner = is_letter(nb.e0) && is_letter(nb.e1) && cp2 != '\'' && cp3 != '\'';
        if (pos >= ts && !inner) {
          if (needs_far_nbr(nb.e0, nb.e1)) nb = make_nbr(S, nullptr, j);
          if (nb.e0 == K_WS && is_crlf(nb.c1)) a.rq_ws = (uint8_t)(rq_after(fam, S, ws, te, j, P.rqc, true, false) & 0x3);
          decide(j, nb, a, pos);
        }
        cp3 = cp2;
        cp2 = ci_cp8(wp);
        wp = w0;
        w0 = wn;
      }
    }
  }
  if (FAM == FAM_O200K && jlo < jhi) {
    Slider w;
    w.start(S, ws, jlo);
    // chain states of the three chars before jlo (valid for o200k only where
    // they belong to this thread; other cases are deferred below)
    bool l1 = true, l2 = true, l3 = true;
    if constexpr (FAM == FAM_O200K) {
      l1 = jlo >= 1 ? P.chain[jlo - 1] != 0 : true;
      l2 = jlo >= 2 ? P.chain[jlo - 2] != 0 : true;
      l3 = jlo >= 3 ? P.chain[jlo - 3] != 0 : true;
    }
    for (int j = jlo;;) {
      Aggs a{};
      bool ch = true;
      if constexpr (FAM == FAM_O200K) {
        const S2 after = s2_trivial(fam, w.b) ? before : s2_combine(before, s2_element(fam, w.b, w.pos, w.p1, w.p2));
        s2_values(before, after, w.pos, a, ch);
        before = after;
        P.chain[j] = ch ? 1 : 0;
      } else if (w.b.e0 == K_NUM || w.b.e0 == K_WS) {   // the only chars whose rules read scan values
        const S2L after = s2l_combine(before, s2l_element(w.b.e0, w.b.e1, w.b.c0, w.pos));
        s2l_values(before, after, w.pos, a);
        before = after;
      }
      if (w.pos >= ts) {
        const Nbr &nb = w.b;
        const bool want_ws = nb.e0 == K_WS && is_crlf(nb.c1);
        const bool want_up = FAM == FAM_O200K && nb.e0 == K_LU && nb.e1 == K_LB;
        if (want_ws || want_up) {
          const int q = rq_after(fam, S, ws, te, j, P.rqc, want_ws, want_up);
          a.rq_ws = (uint8_t)(q & 0x3);
          a.rq_up = (uint8_t)((q >> 8) & 0x3);
        }
        // (chain states are read only next to an apostrophe: c0 with l1, c2 with l2, c3 with l3)
        if (FAM == FAM_O200K && j < c0 + 3 &&
            (nb.c0 == '\'' || nb.c1 == '\'' || nb.c2 == '\'' || nb.c3 == '\'')) {
          deferred |= 1u << (j - c0);
          P.dagg[tid][j - c0] = (uint16_t)(a.nidx3 | (a.w_start << 2) | (a.w_prev_other << 3) |
                                           (a.w_ncw_before << 4) | (a.case_prev << 5) | (a.rq_ws << 7) |
                                           (a.rq_up << 9));
        } else {
          Nbr nbl = nb;
          nbl.l1 = l1; nbl.l2 = l2; nbl.l3 = l3;
          decide(j, nbl, a, w.pos);
        }
      }
      l3 = l2; l2 = l1; l1 = ch;
      if (++j >= jhi) break;
      w.step(S, ws, j);
    }
  }
  __syncthreads();
  for (uint32_t m = deferred; m; m &= m - 1) {
    const int j = c0 + __ffs(m) - 1;
    const int64_t pos = ws + S.lead(j);
    const Nbr nb = make_nbr(S, P.chain, j);
    const uint16_t g = P.dagg[tid][j - c0];
    Aggs a;
    a.nidx3 = g & 3;
    a.w_start = (g >> 2) & 1;
    a.w_prev_other = (g >> 3) & 1;
    a.w_ncw_before = (g >> 4) & 1;
    a.case_prev = (g >> 5) & 3;
    a.rq_ws = (g >> 7) & 3;
    a.rq_up = (g >> 9) & 3;
    decide(j, nb, a, pos);
  }
  // --- compaction of piece starts.  The count scan also carries the latest
  // piece start (pos * 2 + placeholder bit), so each tile learns the start of
  // the piece running into it and can classify every piece by length as soon
  // as its successor's start is known: pieces longer than SMALL_MAX bytes are
  // listed for the warp BPE kernel (three buckets by length, so that the
  // longest are taken first) or, beyond MID_MAX bytes, the block kernel.
  int my_first = INT_MAX, my_last = -1;
  for (uint32_t m = starts; m; m &= m - 1) {
    const int b = __ffs(m) - 1;
    const int code = (int)(ws + S.lead(c0 + b)) * 2 + (int)((placeholder >> b) & 1);
    if (my_first == INT_MAX) my_first = code;
    my_last = code;
  }
  auto cnt_op = [](int2 a, int2 b) { return make_int2(a.x + b.x, max(a.y, b.y)); };
  int2 tile_agg;
  const int2 my_cnt = block_exclusive_scan<NT>(make_int2(__popc(starts), my_last), cnt_op, make_int2(0, -1),
                                                      P.i2_tmp, &tile_agg);
  int tile_first;
  const int next_after_me = block_exclusive_suffix<NT>(my_first, [](int a, int b) { return min(a, b); },
                                                               INT_MAX, P.i_tmp, &tile_first);
  if (tid < 32) {
    const int2 pb = warp_lookback(t, tile_agg, cnt_op, make_int2(0, -1), W.cnt_agg, W.cnt_inc, W.cnt_flag, W.status,
                                  &W.counters[CTR_TIMEOUT], W.spin_limit, false, t == W.withhold_tile);
    if (tid == 0) {
      P.piece_base = pb.x;
      P.prev_last = pb.y;
      if (t == ntiles - 1) {
        W.counters[3] = pb.x + tile_agg.x;
        W.piece_start[pb.x + tile_agg.x] = (int32_t)total;
      }
    }
  }
  __syncthreads();
  const bool last_tile = t == ntiles - 1;
  const int64_t lcap = list_cap(W.cap_bytes);
  auto classify = [&](int index, int code, int64_t end) {
    const int64_t len = end - (code >> 1);
    if ((code & 1) || len <= SMALL_MAX) return;
    if (len > MID_MAX) {
      W.huge_list[atomicAdd(&W.counters[6], 1)] = index;
    } else {
      const int b = mid_bucket(len);
      W.long_list[b * lcap + atomicAdd(&W.counters[mid_bucket_counter(b)], 1)] = index;
    }
  };
  int k = P.piece_base + my_cnt.x;
  int prev_code = -1;
  for (uint32_t m = starts; m; m &= m - 1) {
    const int b = __ffs(m) - 1;
    const int j = c0 + b;
    const int32_t pos = (int32_t)(ws + S.lead(j));
    const bool ph = (placeholder >> b) & 1;
    W.piece_start[k] = ph ? (int32_t)(pos | 0x80000000u) : pos;
    if (S.rsb[S.lead(j)]) {                   // first piece of the requests starting here
      int r = S.r0 + (int)lower_bound64(A.offs + S.r0, S.r1 - S.r0, base + pos);
      for (; r < S.r1 && __ldg(&A.offs[r]) == base + pos; ++r) W.req_piece[r] = k;
    }
    if (prev_code >= 0) classify(k - 1, prev_code, pos);
    prev_code = pos * 2 + (ph ? 1 : 0);
    ++k;
  }
  if (prev_code >= 0) {                       // my last piece ends at the next start of the tile
    if (next_after_me != INT_MAX) classify(k - 1, prev_code, next_after_me >> 1);
    else if (last_tile) classify(k - 1, prev_code, total);
  }
  if (tid == 0 && P.prev_last >= 0) {         // the piece running into this tile
    if (tile_agg.x > 0) classify(P.piece_base - 1, P.prev_last, tile_first >> 1);
    else if (last_tile) classify(P.piece_base - 1, P.prev_last, total);
  }
}

// Threads per window: 512 (8 bytes each) for workspaces up to
// PT_NARROW_MAX_BYTES, whose batches leave most SMs idle at 16 bytes a
// thread; 256 (16 bytes each) above, where the GPU is full either way and
// fewer threads mean fewer instructions.
constexpr int64_t PT_NARROW_MAX_BYTES = 4ll << 20;
static bool pt_narrow(const Work &W) { return W.cap_bytes <= PT_NARROW_MAX_BYTES; }


void launch_prepass(const Tables &T, const Work &W, int grid, cudaStream_t s) {
  if (pt_narrow(W)) k_prepass<WIN / 8><<<grid, WIN / 8, 0, s>>>(T, W);
  else k_prepass<WIN / 16><<<grid, WIN / 16, 0, s>>>(T, W);
}
template <int NT>
static void launch_pretok_nt(const Tables &T, const Work &W, int grid, cudaStream_t s) {
  if (T.family == FAM_O200K) k_pretok<FAM_O200K, NT><<<grid, NT, sizeof(PretokSmem<NT>), s>>>(T, W);
  else if (T.family == FAM_DEEPSEEK) k_pretok<FAM_DEEPSEEK, NT><<<grid, NT, sizeof(PretokSmem<NT>), s>>>(T, W);
  else k_pretok<FAM_CL100K, NT><<<grid, NT, sizeof(PretokSmem<NT>), s>>>(T, W);
}
void launch_pretok(const Tables &T, const Work &W, int grid, cudaStream_t s) {
  if (pt_narrow(W)) launch_pretok_nt<WIN / 8>(T, W, grid, s);
  else launch_pretok_nt<WIN / 16>(T, W, grid, s);
}
template <int FAM, int NT>
static cudaError_t configure_one() {
  return cudaFuncSetAttribute(k_pretok<FAM, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sizeof(PretokSmem<NT>));
}
cudaError_t pretok_configure() {
  cudaError_t e;
  if ((e = configure_one<FAM_CL100K, WIN / 8>()) != cudaSuccess) return e;
  if ((e = configure_one<FAM_O200K, WIN / 8>()) != cudaSuccess) return e;
  if ((e = configure_one<FAM_DEEPSEEK, WIN / 8>()) != cudaSuccess) return e;
  if ((e = configure_one<FAM_CL100K, WIN / 16>()) != cudaSuccess) return e;
  if ((e = configure_one<FAM_DEEPSEEK, WIN / 16>()) != cudaSuccess) return e;
  return configure_one<FAM_O200K, WIN / 16>();
}

}  // namespace tt
