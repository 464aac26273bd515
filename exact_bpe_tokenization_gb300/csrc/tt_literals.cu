// tt_literals.cu - added-token literal extraction before the pattern family
// (TokTier: Exact Stateful CPU+GPU Tokenization for Agentic LLM Serving,
// §4.4: added and special tokens are literal strings the model reserves as
// single IDs; a leftmost-longest literal pass extracts them before the
// tokenizer family handles the remaining segments).
//
// Candidates: at every byte position the longest literal that starts there
// and ends inside its request (literals are grouped by first byte, longest
// first).  Literals are at most LIT_MAX_LEN bytes, so whether an earlier
// candidate reaches over position x is decided within LIT_MAX_LEN bytes
// before x.  A candidate that no earlier candidate reaches over (a head) is
// always taken: nothing before it can cover it.  The candidates after a head
// whose literals chain-overlap it form its cluster, and the leftmost-longest
// choice inside a cluster depends on nothing outside it; so the heads are
// independent starting points.
//
// k_lit_find: one CTA per 4,016-byte tile; writes every byte's candidate
// length (0: none), finds the heads with a max-scan of "reach" (candidate
// end) over the tile and the LIT_MAX_LEN bytes before it, and lists the heads.
// k_lit_pick: a thread per head walks its cluster in position order, taking a
// candidate when it starts at or after the end of the last one taken (the
// cluster ends where no candidate reaches further) -- in ordinary text every
// candidate is a head and the walk is its own literal.
// A taken literal marks its first byte and the byte after it as segment
// starts and its other bytes as inner bytes; the pre-tokenizer then treats a
// segment start like a request start (runs are cut there) and never starts a
// piece on an inner byte, so each literal is one piece, which the whole-piece
// probe maps to its reserved ID.
#include "tt_common.cuh"
#include "tt_kernels.h"

namespace tt {

namespace {

constexpr int LF_THREADS = 256;
constexpr int LF_BYTES = 16;              // bytes per thread: 256 x 16 >= TILE
static_assert(LF_THREADS * LF_BYTES >= TILE, "a tile per CTA");

// first request index r with offs[r] > v, minus one: the request holding v
__device__ __forceinline__ int64_t request_of(const int64_t *offs, int64_t n, int64_t v) {
  int64_t lo = 0, hi = n + 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (__ldg(&offs[mid]) <= v) lo = mid + 1;
    else hi = mid;
  }
  return lo - 1;
}

// bytes a[0..len) == b[0..len)
__device__ __forceinline__ bool same_bytes(const uint8_t *a, const uint8_t *b, int len) {
  for (int i = 0; i < len; i += 8)
    if (load8(a + i, len - i) != load8(b + i, len - i)) return false;
  return true;
}

}  // namespace

// length of the longest literal that starts at batch byte x and ends inside
// its request, 0 if none; *rend caches the end of the request holding the
// previous query (queries come in increasing x)
__device__ __forceinline__ int candidate_len(const Tables &T, const CallArgs &A, int64_t base, int64_t total,
                                             const uint8_t *g, int64_t x, int64_t *rend) {
  const uint8_t b = __ldg(g + x);
  const int lo = __ldg(&T.lit_first[b]), hi = __ldg(&T.lit_first[b + 1]);
  for (int q = lo; q < hi; ++q) {           // longest first
    const int li = __ldg(&T.lit_order[q]);
    const int off = __ldg(&T.lit_off[li]), len = __ldg(&T.lit_off[li + 1]) - off;
    if (x + len > total || !same_bytes(g + x, T.lit_bytes + off, len)) continue;
    if (x >= *rend) {
      const int64_t r = request_of(A.offs, A.n, base + x);
      *rend = __ldg(&A.offs[r + 1]) - base;
    }
    if (x + len <= *rend) return len;       // else it would run into the next request
  }
  return 0;
}

__global__ void __launch_bounds__(LF_THREADS) k_lit_find(Tables T, Work W) {
  __shared__ int red[LF_THREADS / 32];
  const CallArgs A = *W.args;
  const int tid = threadIdx.x;
  if (A.n <= 0) return;
  int64_t base, total;
  if (!batch_extent(A, base, total)) return;
  const int ntiles = (int)((total + TILE - 1) / TILE);
  const int t = blockIdx.x;
  if (t >= ntiles) return;
  const int64_t ts = (int64_t)t * TILE, te = ts + TILE < total ? ts + TILE : total;
  const uint8_t *g = A.utf8 + base;
  auto mx = [](int a, int b) { return a > b ? a : b; };
  // candidates of the LIT_MAX_LEN bytes before the tile only reach into it
  int reach_before = -1;
  {
    const int64_t y = ts - LIT_MAX_LEN + tid;
    int64_t rend = -1;
    if (tid < LIT_MAX_LEN && y >= 0) {
      const int len = candidate_len(T, A, base, total, g, y, &rend);
      if (len) reach_before = (int)(y + len);
    }
  }
  int halo_reach;
  block_exclusive_scan<LF_THREADS>(reach_before, mx, -1, red, &halo_reach);
  int len[LF_BYTES];
  int my_reach = -1;
  int64_t rend = -1;
#pragma unroll
  for (int k = 0; k < LF_BYTES; ++k) {
    const int64_t x = ts + (int64_t)LF_BYTES * tid + k;
    len[k] = x < te ? candidate_len(T, A, base, total, g, x, &rend) : 0;
    if (x < te) W.lit_len[x] = (uint8_t)len[k];
    if (len[k]) my_reach = mx(my_reach, (int)(x + len[k]));
  }
  int carry = mx(halo_reach, block_exclusive_scan<LF_THREADS>(my_reach, mx, -1, red, (int *)nullptr));
  uint32_t heads = 0;
#pragma unroll
  for (int k = 0; k < LF_BYTES; ++k) {
    if (!len[k]) continue;
    const int x = (int)(ts + LF_BYTES * tid + k);
    if (carry <= x) heads |= 1u << k;        // nothing earlier reaches over x
    carry = mx(carry, x + len[k]);
  }
  int tile_total;
  int at = block_exclusive_scan<LF_THREADS>(__popc(heads), [](int a, int b) { return a + b; }, 0, red, &tile_total);
#pragma unroll
  for (int k = 0; k < LF_BYTES; ++k)
    if (heads >> k & 1u) W.lit_cand[(int64_t)t * TILE + at++] = LF_BYTES * tid + k;
  if (tid == 0) W.lit_cnt[t] = tile_total;
}

__device__ __forceinline__ void mark_literal(uint8_t *flag, int64_t x, int len) {
  flag[x] = LIT_SEG;
  for (int q = 1; q < len; ++q) flag[x + q] = LIT_INNER;
  flag[x + len] = LIT_SEG;                  // (at a request start or the batch end: harmless)
}

__global__ void __launch_bounds__(256) k_lit_pick(Tables T, Work W) {
  const CallArgs A = *W.args;
  const int lane = threadIdx.x & 31;
  if (A.n <= 0) return;
  int64_t base, total;
  if (!batch_extent(A, base, total)) return;
  const int ntiles = (int)((total + TILE - 1) / TILE);
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < ntiles; t += nwarps) {
    const int cnt = __ldcg(&W.lit_cnt[t]);
    for (int i = lane; i < cnt; i += 32) {   // a head: taken, then its cluster
      const int64_t x = (int64_t)t * TILE + __ldcg(&W.lit_cand[(int64_t)t * TILE + i]);
      int64_t cover = x + __ldcg(&W.lit_len[x]), reach = cover;
      mark_literal(W.lit_flag, x, (int)(cover - x));
      for (int64_t p = x + 1; p < reach; ++p) {
        const int l = __ldcg(&W.lit_len[p]);
        if (!l) continue;
        if (p + l > reach) reach = p + l;
        if (p >= cover) {
          mark_literal(W.lit_flag, p, l);
          cover = p + l;
        }
      }
    }
  }
}

void launch_lit_find(const Tables &T, const Work &W, int grid, cudaStream_t s) {
  k_lit_find<<<grid, LF_THREADS, 0, s>>>(T, W);
}
void launch_lit_pick(const Tables &T, const Work &W, int grid, cudaStream_t s) {
  k_lit_pick<<<grid, 256, 0, s>>>(T, W);
}

}  // namespace tt
