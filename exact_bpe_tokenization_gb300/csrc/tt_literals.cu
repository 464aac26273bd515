// tt_literals.cu - added-token literal extraction before the pattern family
// (TokTier: Exact Stateful CPU+GPU Tokenization for Agentic LLM Serving,
// §4.4: added and special tokens are literal strings the model reserves as
// single IDs; a leftmost-longest literal pass extracts them before the
// tokenizer family handles the remaining segments).
//
// k_lit_find: one CTA per 4,016-byte tile; each byte position gets the
// longest literal that starts there and ends inside its request (literals
// are grouped by first byte, longest first), and the tile's candidates are
// compacted in position order.
// k_lit_pick: a warp per request walks the candidates of its tiles in order
// (tiles without any are skipped 32 at a time) and takes every candidate
// that starts at or after the end of the last one taken: leftmost-longest.
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

__global__ void __launch_bounds__(LF_THREADS) k_lit_find(Tables T, Work W) {
  __shared__ int red[LF_THREADS / 32];
  const CallArgs A = *W.args;
  const int tid = threadIdx.x;
  if (A.n <= 0) return;
  const int64_t base = __ldg(&A.offs[0]);
  const int64_t total = __ldg(&A.offs[A.n]) - base;
  if (total > W.cap_bytes || total < 0 || base < 0) return;
  const int ntiles = (int)((total + TILE - 1) / TILE);
  const int t = blockIdx.x;
  if (t >= ntiles) return;
  const int64_t ts = (int64_t)t * TILE, te = ts + TILE < total ? ts + TILE : total;
  const uint8_t *g = A.utf8 + base;
  uint32_t found = 0;
  int code[LF_BYTES];
  int64_t rend = -1;                        // end of the request holding my latest candidate
#pragma unroll
  for (int k = 0; k < LF_BYTES; ++k) {
    code[k] = 0;
    const int64_t x = ts + (int64_t)LF_BYTES * tid + k;
    if (x >= te) continue;
    const uint8_t b = __ldg(g + x);
    const int lo = __ldg(&T.lit_first[b]), hi = __ldg(&T.lit_first[b + 1]);
    for (int q = lo; q < hi; ++q) {           // longest first
      const int li = __ldg(&T.lit_order[q]);
      const int off = __ldg(&T.lit_off[li]), len = __ldg(&T.lit_off[li + 1]) - off;
      if (x + len > total || !same_bytes(g + x, T.lit_bytes + off, len)) continue;
      if (x >= rend) {                        // (rend only grows: my positions increase)
        const int64_t r = request_of(A.offs, A.n, base + x);
        rend = __ldg(&A.offs[r + 1]) - base;
      }
      if (x + len > rend) continue;           // would run into the next request
      code[k] = (int)(x - ts) | (li << 12);
      found |= 1u << k;
      break;
    }
  }
  int tile_total;
  int at = block_exclusive_scan<LF_THREADS>(__popc(found), [](int a, int b) { return a + b; }, 0, red, &tile_total);
#pragma unroll
  for (int k = 0; k < LF_BYTES; ++k)
    if (found >> k & 1u) W.lit_cand[(int64_t)t * TILE + at++] = code[k];
  if (tid == 0) W.lit_cnt[t] = tile_total;
}

__global__ void __launch_bounds__(256) k_lit_pick(Tables T, Work W) {
  const CallArgs A = *W.args;
  const int lane = threadIdx.x & 31;
  if (A.n <= 0) return;
  const int64_t base = __ldg(&A.offs[0]);
  const int64_t total = __ldg(&A.offs[A.n]) - base;
  if (total > W.cap_bytes || total < 0 || base < 0) return;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < A.n; r += nwarps) {
    const int64_t rs = __ldg(&A.offs[r]) - base, re = __ldg(&A.offs[r + 1]) - base;
    if (re <= rs || rs < 0 || re > total) continue;
    const int t0 = (int)(rs / TILE), t1 = (int)((re - 1) / TILE);
    int64_t cover = rs;                       // bytes below cover lie inside a taken literal
    for (int tb = t0; tb <= t1; tb += 32) {
      const int c = tb + lane <= t1 ? __ldcg(&W.lit_cnt[tb + lane]) : 0;
      for (unsigned m = __ballot_sync(0xffffffffu, c > 0); m; m &= m - 1) {
        const int src = __ffs(m) - 1;
        const int tt = tb + src, cnt = __shfl_sync(0xffffffffu, c, src);
        for (int i0 = 0; i0 < cnt; i0 += 32) {
          int64_t x = -1;
          int len = 0;
          if (i0 + lane < cnt) {
            const int code = __ldcg(&W.lit_cand[(int64_t)tt * TILE + i0 + lane]);
            const int li = code >> 12;
            x = (int64_t)tt * TILE + (code & 0xFFF);
            len = __ldg(&T.lit_off[li + 1]) - __ldg(&T.lit_off[li]);
            if (x < rs || x >= re) x = -1;      // another request's candidate
          }
          unsigned sel = 0;
          for (int j = 0; j < 32; ++j) {        // in position order, the same on every lane
            const int64_t xj = __shfl_sync(0xffffffffu, x, j);
            const int lj = __shfl_sync(0xffffffffu, len, j);
            if (xj >= 0 && xj >= cover) { sel |= 1u << j; cover = xj + lj; }
          }
          if (sel >> lane & 1u) {
            W.lit_flag[x] = LIT_SEG;
            for (int q = 1; q < len; ++q) W.lit_flag[x + q] = LIT_INNER;
            if (x + len < re) W.lit_flag[x + len] = LIT_SEG;
          }
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
