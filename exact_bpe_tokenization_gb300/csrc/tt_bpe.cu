// tt_bpe.cu - segmented byte-level BPE over the piece table and output
// compaction (TokTier: Exact Stateful CPU+GPU Tokenization for Agentic LLM
// Serving, §4.2 "segmented BPE" and §4.3 "output compaction").
//
// Every piece is encoded independently.  A piece whose bytes are a
// vocabulary entry is emitted as that one ID (the whole-piece shortcut).
// Otherwise merging proceeds in rounds: the lowest rank present among
// adjacent pairs names one pair, and every leftmost non-overlapping
// occurrence of it is merged in one sweep; only pairs next to a merge are
// looked up again.  With a well-ordered merge list (checked when the handle
// is created) a round equals that many single leftmost merges.
//
// Execution units by piece length: a thread per piece up to 32 bytes
// (state in thread-local arrays); a 512-thread block per longer piece
// (state in global memory, compacted in place each round).  IDs land in a
// byte-indexed scratch array; k_ids scans the per-piece counts with
// decoupled look-back and writes the final contiguous IDs.
#include <limits.h>

#include "tt_common.cuh"
#include "tt_kernels.h"

namespace tt {

// whole-piece vocabulary probe; b points to len bytes (any memory space)
__device__ __forceinline__ int vocab_probe(const Tables &T, const uint8_t *b, int len) {
  const uint64_t h = hash_bytes(b, len);
  const uint32_t fp = vocab_fp(h);
  uint32_t s = (uint32_t)h & T.vocab_mask;
  for (;;) {
    const uint64_t e = __ldg(&T.vocab_tab[s]);
    if (e == 0) return -1;
    if ((uint32_t)(e >> 32) == fp && (int)((e >> 20) & 0xFFF) == len) {
      const int id = (int)(e & 0xFFFFF);
      const uint8_t *v = T.vbytes + __ldg(&T.voff[id]);
      bool same = true;
      for (int i = 0; i < len && same; ++i) same = __ldg(&v[i]) == b[i];
      if (same) return id;
    }
    s = (s + 1) & T.vocab_mask;
  }
}

// ---------------------------------------------------------------- small
__global__ void __launch_bounds__(BPE_SMALL_THREADS) k_bpe_small(Tables T, Work W) {
  const CallArgs A = *W.args;
  if (A.n <= 0) return;
  const int64_t base = __ldg(&A.offs[0]);
  const int64_t total = __ldg(&A.offs[A.n]) - base;
  if (total > W.cap_bytes || total < 0 || base < 0) return;
  const int np = __ldcg(&W.counters[3]);
  const uint8_t *g = A.utf8 + base;
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < np; k += gridDim.x * blockDim.x) {
    const int32_t s = __ldcg(&W.piece_start[k]);
    if (s < 0) { W.n_ids[k] = 0; continue; }                         // rejected request
    const int32_t e = __ldcg(&W.piece_start[k + 1]) & 0x7FFFFFFF;
    const int len = e - s;
    if (len <= 0 || e > total) { W.n_ids[k] = 0; set_status(W.status, ST_INVALID_ARG); continue; }
    if (len > SMALL_MAX) {
      W.long_list[atomicAdd(&W.counters[2], 1)] = k;
      continue;
    }
    uint8_t buf[SMALL_MAX];
    for (int i = 0; i < len; ++i) buf[i] = __ldg(g + s + i);
    int32_t *out = W.scratch + s;
    if (len <= T.max_tok_len) {
      const int id = vocab_probe(T, buf, len);
      if (id >= 0) { out[0] = id; W.n_ids[k] = 1; continue; }
    }
    int ids[SMALL_MAX], rk[SMALL_MAX];
    int n = len;
    for (int i = 0; i < n; ++i) ids[i] = __ldg(&T.byte_id[buf[i]]);
    for (int i = 0; i + 1 < n; ++i) rk[i] = pair_rank(T, ids[i], ids[i + 1]);
    for (;;) {
      int r = INT_MAX;
      for (int i = 0; i + 1 < n; ++i)
        if (rk[i] >= 0 && rk[i] < r) r = rk[i];
      if (r == INT_MAX) break;
      const int res = __ldg(&T.merge_result[r]);
      // one sweep: merge every leftmost non-overlapping occurrence of rank r;
      // ranks of untouched pairs are kept, pairs next to a merge are looked up
      int w = 0, i = 0;
      bool prev_merged = false;
      while (i < n) {
        const bool m = (i + 1 < n) && rk[i] == r;
        const int tok = m ? res : ids[i];
        if (w > 0) rk[w - 1] = (m || prev_merged) ? pair_rank(T, ids[w - 1], tok) : rk[i - 1];
        ids[w] = tok;
        prev_merged = m;
        ++w;
        i += m ? 2 : 1;
      }
      n = w;
    }
    for (int i = 0; i < n; ++i) out[i] = ids[i];
    W.n_ids[k] = n;
  }
}

// ---------------------------------------------------------------- long
__global__ void __launch_bounds__(BPE_LONG_THREADS) k_bpe_long(Tables T, Work W) {
  constexpr int NT = BPE_LONG_THREADS;
  __shared__ int red[NT / 32];
  __shared__ uint8_t sel_s[NT];
  __shared__ int s_whole;
  const CallArgs A = *W.args;
  const int tid = threadIdx.x;
  if (A.n <= 0) return;
  const int64_t base = __ldg(&A.offs[0]);
  const int64_t total = __ldg(&A.offs[A.n]) - base;
  if (total > W.cap_bytes || total < 0 || base < 0) return;
  const int nl = __ldcg(&W.counters[2]);
  const uint8_t *g = A.utf8 + base;
  auto plus = [](int a, int b) { return a + b; };
  auto mx = [](int a, int b) { return a > b ? a : b; };
  auto mn = [](int a, int b) { return a < b ? a : b; };
  for (int li = blockIdx.x; li < nl; li += gridDim.x) {
    const int k = __ldcg(&W.long_list[li]);
    const int32_t s = __ldcg(&W.piece_start[k]);
    const int32_t e = __ldcg(&W.piece_start[k + 1]) & 0x7FFFFFFF;
    const int len = e - s;
    if (len <= 0 || e > total) {
      if (tid == 0) W.n_ids[k] = 0;
      continue;
    }
    const uint8_t *b = g + s;
    int32_t *tok = W.scratch + s;
    int32_t *rk = W.tmp_a + s;
    if (len <= T.max_tok_len) {
      if (tid == 0) s_whole = vocab_probe(T, b, len);
      __syncthreads();
      const int whole = s_whole;
      __syncthreads();
      if (whole >= 0) {
        if (tid == 0) { tok[0] = whole; W.n_ids[k] = 1; }
        continue;
      }
    }
    int n = len;
    for (int i = tid; i < n; i += NT) tok[i] = __ldg(&T.byte_id[__ldg(b + i)]);
    __syncthreads();
    for (int i = tid; i + 1 < n; i += NT) rk[i] = pair_rank(T, tok[i], tok[i + 1]);
    __syncthreads();
    for (;;) {
      int lm = INT_MAX;
      for (int i = tid; i + 1 < n; i += NT)
        if (rk[i] >= 0 && rk[i] < lm) lm = rk[i];
      int r;
      block_exclusive_scan<NT>(lm, mn, INT_MAX, red, &r);
      if (r == INT_MAX) break;
      const int res = __ldg(&T.merge_result[r]);
      // in-place compaction, chunk by chunk; carries: run start (position
      // after the last non-hit), kept count, selected flag of the previous
      // element
      int carry_run = 0, carry_keep = 0;
      bool prev_sel = false;
      for (int c = 0; c < n; c += NT) {
        const int i = c + tid;
        const bool hit = i + 1 < n && rk[i] == r;
        const int tv = i < n ? tok[i] : 0;
        const int v = (i < n && !hit) ? i + 1 : -1;
        int chunk_max;
        const int ex_run = block_exclusive_scan<NT>(v, mx, -1, red, &chunk_max);
        const int run = mx(carry_run, mx(ex_run, v));      // inclusive; v = -1 for hits
        const bool sel = hit && ((i - run) % 2 == 0);
        sel_s[tid] = sel;
        __syncthreads();
        const bool removed = tid == 0 ? prev_sel : sel_s[tid - 1] != 0;
        const bool keep = i < n && !removed;
        int chunk_keep;
        const int ex_keep = block_exclusive_scan<NT>(keep ? 1 : 0, plus, 0, red, &chunk_keep);
        if (keep) tok[carry_keep + ex_keep] = sel ? res : tv;   // reads of this chunk are done
        const bool last_sel = sel_s[NT - 1] != 0;
        carry_run = mx(carry_run, chunk_max);
        carry_keep += chunk_keep;
        prev_sel = last_sel;
        __syncthreads();
      }
      n = carry_keep;
      for (int i = tid; i + 1 < n; i += NT) rk[i] = pair_rank(T, tok[i], tok[i + 1]);
      __syncthreads();
    }
    if (tid == 0) W.n_ids[k] = n;
    __syncthreads();
  }
}

// ---------------------------------------------------------------- ids
__global__ void __launch_bounds__(IDS_THREADS) k_ids(Tables T, Work W) {
  constexpr int PER = IDS_CHUNK / IDS_THREADS;
  __shared__ int s_off[IDS_CHUNK];
  __shared__ int red[IDS_THREADS / 32];
  __shared__ int s_tile, s_base;
  const CallArgs A = *W.args;
  const int tid = threadIdx.x;
  if (A.n <= 0) return;
  const int64_t base = __ldg(&A.offs[0]);
  const int64_t total = __ldg(&A.offs[A.n]) - base;
  if (total > W.cap_bytes || total < 0 || base < 0) return;
  const int np = __ldcg(&W.counters[3]);
  const int nchunks = (np + IDS_CHUNK - 1) / IDS_CHUNK;
  if (tid == 0) s_tile = atomicAdd(&W.counters[1], 1);
  __syncthreads();
  const int t = s_tile;
  if (t >= nchunks) return;
  const int k0 = t * IDS_CHUNK;
  int cnt[PER];
  int sum = 0;
#pragma unroll
  for (int m = 0; m < PER; ++m) {
    const int k = k0 + tid * PER + m;
    cnt[m] = k < np ? __ldcg(&W.n_ids[k]) : 0;
    sum += cnt[m];
  }
  int chunk_total;
  const int ex = block_exclusive_scan<IDS_THREADS>(sum, [](int a, int b) { return a + b; }, 0, red, &chunk_total);
  if (tid == 0) {
    s_base = lookback(t, chunk_total, [](int a, int b) { return a + b; }, 0, W.ids_agg, W.ids_inc, W.ids_flag,
                      W.status, W.spin_limit);
    if (t == nchunks - 1) {
      W.id_off[np] = s_base + chunk_total;
      W.counters[4] = s_base + chunk_total;
    }
  }
  __syncthreads();
  int off = s_base + ex;
#pragma unroll
  for (int m = 0; m < PER; ++m) {
    const int k = k0 + tid * PER + m;
    s_off[tid * PER + m] = off;
    if (k < np) W.id_off[k] = off;
    off += cnt[m];
  }
  __syncthreads();
  for (int q = tid; q < IDS_CHUNK; q += IDS_THREADS) {
    const int k = k0 + q;
    if (k >= np) break;
    const int c = __ldcg(&W.n_ids[k]);
    const int32_t st = __ldcg(&W.piece_start[k]) & 0x7FFFFFFF;
    const int o = s_off[q];
    if (c < 0 || o < 0 || (int64_t)o + c > total || (int64_t)st + c > total) {   // never for a sound piece table
      set_status(W.status, ST_INVALID_ARG);
      continue;
    }
    for (int j = 0; j < c; ++j) A.out_ids[o + j] = __ldcg(&W.scratch[st + j]);
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

__global__ void k_req(Tables T, Work W) {
  const CallArgs A = *W.args;
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (A.n <= 0 || r > A.n) return;
  const int64_t base = __ldg(&A.offs[0]);
  const int64_t total = __ldg(&A.offs[A.n]) - base;
  if (total > W.cap_bytes || total < 0 || base < 0) { A.out_id_offsets[r] = 0; return; }
  const int np = __ldcg(&W.counters[3]);
  const int tokens = __ldcg(&W.counters[4]);
  const int k = lower_bound_piece(W.piece_start, np, __ldg(&A.offs[r]) - base);
  A.out_id_offsets[r] = k < np ? __ldcg(&W.id_off[k]) : tokens;
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
  const int64_t base = __ldg(&A.offs[0]);
  const int64_t total = __ldg(&A.offs[A.n]) - base;
  if (total > W.cap_bytes || total < 0 || base < 0) return;
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
  const int64_t base = __ldg(&A.offs[0]);
  const int64_t total = __ldg(&A.offs[A.n]) - base;
  if (total > W.cap_bytes || total < 0 || base < 0) { A.hook_offsets[r] = 0; return; }
  const int np = __ldcg(&W.counters[3]);
  const int k = lower_bound_piece(W.piece_start, np, __ldg(&A.offs[r]) - base);
  A.hook_offsets[r] = k - W.bad_pre[r];
}

void launch_bpe_small(const Tables &T, const Work &W, int grid, cudaStream_t s) {
  k_bpe_small<<<grid, BPE_SMALL_THREADS, 0, s>>>(T, W);
}
void launch_bpe_long(const Tables &T, const Work &W, int grid, cudaStream_t s) {
  k_bpe_long<<<grid, BPE_LONG_THREADS, 0, s>>>(T, W);
}
void launch_ids(const Tables &T, const Work &W, int grid, cudaStream_t s) { k_ids<<<grid, IDS_THREADS, 0, s>>>(T, W); }
void launch_req(const Tables &T, const Work &W, int grid, cudaStream_t s) { k_req<<<grid, 256, 0, s>>>(T, W); }
void launch_hook_pre(const Work &W, cudaStream_t s) { k_hook_pre<<<1, 1024, 0, s>>>(W); }
void launch_hook_pieces(const Work &W, int grid, cudaStream_t s) { k_hook_pieces<<<grid, 256, 0, s>>>(W); }
void launch_hook_offsets(const Work &W, int grid, cudaStream_t s) { k_hook_offsets<<<grid, 256, 0, s>>>(W); }

}  // namespace tt
