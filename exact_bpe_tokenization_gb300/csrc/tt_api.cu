// tt_api.cu - the C ABI of the exact BPE tokenizer (include/toktier.h):
// handle creation (vocabulary validation and device table build), per-stream
// workspaces, kernel sequencing (direct launches or a captured CUDA graph per
// stream and capacity bucket), status, the pre-tokenizer test hook and
// per-kernel timing.
//
// Design notes (TokTier: Exact Stateful CPU+GPU Tokenization for Agentic LLM
// Serving, §4.3): piece counts, dispatch lists and output lengths stay in
// device memory; kernel geometry depends on buffer capacity, not on counts,
// so the whole bytes-to-IDs chain can be captured once per size bucket and
// replayed with new buffers.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/toktier.h"
#include "tt_common.cuh"
#include "tt_kernels.h"
#include "tt_char_classes.inc"   // TT_CLASS_RANGES, TT_CLASS_RANGE_COUNT, TT_CLASS_DIGEST (generated)

using namespace tt;

namespace {

constexpr int N_KERNELS = 8;
const char *KERNEL_NAMES[N_KERNELS] = {"k_lit_find", "k_lit_pick", "k_prepass", "k_pretok",
                                       "k_bpe_warp", "k_bpe_long", "k_idscan", "k_ids"};

struct Workspace {
  Work W{};
  void *mem = nullptr;
  size_t mem_bytes = 0;
  int64_t cap_bytes = 0, cap_reqs = 0;
  cudaGraphExec_t graph = nullptr;
  cudaStream_t cap_stream = nullptr;   // private stream the graph is captured on
  cudaStream_t side = nullptr;         // second branch: block BPE of the listed huge pieces
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // device staging for tt_encode_host (bytes, offsets, ids, id offsets)
  void *stage = nullptr;
  size_t stage_bytes = 0;
  int64_t *h_offs = nullptr;       // rebased host offsets (pinned, so the copy is a plain DMA)
  size_t h_offs_cap = 0;
  DevStatus *h_status = nullptr;   // pinned: [0] the status read back, [1] the value that resets it
};

struct Pending { int kernel; cudaEvent_t a, b; };

uint64_t next_pow2(uint64_t x) {
  uint64_t p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

struct tt_tokenizer {
  int family = 0;
  int device = 0;
  Tables T{};
  std::vector<void *> dev_allocs;
  DevStatus *d_status = nullptr;
  std::mutex mu;
  // workspaces by (stream, capacity bucket): each batch size runs on the
  // geometry of its own bucket, whatever ran on the stream before
  std::map<std::pair<cudaStream_t, int64_t>, Workspace *> ws;
  std::atomic<int64_t> launches{0};
  bool profiling = false;
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> event_pool;
  double prof_ms[N_KERNELS] = {0};
  int64_t prof_n[N_KERNELS] = {0};
  bool graphs_enabled = true;
  // look-back wait settings given to every workspace (tt_debug_lookback)
  int32_t spin_limit = 1 << 22;
  int32_t withhold_tile = -1;
  // host copies of the vocabulary (rebuilt with added-token literals)
  std::vector<uint8_t> hv_bytes;
  std::vector<int64_t> hv_off;         // [n_vocab + 1], from 0
  int64_t n_vocab = 0;
  int vocab_max_len = 0;
};

// kernels of one encode: six, and the two literal kernels when the handle
// has added-token literals
static int launches_per_encode(const tt_tokenizer *h) { return 6 + (h->T.n_lit ? 2 : 0); }

#define TT_CUDA(call)                                                   \
  do {                                                                  \
    cudaError_t e_ = (call);                                            \
    if (e_ != cudaSuccess) {                                            \
      fprintf(stderr, "toktier: %s failed: %s\n", #call, cudaGetErrorString(e_)); \
      return TT_ERR_CUDA;                                               \
    }                                                                   \
  } while (0)

static tt_status upload(tt_tokenizer *h, const void *src, size_t bytes, void **dst) {
  void *p = nullptr;
  if (cudaMalloc(&p, bytes ? bytes : 16) != cudaSuccess) return TT_ERR_OOM;
  h->dev_allocs.push_back(p);
  if (bytes) TT_CUDA(cudaMemcpy(p, src, bytes, cudaMemcpyHostToDevice));
  *dst = p;
  return TT_OK;
}

// raw kind of a code point from the probed property mask
// (bits: L Lu Ll Lt Lm Lo M N \s)
static uint8_t kind_from_mask(uint32_t m) {
  if (m & 0x100) return K_WS;
  if (m & 0x080) return K_NUM;
  if (m & (0x002 | 0x008)) return K_LU;
  if (m & 0x004) return K_LL;
  if (m & (0x010 | 0x020)) return K_LB;
  if (m & 0x040) return K_MARK;
  return K_OTHER;
}

static tt_status build_class_tables(tt_tokenizer *h) {
  std::vector<uint8_t> kind(0x110000, K_OTHER);
  for (int i = 0; i < TT_CLASS_RANGE_COUNT; ++i)
    for (uint32_t c = TT_CLASS_RANGES[i][0]; c <= TT_CLASS_RANGES[i][1]; ++c) kind[c] = kind_from_mask(TT_CLASS_RANGES[i][2]);
  if (h->T.family == FAM_DEEPSEEK) {
    // the second splitter's set: Hiragana, Katakana, CJK Unified Ideographs
    for (uint32_t c = 0x3040; c <= 0x30FF; ++c) kind[c] |= K_HAN_FLAG;
    for (uint32_t c = 0x4E00; c <= 0x9FFF; ++c) kind[c] |= K_HAN_FLAG;
  }
  std::vector<uint16_t> stage1(0x110000 / 256);
  std::vector<uint8_t> stage2;
  std::map<std::string, int> seen;
  for (int blk = 0; blk < 0x110000 / 256; ++blk) {
    std::string key(reinterpret_cast<const char *>(&kind[blk * 256]), 256);
    auto it = seen.find(key);
    int idx;
    if (it == seen.end()) {
      idx = (int)seen.size();
      seen.emplace(key, idx);
      stage2.insert(stage2.end(), kind.begin() + blk * 256, kind.begin() + blk * 256 + 256);
    } else {
      idx = it->second;
    }
    stage1[blk] = (uint16_t)idx;
  }
  void *p1, *p2;
  tt_status s;
  if ((s = upload(h, stage1.data(), stage1.size() * 2, &p1)) != TT_OK) return s;
  if ((s = upload(h, stage2.data(), stage2.size(), &p2)) != TT_OK) return s;
  h->T.cls1 = (const uint16_t *)p1;
  h->T.cls2 = (const uint8_t *)p2;
  return TT_OK;
}

// Whole-piece table, token bytes and offsets for the handle's vocabulary plus
// n added-token literals (bytes lb[lo[k] .. lo[k+1]) reserved as ID ids[k],
// every ID >= n_vocab): literal IDs get their bytes at their offsets (IDs
// between them, none), and the literals enter the hash table first, so that a
// piece whose bytes are a literal -- only a literal cut out before the
// family, since any other occurrence of those bytes would have been cut out
// too -- probes to the literal's ID.
static tt_status upload_vocab(tt_tokenizer *h, const uint8_t *lb, const int64_t *lo, const int32_t *ids, int64_t n) {
  int64_t n_ids = h->n_vocab;
  for (int64_t k = 0; k < n; ++k) n_ids = std::max<int64_t>(n_ids, (int64_t)ids[k] + 1);
  std::vector<int32_t> owner((size_t)(n_ids - h->n_vocab), -1);
  for (int64_t k = 0; k < n; ++k) owner[(size_t)(ids[k] - h->n_vocab)] = (int32_t)k;
  std::vector<uint8_t> bytes = h->hv_bytes;
  std::vector<int32_t> voff((size_t)n_ids + 1);
  for (int64_t i = 0; i <= h->n_vocab; ++i) voff[(size_t)i] = (int32_t)h->hv_off[(size_t)i];
  int max_len = h->vocab_max_len;
  for (int64_t i = h->n_vocab; i < n_ids; ++i) {
    const int32_t k = owner[(size_t)(i - h->n_vocab)];
    if (k >= 0) {
      bytes.insert(bytes.end(), lb + lo[k], lb + lo[k + 1]);
      max_len = std::max<int>(max_len, (int)(lo[k + 1] - lo[k]));
    }
    voff[(size_t)i + 1] = (int32_t)bytes.size();
  }
  const uint64_t vcap = next_pow2((uint64_t)std::max<int64_t>(2 * (h->n_vocab + n), 1024));
  std::vector<uint4> vtab(vcap, make_uint4(0, 0, 0, 0));
  auto insert = [&](int64_t id) {
    const int len = voff[(size_t)id + 1] - voff[(size_t)id];
    const uint8_t *b = bytes.data() + voff[(size_t)id];
    uint64_t sl = hash_bytes(b, len) & (vcap - 1);
    while (vtab[sl].w != 0) sl = (sl + 1) & (vcap - 1);
    uint32_t e[4];
    vocab_entry(b, len, (int)id, e);
    vtab[sl] = make_uint4(e[0], e[1], e[2], e[3]);
  };
  for (int64_t k = 0; k < n; ++k) insert(ids[k]);
  for (int64_t i = 0; i < h->n_vocab; ++i) insert(i);
  void *p;
  tt_status s;
  if ((s = upload(h, vtab.data(), vtab.size() * sizeof(uint4), &p)) != TT_OK) return s;
  h->T.vocab_tab = (const uint4 *)p;
  h->T.vocab_mask = (uint32_t)(vcap - 1);
  if ((s = upload(h, bytes.data(), bytes.size(), &p)) != TT_OK) return s;
  h->T.vbytes = (const uint8_t *)p;
  if ((s = upload(h, voff.data(), voff.size() * 4, &p)) != TT_OK) return s;
  h->T.voff = (const int32_t *)p;
  h->T.max_tok_len = max_len;
  return TT_OK;
}

extern "C" tt_status tt_create(const int32_t *merge_pairs, int64_t n_merges, const uint8_t *vocab_bytes,
                               const int64_t *vocab_offsets, int64_t n_vocab, int32_t pattern_family,
                               tt_tokenizer **out) {
  if (!out) return TT_ERR_INVALID_ARG;
  *out = nullptr;
  if (pattern_family != TT_FAMILY_CL100K_STYLE && pattern_family != TT_FAMILY_O200K_STYLE &&
      pattern_family != TT_FAMILY_DEEPSEEK_STYLE)
    return TT_ERR_BAD_FAMILY;
  if (!vocab_offsets || n_vocab < 256 || n_vocab > (1 << MAX_VOCAB_BITS) || n_merges < 0 ||
      n_merges > (1 << MAX_RANK_BITS) - 1 || (n_merges > 0 && !merge_pairs))
    return n_vocab > (1 << MAX_VOCAB_BITS) || n_merges > (1 << MAX_RANK_BITS) - 1 ? TT_ERR_BAD_VOCAB : TT_ERR_INVALID_ARG;
  // ---- vocabulary
  const int64_t vbase = vocab_offsets[0];
  if (vbase < 0) return TT_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n_vocab; ++i) {
    const int64_t len = vocab_offsets[i + 1] - vocab_offsets[i];
    if (len < 1 || len > 4095) return TT_ERR_BAD_VOCAB;
  }
  const int64_t vtotal = vocab_offsets[n_vocab] - vbase;
  if (vtotal > INT32_MAX || (vtotal > 0 && !vocab_bytes)) return TT_ERR_BAD_VOCAB;
  std::unordered_map<std::string, int32_t> index;
  index.reserve((size_t)n_vocab * 2);
  int max_len = 0;
  for (int64_t i = 0; i < n_vocab; ++i) {
    const int64_t len = vocab_offsets[i + 1] - vocab_offsets[i];
    std::string key(reinterpret_cast<const char *>(vocab_bytes + vocab_offsets[i]), (size_t)len);
    if (!index.emplace(std::move(key), (int32_t)i).second) return TT_ERR_BAD_VOCAB;   // duplicate string
    if (len > max_len) max_len = (int)len;
  }
  std::vector<int32_t> byte_id(256);
  for (int b = 0; b < 256; ++b) {
    auto it = index.find(std::string(1, (char)b));
    if (it == index.end()) return TT_ERR_BAD_VOCAB;
    byte_id[b] = it->second;
  }
  // ---- merges: operands, results, duplicates, well-ordering
  std::vector<int32_t> result((size_t)n_merges);
  std::vector<int64_t> creator((size_t)n_vocab, -1);
  std::unordered_map<uint64_t, int64_t> pairs;
  pairs.reserve((size_t)n_merges * 2);
  for (int64_t k = 0; k < n_merges; ++k) {
    const int32_t l = merge_pairs[2 * k], r = merge_pairs[2 * k + 1];
    if (l < 0 || r < 0 || l >= n_vocab || r >= n_vocab) return TT_ERR_BAD_VOCAB;
    std::string cat(reinterpret_cast<const char *>(vocab_bytes + vocab_offsets[l]),
                    (size_t)(vocab_offsets[l + 1] - vocab_offsets[l]));
    cat.append(reinterpret_cast<const char *>(vocab_bytes + vocab_offsets[r]),
               (size_t)(vocab_offsets[r + 1] - vocab_offsets[r]));
    auto it = index.find(cat);
    if (it == index.end()) return TT_ERR_BAD_VOCAB;
    result[k] = it->second;
    if (!pairs.emplace(pair_key((uint32_t)l, (uint32_t)r), k).second) return TT_ERR_BAD_VOCAB;
    if (creator[result[k]] >= 0) return TT_ERR_BAD_VOCAB;                 // two merges, one result
    creator[result[k]] = k;
  }
  for (int64_t k = 0; k < n_merges; ++k) {
    const int32_t ops[2] = {merge_pairs[2 * k], merge_pairs[2 * k + 1]};
    for (int32_t x : ops)
      if (creator[x] >= k) return TT_ERR_BAD_VOCAB;                        // used before it is made
  }

  tt_tokenizer *h = new tt_tokenizer();
  h->family = pattern_family;
  cudaGetDevice(&h->device);
  tt_status s;
  auto fail = [&](tt_status st) { tt_destroy(h); return st; };
  if (pretok_configure() != cudaSuccess) return fail(TT_ERR_CUDA);
  if (bpe_configure() != cudaSuccess) return fail(TT_ERR_CUDA);
  // ---- pair table: load factor <= 1/8, so that the lookups of pairs that
  // are not merges (most of them) end after about one probe
  const uint64_t pcap = next_pow2((uint64_t)std::max<int64_t>(8 * n_merges, 1024));
  std::vector<uint4> ptab(pcap, make_uint4(PAIR_EMPTY, PAIR_EMPTY, 0xFFFFFFFFu, 0xFFFFFFFFu));
  for (int64_t k = 0; k < n_merges; ++k) {
    const uint32_t l = (uint32_t)merge_pairs[2 * k], r = (uint32_t)merge_pairs[2 * k + 1];
    uint64_t sl = pair_hash(l, r) & (pcap - 1);
    while (ptab[sl].x != PAIR_EMPTY) sl = (sl + 1) & (pcap - 1);
    ptab[sl] = make_uint4(l, r, (uint32_t)k, (uint32_t)result[k]);
  }
  h->n_vocab = n_vocab;
  h->vocab_max_len = max_len;
  h->hv_bytes.assign(vocab_bytes + vbase, vocab_bytes + vbase + vtotal);
  h->hv_off.resize((size_t)n_vocab + 1);
  for (int64_t i = 0; i <= n_vocab; ++i) h->hv_off[i] = vocab_offsets[i] - vbase;
  void *p;
  if ((s = upload(h, ptab.data(), ptab.size() * sizeof(uint4), &p)) != TT_OK) return fail(s);
  h->T.pair_tab = (const uint4 *)p;
  h->T.pair_mask = (uint32_t)(pcap - 1);
  if ((s = upload(h, result.data(), result.size() * 4, &p)) != TT_OK) return fail(s);
  h->T.merge_result = (const int32_t *)p;
  // ---- context table: per (token, side, byte) the lowest rank of a merge
  // that can take the token from that side (load factor <= 1/4)
  {
    std::unordered_map<uint32_t, uint32_t> lowest;
    lowest.reserve((size_t)n_merges * 2);
    for (int64_t k = 0; k < n_merges; ++k) {
      const uint32_t l = (uint32_t)merge_pairs[2 * k], r = (uint32_t)merge_pairs[2 * k + 1];
      const uint8_t last_l = vocab_bytes[vocab_offsets[l + 1] - 1], first_r = vocab_bytes[vocab_offsets[r]];
      lowest.emplace(ctx_key(r, 0, last_l), (uint32_t)k);    // ranks ascend with k: the first is the lowest
      lowest.emplace(ctx_key(l, 1, first_r), (uint32_t)k);
    }
    const uint64_t ccap = next_pow2((uint64_t)std::max<size_t>(4 * lowest.size(), 1024));
    std::vector<uint2> ctab(ccap, make_uint2(CTX_EMPTY, 0));
    for (const auto &kv : lowest) {
      uint64_t sl = ctx_hash(kv.first) & (ccap - 1);
      while (ctab[sl].x != CTX_EMPTY) sl = (sl + 1) & (ccap - 1);
      ctab[sl] = make_uint2(kv.first, kv.second);
    }
    if ((s = upload(h, ctab.data(), ctab.size() * sizeof(uint2), &p)) != TT_OK) return fail(s);
    h->T.ctx_tab = (const uint2 *)p;
    h->T.ctx_mask = (uint32_t)(ccap - 1);
    // the byte tokens' pairs and context entries, indexed directly
    std::vector<int2> bpair(65536, make_int2(-1, -1));
    std::vector<int32_t> bctx(2 * 65536, INT32_MAX);
    for (int b0 = 0; b0 < 256; ++b0) {
      for (int b1 = 0; b1 < 256; ++b1) {
        auto it = pairs.find(pair_key((uint32_t)byte_id[b0], (uint32_t)byte_id[b1]));
        if (it != pairs.end()) bpair[b0 << 8 | b1] = make_int2((int)it->second, result[it->second]);
        for (uint32_t side = 0; side < 2; ++side) {
          auto jt = lowest.find(ctx_key((uint32_t)byte_id[b0], side, (uint32_t)b1));
          if (jt != lowest.end()) bctx[side << 16 | b0 << 8 | b1] = (int32_t)jt->second;
        }
      }
    }
    if ((s = upload(h, bpair.data(), bpair.size() * sizeof(int2), &p)) != TT_OK) return fail(s);
    h->T.bpair = (const int2 *)p;
    if ((s = upload(h, bctx.data(), bctx.size() * sizeof(int32_t), &p)) != TT_OK) return fail(s);
    h->T.bctx = (const int32_t *)p;
  }
  if ((s = upload_vocab(h, nullptr, nullptr, nullptr, 0)) != TT_OK) return fail(s);
  if ((s = upload(h, byte_id.data(), 256 * 4, &p)) != TT_OK) return fail(s);
  h->T.byte_id = (const int32_t *)p;
  h->T.family = pattern_family;
  if ((s = build_class_tables(h)) != TT_OK) return fail(s);
  DevStatus init = {0, 0, ~0ull};
  if ((s = upload(h, &init, sizeof(init), &p)) != TT_OK) return fail(s);
  h->d_status = (DevStatus *)p;
  const char *env = getenv("TOKTIER_NO_GRAPHS");
  if (env && env[0] == '1') h->graphs_enabled = false;
  *out = h;
  return TT_OK;
}

// strict UTF-8 (RFC 3629): no overlongs, surrogates or code points past U+10FFFF
static bool valid_utf8(const uint8_t *b, int64_t n) {
  for (int64_t i = 0; i < n;) {
    const uint8_t c = b[i];
    int len;
    uint32_t cp;
    if (c < 0x80) { ++i; continue; }
    if (c >= 0xC2 && c <= 0xDF) { len = 2; cp = c & 0x1F; }
    else if (c >= 0xE0 && c <= 0xEF) { len = 3; cp = c & 0x0F; }
    else if (c >= 0xF0 && c <= 0xF4) { len = 4; cp = c & 0x07; }
    else return false;
    if (i + len > n) return false;
    for (int q = 1; q < len; ++q) {
      if ((b[i + q] & 0xC0) != 0x80) return false;
      cp = (cp << 6) | (b[i + q] & 0x3F);
    }
    if ((len == 3 && cp < 0x800) || (len == 4 && (cp < 0x10000 || cp > 0x10FFFF)) || (cp >= 0xD800 && cp <= 0xDFFF))
      return false;
    i += len;
  }
  return true;
}

static void free_workspace(Workspace *w);

extern "C" tt_status tt_set_added_tokens(tt_tokenizer *h, const uint8_t *literal_bytes, const int64_t *literal_offsets,
                                         const int32_t *literal_ids, int64_t n_literals) {
  if (!h || n_literals < 0) return TT_ERR_INVALID_ARG;
  if (n_literals > LIT_MAX_COUNT) return TT_ERR_BAD_VOCAB;
  if (n_literals > 0 && (!literal_bytes || !literal_offsets || !literal_ids)) return TT_ERR_INVALID_ARG;
  std::vector<int64_t> lo((size_t)n_literals + 1, 0);
  std::unordered_map<std::string, int64_t> strings;
  std::unordered_map<int32_t, int64_t> used;
  for (int64_t k = 0; k < n_literals; ++k) {
    const int64_t len = literal_offsets[k + 1] - literal_offsets[k];
    if (len < 1 || len > LIT_MAX_LEN || literal_offsets[k] < literal_offsets[0]) return TT_ERR_BAD_VOCAB;
    const uint8_t *b = literal_bytes + literal_offsets[k];
    if (!valid_utf8(b, len)) return TT_ERR_BAD_VOCAB;
    const int32_t id = literal_ids[k];
    if (id < h->n_vocab || id >= (1 << MAX_VOCAB_BITS)) return TT_ERR_BAD_VOCAB;
    if (!strings.emplace(std::string(reinterpret_cast<const char *>(b), (size_t)len), k).second) return TT_ERR_BAD_VOCAB;
    if (!used.emplace(id, k).second) return TT_ERR_BAD_VOCAB;
    lo[(size_t)k + 1] = lo[(size_t)k] + len;
  }
  std::lock_guard<std::mutex> lock(h->mu);
  // literal tables: bytes, offsets, and an order by (first byte, length
  // descending) with the range of each first byte
  std::vector<uint8_t> lb((size_t)std::max<int64_t>(lo[(size_t)n_literals], 1));
  std::vector<int32_t> loff32((size_t)n_literals + 1), order((size_t)std::max<int64_t>(n_literals, 1)), first(257, 0);
  for (int64_t k = 0; k < n_literals; ++k) {
    memcpy(lb.data() + lo[(size_t)k], literal_bytes + literal_offsets[k], (size_t)(lo[(size_t)k + 1] - lo[(size_t)k]));
    loff32[(size_t)k + 1] = (int32_t)lo[(size_t)k + 1];
    order[(size_t)k] = (int32_t)k;
  }
  std::sort(order.begin(), order.begin() + n_literals, [&](int32_t a, int32_t b) {
    const uint8_t fa = lb[(size_t)lo[(size_t)a]], fb = lb[(size_t)lo[(size_t)b]];
    if (fa != fb) return fa < fb;
    return lo[(size_t)a + 1] - lo[(size_t)a] > lo[(size_t)b + 1] - lo[(size_t)b];
  });
  for (int64_t k = 0; k < n_literals; ++k) first[lb[(size_t)lo[(size_t)order[(size_t)k]]] + 1] += 1;
  for (int c = 0; c < 256; ++c) first[(size_t)c + 1] += first[(size_t)c];
  tt_status s;
  void *p;
  if ((s = upload(h, lb.data(), lb.size(), &p)) != TT_OK) return s;
  h->T.lit_bytes = (const uint8_t *)p;
  if ((s = upload(h, loff32.data(), loff32.size() * 4, &p)) != TT_OK) return s;
  h->T.lit_off = (const int32_t *)p;
  if ((s = upload(h, order.data(), order.size() * 4, &p)) != TT_OK) return s;
  h->T.lit_order = (const int32_t *)p;
  if ((s = upload(h, first.data(), first.size() * 4, &p)) != TT_OK) return s;
  h->T.lit_first = (const int32_t *)p;
  if ((s = upload_vocab(h, lb.data(), lo.data(), literal_ids, n_literals)) != TT_OK) return s;
  h->T.n_lit = (int32_t)n_literals;
  // captured graphs hold the old tables and kernel sequence
  for (auto &kv : h->ws)
    if (kv.second->graph) {
      cudaGraphExecDestroy(kv.second->graph);
      kv.second->graph = nullptr;
    }
  return TT_OK;
}

static void free_workspace(Workspace *w) {
  if (!w) return;
  if (w->graph) cudaGraphExecDestroy(w->graph);
  if (w->cap_stream) cudaStreamDestroy(w->cap_stream);
  if (w->side) cudaStreamDestroy(w->side);
  if (w->ev_fork) cudaEventDestroy(w->ev_fork);
  if (w->ev_join) cudaEventDestroy(w->ev_join);
  if (w->mem) cudaFree(w->mem);
  if (w->stage) cudaFree(w->stage);
  if (w->h_offs) cudaFreeHost(w->h_offs);
  if (w->h_status) cudaFreeHost(w->h_status);
  delete w;
}

extern "C" void tt_destroy(tt_tokenizer *h) {
  if (!h) return;
  cudaDeviceSynchronize();
  for (auto &kv : h->ws) free_workspace(kv.second);
  for (auto &pd : h->pending) { cudaEventDestroy(pd.a); cudaEventDestroy(pd.b); }
  for (cudaEvent_t e : h->event_pool) cudaEventDestroy(e);
  for (void *p : h->dev_allocs) cudaFree(p);
  delete h;
}

// Carve the workspace of one capacity bucket out of one allocation.
static tt_status make_workspace(tt_tokenizer *h, int64_t cap_bytes, int64_t cap_reqs, Workspace **out) {
  Workspace *w = new Workspace();
  w->cap_bytes = cap_bytes;
  w->cap_reqs = cap_reqs;
  const int64_t tiles = (cap_bytes + TILE - 1) / TILE + 1;
  const int64_t chunks = (cap_bytes + 1 + IDS_CHUNK - 1) / IDS_CHUNK + 2;
  struct Item { void **dst; size_t bytes; };
  Work &W = w->W;
  std::vector<Item> items = {
      {(void **)&W.s1_sum, sizeof(int2) * tiles},       {(void **)&W.rq_sum, 2 * (size_t)tiles},
      {(void **)&W.s2_agg, sizeof(S2) * tiles},         {(void **)&W.s2_inc, sizeof(S2) * tiles},
      {(void **)&W.s2_flag, 4 * (size_t)tiles},         {(void **)&W.cnt_agg, sizeof(int2) * tiles},
      {(void **)&W.cnt_inc, sizeof(int2) * tiles},      {(void **)&W.cnt_flag, 4 * (size_t)tiles},
      {(void **)&W.ids_agg, 4 * (size_t)chunks},        {(void **)&W.ids_inc, 4 * (size_t)chunks},
      {(void **)&W.counters, 4 * 16},
      {(void **)&W.piece_start, 4 * (size_t)(cap_bytes + 2)}, {(void **)&W.n_ids, 4 * (size_t)(cap_bytes + 1)},
      {(void **)&W.scratch, 4 * (size_t)(cap_bytes + 1)},
      {(void **)&W.tmp_a, 4 * (size_t)(cap_bytes + 1)},       {(void **)&W.tmp_b, 4 * (size_t)(cap_bytes + 1)},
      {(void **)&W.tmp_c, 4 * (size_t)(cap_bytes + 1)},
      {(void **)&W.long_list, 4 * 3 * (size_t)list_cap(cap_bytes)},
      {(void **)&W.huge_list, 4 * (size_t)(cap_bytes / (MID_MAX + 1) + 2)},
      {(void **)&W.bad, (size_t)cap_reqs + 1},          {(void **)&W.bad_pre, 4 * (size_t)(cap_reqs + 2)},
      {(void **)&W.req_piece, 4 * (size_t)(cap_reqs + 1)},
      {(void **)&W.lit_cand, 4 * (size_t)tiles * TILE}, {(void **)&W.lit_cnt, 4 * (size_t)tiles},
      {(void **)&W.lit_flag, (size_t)cap_bytes + 8},   {(void **)&W.lit_len, (size_t)cap_bytes + 8},
      {(void **)&W.args, sizeof(CallArgs)},
  };
  size_t total = 0;
  for (auto &it : items) total += (it.bytes + 255) & ~(size_t)255;
  if (cudaMalloc(&w->mem, total) != cudaSuccess) { delete w; return TT_ERR_OOM; }
  w->mem_bytes = total;
  size_t off = 0;
  for (auto &it : items) {
    *it.dst = (char *)w->mem + off;
    off += (it.bytes + 255) & ~(size_t)255;
  }
  W.cap_bytes = cap_bytes;
  W.cap_reqs = cap_reqs;
  W.cap_tiles = (int32_t)tiles;
  W.spin_limit = h->spin_limit;
  W.withhold_tile = h->withhold_tile;
  W.status = h->d_status;
  if (cudaMemset(w->mem, 0, total) != cudaSuccess) { free_workspace(w); return TT_ERR_CUDA; }
  *out = w;
  return TT_OK;
}

// The workspace of `stream`, grown to hold (bytes, reqs).  Caller holds h->mu.
// Capacities are powers of two (>= 64 KiB, >= 64 requests) so that a stream
// sees few distinct buckets; growing drops the old bucket and its graph.
static tt_status get_workspace(tt_tokenizer *h, cudaStream_t stream, int64_t bytes, int64_t reqs, Workspace **out) {
  const int64_t cb = (int64_t)next_pow2((uint64_t)std::max<int64_t>(bytes, 1 << 16));
  int64_t cr = (int64_t)next_pow2((uint64_t)std::max<int64_t>(reqs, 64));
  const auto key = std::make_pair(stream, cb);
  auto it = h->ws.find(key);
  if (it != h->ws.end()) {
    Workspace *old = it->second;
    if (old->cap_reqs >= cr) {
      *out = old;
      return TT_OK;
    }
    cr = std::max(cr, old->cap_reqs);          // more requests than before: rebuild this bucket
    cudaStreamSynchronize(stream);
    free_workspace(old);
    h->ws.erase(it);
  }
  Workspace *w;
  tt_status s = make_workspace(h, cb, cr, &w);
  if (s != TT_OK) return s;
  h->ws[key] = w;
  *out = w;
  return TT_OK;
}

static cudaEvent_t pool_event(tt_tokenizer *h) {
  if (!h->event_pool.empty()) {
    cudaEvent_t e = h->event_pool.back();
    h->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e;
  cudaEventCreate(&e);
  return e;
}

// grid sizes, all from capacity
static int grid_tiles(const Workspace *w) { return (int)((w->cap_bytes + TILE - 1) / TILE); }
static int grid_reqs(const Workspace *w) { return (int)((w->cap_reqs + 1 + 255) / 256); }
static int grid_chunks(const Workspace *w) {   // CTAs striding over the 512-piece ID chunks
  const int64_t g = (w->cap_bytes + 1 + IDS_CHUNK - 1) / IDS_CHUNK;
  // at 32 registers 8 CTAs fit an SM: fewer chunks a CTA in turn hide more of
  // each chunk's latency in batches (burst 0.047 -> 0.039 ms); workspaces of
  // up to 4 MiB hold too few chunks to fill even 5 a SM (the extra CTAs only
  // cost launch time: 1M-char request 0.0125 -> 0.0143 ms)
  const int per_sm = w->cap_bytes > (4ll << 20) ? 8 : 5;
  return (int)std::min<int64_t>(std::max<int64_t>(g, 1), 152 * per_sm);
}
static int grid_pieces(const Workspace *w) {   // a thread per piece (test hook)
  const int64_t g = (w->cap_bytes / 4 + 255) / 256;
  return (int)std::min<int64_t>(std::max<int64_t>(g, 1), 152 * 8);
}
// persistent warps taking tickets: all resident at once, fewer for small
// workspaces
static int64_t warp_grid(int64_t cap_bytes) {
  const int64_t warps = cap_bytes / 128 + 1;   // about one ticket per 128 bytes
  const int64_t g = (warps + BPE_WARP_THREADS / 32 - 1) / (BPE_WARP_THREADS / 32);
  return std::min<int64_t>(std::max<int64_t>(g, 1), 152 * BPE_WARP_CTAS_PER_SM);
}
static int grid_warp(const Workspace *w) { return (int)warp_grid(w->cap_bytes); }
static int grid_lit_pick(const Workspace *w) {   // a warp per tile
  return (int)std::min<int64_t>((grid_tiles(w) + 7) / 8, 152 * 8);
}
static int grid_long(const Workspace *w) {
  return (int)std::min<int64_t>(std::max<int64_t>(w->cap_bytes / (MID_MAX + 1), 1), 152 * 2);
}

// Enqueue the kernels of one encode on `stream`.  Untimed, the BPE of the
// huge pieces (k_bpe_long) runs on a second stream beside the warp kernel
// (k_bpe_warp, every other piece), forked after k_pretok and joined before
// k_idscan; under capture these become two parallel graph branches.  Timed
// (profiling), every kernel runs in turn on `stream` between events.
static tt_status enqueue_encode(tt_tokenizer *h, Workspace *w, cudaStream_t stream, bool timed) {
  const Tables &T = h->T;
  const Work &W = w->W;
  TT_CUDA(cudaMemsetAsync(W.counters, 0, 4 * 16, stream));
  TT_CUDA(cudaMemsetAsync(W.bad, 0, (size_t)w->cap_reqs + 1, stream));
  if (T.n_lit) TT_CUDA(cudaMemsetAsync(W.lit_flag, 0, (size_t)w->cap_bytes + 8, stream));
  if (!timed) {
    if (!w->side) TT_CUDA(cudaStreamCreateWithFlags(&w->side, cudaStreamNonBlocking));
    if (!w->ev_fork) TT_CUDA(cudaEventCreateWithFlags(&w->ev_fork, cudaEventDisableTiming));
    if (!w->ev_join) TT_CUDA(cudaEventCreateWithFlags(&w->ev_join, cudaEventDisableTiming));
    if (T.n_lit) {
      launch_lit_find(T, W, grid_tiles(w), stream);
      launch_lit_pick(T, W, grid_lit_pick(w), stream);
    }
    launch_prepass(T, W, grid_tiles(w), stream);
    launch_pretok(T, W, grid_tiles(w), stream);
    TT_CUDA(cudaEventRecord(w->ev_fork, stream));
    TT_CUDA(cudaStreamWaitEvent(w->side, w->ev_fork, 0));
    launch_bpe_long(T, W, grid_long(w), w->side);
    TT_CUDA(cudaEventRecord(w->ev_join, w->side));
    launch_bpe_warp(T, W, grid_warp(w), stream);
    TT_CUDA(cudaStreamWaitEvent(stream, w->ev_join, 0));
    launch_idscan(W, stream);
    launch_ids(T, W, grid_chunks(w), stream);
    TT_CUDA(cudaGetLastError());
    h->launches += launches_per_encode(h);
    return TT_OK;
  }
  for (int kidx = T.n_lit ? 0 : 2; kidx < N_KERNELS; ++kidx) {
    cudaEvent_t a = pool_event(h), b = pool_event(h);
    cudaEventRecord(a, stream);
    switch (kidx) {
      case 0: launch_lit_find(T, W, grid_tiles(w), stream); break;
      case 1: launch_lit_pick(T, W, grid_lit_pick(w), stream); break;
      case 2: launch_prepass(T, W, grid_tiles(w), stream); break;
      case 3: launch_pretok(T, W, grid_tiles(w), stream); break;
      case 4: launch_bpe_warp(T, W, grid_warp(w), stream); break;
      case 5: launch_bpe_long(T, W, grid_long(w), stream); break;
      case 6: launch_idscan(W, stream); break;
      case 7: launch_ids(T, W, grid_chunks(w), stream); break;
    }
    cudaEventRecord(b, stream);
    h->pending.push_back({kidx, a, b});
  }
  TT_CUDA(cudaGetLastError());
  h->launches += launches_per_encode(h);
  return TT_OK;
}

static tt_status check_batch_args(tt_tokenizer *h, const void *d_utf8, const int64_t *offs, int64_t n,
                                  const void *out_ids, const int64_t *out_offs, int64_t max_bytes) {
  if (!h || n < 0 || !offs || !out_offs) return TT_ERR_INVALID_ARG;
  if (n > 0 && max_bytes != 0 && (!d_utf8 || !out_ids)) return TT_ERR_INVALID_ARG;
  return TT_OK;
}

static tt_status encode_bounded(tt_tokenizer *h, const uint8_t *d_utf8, const int64_t *d_byte_offsets,
                                int64_t n_requests, int64_t max_total_bytes, int32_t *d_out_ids,
                                int64_t *d_out_id_offsets, int32_t *d_out_spans, tt_stream_t stream_,
                                const uint8_t *src = nullptr) {
  tt_status s = check_batch_args(h, d_utf8, d_byte_offsets, n_requests, d_out_ids, d_out_id_offsets, max_total_bytes);
  if (s != TT_OK) return s;
  if (max_total_bytes < 0 || max_total_bytes >= S2_MAX_POS - 64) return TT_ERR_CAPACITY;
  cudaStream_t stream = (cudaStream_t)stream_;
  if (n_requests == 0) {
    TT_CUDA(cudaMemsetAsync(d_out_id_offsets, 0, sizeof(int64_t), stream));
    return TT_OK;
  }
  std::lock_guard<std::mutex> lock(h->mu);
  Workspace *w;
  if ((s = get_workspace(h, stream, max_total_bytes, n_requests, &w)) != TT_OK) return s;
  CallArgs args = {d_utf8, d_byte_offsets, n_requests, d_out_ids, d_out_id_offsets, nullptr, nullptr, d_out_spans, src,
                   max_total_bytes};
  TT_CUDA(cudaMemcpyAsync(w->W.args, &args, sizeof(args), cudaMemcpyHostToDevice, stream));
  if (h->profiling || !h->graphs_enabled) return enqueue_encode(h, w, stream, h->profiling);
  if (!w->graph) {
    // capture on a private stream (the caller's may be the legacy default
    // stream, which cannot be captured); the graph is launched on the caller's
    if (!w->cap_stream) TT_CUDA(cudaStreamCreateWithFlags(&w->cap_stream, cudaStreamNonBlocking));
    cudaGraph_t g;
    TT_CUDA(cudaStreamBeginCapture(w->cap_stream, cudaStreamCaptureModeThreadLocal));
    tt_status es = enqueue_encode(h, w, w->cap_stream, false);
    cudaError_t ce = cudaStreamEndCapture(w->cap_stream, &g);
    h->launches -= launches_per_encode(h);   // captured, not launched
    if (es != TT_OK) return es;
    TT_CUDA(ce);
    cudaError_t ie = cudaGraphInstantiate(&w->graph, g, 0);
    cudaGraphDestroy(g);
    TT_CUDA(ie);
  }
  TT_CUDA(cudaGraphLaunch(w->graph, stream));
  h->launches += launches_per_encode(h);
  return TT_OK;
}

extern "C" tt_status tt_encode_batch_bounded(tt_tokenizer *h, const uint8_t *d_utf8, const int64_t *d_byte_offsets,
                                             int64_t n_requests, int64_t max_total_bytes, int32_t *d_out_ids,
                                             int64_t *d_out_id_offsets, tt_stream_t stream) {
  return encode_bounded(h, d_utf8, d_byte_offsets, n_requests, max_total_bytes, d_out_ids, d_out_id_offsets, nullptr,
                        stream);
}

extern "C" tt_status tt_encode_batch_spans(tt_tokenizer *h, const uint8_t *d_utf8, const int64_t *d_byte_offsets,
                                           int64_t n_requests, int64_t max_total_bytes, int32_t *d_out_ids,
                                           int64_t *d_out_id_offsets, int32_t *d_out_spans, tt_stream_t stream) {
  if (!d_out_spans && n_requests > 0 && max_total_bytes > 0) return TT_ERR_INVALID_ARG;
  return encode_bounded(h, d_utf8, d_byte_offsets, n_requests, max_total_bytes, d_out_ids, d_out_id_offsets,
                        d_out_spans, stream);
}

extern "C" tt_status tt_encode_batch(tt_tokenizer *h, const uint8_t *d_utf8, const int64_t *d_byte_offsets,
                                     int64_t n_requests, int32_t *d_out_ids, int64_t *d_out_id_offsets,
                                     tt_stream_t stream_) {
  tt_status s = check_batch_args(h, d_utf8, d_byte_offsets, n_requests, d_out_ids, d_out_id_offsets, 0);
  if (s != TT_OK) return s;
  cudaStream_t stream = (cudaStream_t)stream_;
  if (n_requests == 0) {
    TT_CUDA(cudaMemsetAsync(d_out_id_offsets, 0, sizeof(int64_t), stream));
    return TT_OK;
  }
  int64_t ends[2];
  TT_CUDA(cudaMemcpyAsync(&ends[0], d_byte_offsets, 8, cudaMemcpyDeviceToHost, stream));
  TT_CUDA(cudaMemcpyAsync(&ends[1], d_byte_offsets + n_requests, 8, cudaMemcpyDeviceToHost, stream));
  TT_CUDA(cudaStreamSynchronize(stream));
  if (ends[0] < 0 || ends[1] < ends[0]) return TT_ERR_INVALID_ARG;
  if (ends[1] > ends[0] && (!d_utf8 || !d_out_ids)) return TT_ERR_INVALID_ARG;
  return tt_encode_batch_bounded(h, d_utf8, d_byte_offsets, n_requests, ends[1] - ends[0], d_out_ids,
                                 d_out_id_offsets, stream_);
}

extern "C" tt_status tt_get_status(tt_tokenizer *h, tt_stream_t stream, int64_t *bad_request) {
  if (!h) return TT_ERR_INVALID_ARG;
  TT_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  DevStatus st;
  TT_CUDA(cudaMemcpy(&st, h->d_status, sizeof(st), cudaMemcpyDeviceToHost));
  DevStatus init = {0, 0, ~0ull};
  TT_CUDA(cudaMemcpy(h->d_status, &init, sizeof(init), cudaMemcpyHostToDevice));
  if (bad_request) *bad_request = st.code == ST_INVALID_UTF8 && st.bad_request != ~0ull ? (int64_t)st.bad_request : -1;
  return (tt_status)st.code;
}

// Device address of a page-locked or managed host buffer, or null for
// ordinary pageable memory.
static void *device_view(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if ((a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeManaged) && a.devicePointer) return a.devicePointer;
  return nullptr;
}

// Enqueue the read-back and reset of the handle's status word into the
// workspace's pinned pair (the caller waits for the stream, then calls
// status_result).
static tt_status enqueue_status_read(tt_tokenizer *h, Workspace *w, cudaStream_t stream) {
  if (!w->h_status) {
    if (cudaMallocHost(&w->h_status, 2 * sizeof(DevStatus)) != cudaSuccess) { w->h_status = nullptr; return TT_ERR_OOM; }
    w->h_status[1] = DevStatus{0, 0, ~0ull};
  }
  TT_CUDA(cudaMemcpyAsync(&w->h_status[0], h->d_status, sizeof(DevStatus), cudaMemcpyDeviceToHost, stream));
  TT_CUDA(cudaMemcpyAsync(h->d_status, &w->h_status[1], sizeof(DevStatus), cudaMemcpyHostToDevice, stream));
  return TT_OK;
}
static tt_status status_result(const Workspace *w) { return (tt_status)w->h_status[0].code; }

extern "C" tt_status tt_encode_host(tt_tokenizer *h, const uint8_t *utf8, const int64_t *byte_offsets,
                                    int64_t n_requests, int32_t *out_ids, int64_t out_capacity,
                                    int64_t *out_id_offsets, tt_stream_t stream_) {
  if (!h || n_requests < 0 || !byte_offsets || !out_id_offsets || out_capacity < 0) return TT_ERR_INVALID_ARG;
  if (n_requests == 0) { out_id_offsets[0] = 0; return TT_OK; }
  const int64_t b0 = byte_offsets[0], b1 = byte_offsets[n_requests];
  if (b0 < 0 || b1 < b0 || (b1 > b0 && (!utf8 || !out_ids))) return TT_ERR_INVALID_ARG;
  for (int64_t r = 0; r < n_requests; ++r)
    if (byte_offsets[r] > byte_offsets[r + 1]) return TT_ERR_INVALID_ARG;
  const int64_t total = b1 - b0;
  if (total >= S2_MAX_POS - 64) return TT_ERR_CAPACITY;
  cudaStream_t stream = (cudaStream_t)stream_;
  // Page-locked output buffers with room for the worst case are written by
  // the kernels directly (no copy back, one wait); anything else is staged.
  int32_t *dv_ids = nullptr;
  int64_t *dv_offs = nullptr;
  if (total > 0 && out_capacity >= total) {
    dv_ids = (int32_t *)device_view(out_ids);
    dv_offs = dv_ids ? (int64_t *)device_view(out_id_offsets) : nullptr;
  }
  const bool direct = dv_ids && dv_offs;
  // page-locked input is read in place by the pre-pass, which copies it to
  // the device tile by tile (not with added-token literals: their search runs
  // before the pre-pass)
  const uint8_t *dv_in = total > 0 && !h->T.n_lit ? (const uint8_t *)device_view(utf8 + b0) : nullptr;
  const size_t in_b = ((size_t)total + 16 + 255) & ~(size_t)255;
  const size_t off_b = ((size_t)(n_requests + 1) * 8 + 255) & ~(size_t)255;
  const size_t out_b = direct ? 0 : ((size_t)total + 1) * 4;
  uint8_t *d_in;
  int64_t *d_offs, *d_out_offs;
  int32_t *d_out;
  Workspace *w;
  {
    std::lock_guard<std::mutex> lock(h->mu);
    tt_status s = get_workspace(h, stream, total, n_requests, &w);
    if (s != TT_OK) return s;
    const size_t need = in_b + 2 * off_b + out_b;
    if (w->stage_bytes < need) {
      if (w->stage) { cudaStreamSynchronize(stream); cudaFree(w->stage); w->stage = nullptr; w->stage_bytes = 0; }
      const size_t sz = next_pow2(need);
      if (cudaMalloc(&w->stage, sz) != cudaSuccess) return TT_ERR_OOM;
      w->stage_bytes = sz;
    }
    char *cur = (char *)w->stage;
    d_in = (uint8_t *)cur;
    d_offs = (int64_t *)(cur + in_b);
    d_out_offs = direct ? dv_offs : (int64_t *)(cur + in_b + off_b);
    d_out = direct ? dv_ids : (int32_t *)(cur + in_b + 2 * off_b);
    // (the previous call on this stream has waited for its copies, so the
    // staging buffer is free to overwrite)
    if (w->h_offs_cap < (size_t)n_requests + 1) {
      if (w->h_offs) { cudaFreeHost(w->h_offs); w->h_offs = nullptr; w->h_offs_cap = 0; }
      const size_t cap = next_pow2((uint64_t)n_requests + 1);
      if (cudaMallocHost(&w->h_offs, cap * sizeof(int64_t)) != cudaSuccess) { w->h_offs = nullptr; return TT_ERR_OOM; }
      w->h_offs_cap = cap;
    }
    for (int64_t r = 0; r <= n_requests; ++r) w->h_offs[r] = byte_offsets[r] - b0;
    if (total && !dv_in) TT_CUDA(cudaMemcpyAsync(d_in, utf8 + b0, (size_t)total, cudaMemcpyHostToDevice, stream));
    TT_CUDA(cudaMemcpyAsync(d_offs, w->h_offs, (size_t)(n_requests + 1) * 8, cudaMemcpyHostToDevice, stream));
  }
  tt_status s = encode_bounded(h, d_in, d_offs, n_requests, total, d_out, d_out_offs, nullptr, stream_, dv_in);
  if (s == TT_OK) s = enqueue_status_read(h, w, stream);
  if (s != TT_OK) {
    cudaStreamSynchronize(stream);   // the staged copies are done before the buffers are reused
    return s;
  }
  if (!direct) TT_CUDA(cudaMemcpyAsync(out_id_offsets, d_out_offs, (size_t)(n_requests + 1) * 8, cudaMemcpyDeviceToHost,
                                       stream));
  TT_CUDA(cudaStreamSynchronize(stream));
  if (direct) return status_result(w);
  const int64_t ntok = out_id_offsets[n_requests];
  if (ntok > out_capacity) return TT_ERR_CAPACITY;
  if (ntok) {
    TT_CUDA(cudaMemcpyAsync(out_ids, d_out, (size_t)ntok * 4, cudaMemcpyDeviceToHost, stream));
    TT_CUDA(cudaStreamSynchronize(stream));
  }
  return status_result(w);
}

extern "C" tt_status tt_pretokenize_batch(tt_tokenizer *h, const uint8_t *d_utf8, const int64_t *d_byte_offsets,
                                          int64_t n_requests, int64_t *d_piece_starts, int64_t *d_piece_offsets,
                                          tt_stream_t stream_) {
  tt_status s = check_batch_args(h, d_utf8, d_byte_offsets, n_requests, d_piece_starts, d_piece_offsets, 0);
  if (s != TT_OK) return s;
  cudaStream_t stream = (cudaStream_t)stream_;
  if (n_requests == 0) {
    TT_CUDA(cudaMemsetAsync(d_piece_offsets, 0, sizeof(int64_t), stream));
    return TT_OK;
  }
  int64_t ends[2];
  TT_CUDA(cudaMemcpyAsync(&ends[0], d_byte_offsets, 8, cudaMemcpyDeviceToHost, stream));
  TT_CUDA(cudaMemcpyAsync(&ends[1], d_byte_offsets + n_requests, 8, cudaMemcpyDeviceToHost, stream));
  TT_CUDA(cudaStreamSynchronize(stream));
  if (ends[0] < 0 || ends[1] < ends[0]) return TT_ERR_INVALID_ARG;
  if (ends[1] > ends[0] && (!d_utf8 || !d_piece_starts)) return TT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(h->mu);
  Workspace *w;
  if ((s = get_workspace(h, stream, ends[1] - ends[0], n_requests, &w)) != TT_OK) return s;
  CallArgs args = {d_utf8, d_byte_offsets, n_requests, nullptr, nullptr, d_piece_starts, d_piece_offsets, nullptr,
                   nullptr, ends[1] - ends[0]};
  TT_CUDA(cudaMemcpyAsync(w->W.args, &args, sizeof(args), cudaMemcpyHostToDevice, stream));
  const Work &W = w->W;
  TT_CUDA(cudaMemsetAsync(W.counters, 0, 4 * 16, stream));
  TT_CUDA(cudaMemsetAsync(W.bad, 0, (size_t)w->cap_reqs + 1, stream));
  int launched = 5;
  if (h->T.n_lit) {
    TT_CUDA(cudaMemsetAsync(W.lit_flag, 0, (size_t)w->cap_bytes + 8, stream));
    launch_lit_find(h->T, W, grid_tiles(w), stream);
    launch_lit_pick(h->T, W, grid_lit_pick(w), stream);
    launched += 2;
  }
  launch_prepass(h->T, W, grid_tiles(w), stream);
  launch_pretok(h->T, W, grid_tiles(w), stream);
  launch_hook_pre(W, stream);
  launch_hook_pieces(W, grid_pieces(w), stream);
  launch_hook_offsets(W, grid_reqs(w), stream);
  TT_CUDA(cudaGetLastError());
  h->launches += launched;
  return TT_OK;
}

extern "C" const char *tt_status_string(tt_status s) {
  switch (s) {
    case TT_OK: return "ok";
    case TT_ERR_INVALID_ARG: return "invalid argument";
    case TT_ERR_BAD_VOCAB: return "vocabulary or merge list rejected";
    case TT_ERR_BAD_FAMILY: return "unknown pattern family";
    case TT_ERR_INVALID_UTF8: return "a request is not valid UTF-8";
    case TT_ERR_CAPACITY: return "batch exceeds a stated bound";
    case TT_ERR_OOM: return "out of memory";
    case TT_ERR_CUDA: return "CUDA runtime error";
    case TT_ERR_TIMEOUT: return "bounded device wait ran out";
  }
  return "unknown status";
}

extern "C" void tt_profile(tt_tokenizer *h, int enable) {
  if (!h) return;
  std::lock_guard<std::mutex> lock(h->mu);
  h->profiling = enable != 0;
}

extern "C" int tt_profile_read(tt_tokenizer *h, const char **names, double *ms, int64_t *launches, int cap) {
  if (!h) return 0;
  std::lock_guard<std::mutex> lock(h->mu);
  for (auto &pd : h->pending) {
    cudaEventSynchronize(pd.b);
    float t = 0.f;
    cudaEventElapsedTime(&t, pd.a, pd.b);
    h->prof_ms[pd.kernel] += t;
    h->prof_n[pd.kernel] += 1;
    h->event_pool.push_back(pd.a);
    h->event_pool.push_back(pd.b);
  }
  h->pending.clear();
  int n = 0;
  for (int k = 0; k < N_KERNELS && n < cap; ++k) {
    if (h->prof_n[k] == 0) continue;          // not launched (the literal kernels without literals)
    if (names) names[n] = KERNEL_NAMES[k];
    if (ms) ms[n] = h->prof_ms[k];
    if (launches) launches[n] = h->prof_n[k];
    h->prof_ms[k] = 0;
    h->prof_n[k] = 0;
    ++n;
  }
  return n;
}

extern "C" int64_t tt_launch_count(tt_tokenizer *h) { return h ? h->launches.load() : 0; }

extern "C" const char *tt_table_digest(void) { return TT_CLASS_DIGEST; }

extern "C" tt_status tt_debug_lookback(tt_tokenizer *h, int32_t spin_limit, int32_t withhold_tile) {
  if (!h || spin_limit < 0 || withhold_tile < -1) return TT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(h->mu);
  cudaDeviceSynchronize();                   // no encode of the handle is in flight while the settings change
  h->spin_limit = spin_limit == 0 ? (1 << 22) : spin_limit;
  h->withhold_tile = withhold_tile;
  for (auto &kv : h->ws) {
    kv.second->W.spin_limit = h->spin_limit;
    kv.second->W.withhold_tile = h->withhold_tile;
    if (kv.second->graph) {                  // the captured kernels hold the old settings
      cudaGraphExecDestroy(kv.second->graph);
      kv.second->graph = nullptr;
    }
  }
  return TT_OK;
}

// ===================================================================
// tt_encode_batch_noalloc: the same kernels as tt_encode_batch_bounded,
// with their scratch carved from one array compiled into the library
// instead of a workspace allocated on demand.  For callers that cannot
// allocate device memory once they are running.
namespace {

constexpr int64_t NA_BYTES = TT_NOALLOC_MAX_BYTES;
constexpr int64_t NA_REQS = TT_NOALLOC_MAX_REQUESTS;
constexpr int64_t NA_TILES = (NA_BYTES + TILE - 1) / TILE + 1;
constexpr int64_t NA_CHUNKS = (NA_BYTES + 1 + IDS_CHUNK - 1) / IDS_CHUNK + 2;
constexpr size_t na_round(size_t x) { return (x + 255) & ~(size_t)255; }

// sizes of the scratch arrays, in the order they are carved
constexpr size_t NA_SIZES[] = {
    sizeof(int2) * NA_TILES, 2 * (size_t)NA_TILES,                     // s1_sum, rq_sum
    sizeof(S2) * NA_TILES, sizeof(S2) * NA_TILES, 4 * (size_t)NA_TILES, // s2_agg, s2_inc, s2_flag
    sizeof(int2) * NA_TILES, sizeof(int2) * NA_TILES, 4 * (size_t)NA_TILES,  // cnt_agg, cnt_inc, cnt_flag
    4 * (size_t)NA_CHUNKS, 4 * (size_t)NA_CHUNKS,                      // ids_agg, ids_inc
    4 * 16,                                                            // counters
    4 * (size_t)(NA_BYTES + 2), 4 * (size_t)(NA_BYTES + 1),            // piece_start, n_ids
    4 * (size_t)(NA_BYTES + 1),                                        // scratch
    4 * (size_t)(NA_BYTES + 1), 4 * (size_t)(NA_BYTES + 1), 4 * (size_t)(NA_BYTES + 1),  // tmp_a, tmp_b, tmp_c
    4 * 3 * (size_t)list_cap(NA_BYTES), 4 * (size_t)(NA_BYTES / (MID_MAX + 1) + 2),  // lists
    (size_t)NA_REQS + 1, 4 * (size_t)(NA_REQS + 2),                    // bad, bad_pre
    4 * (size_t)(NA_REQS + 1),                                         // req_piece
    4 * (size_t)NA_TILES * TILE, 4 * (size_t)NA_TILES, (size_t)NA_BYTES + 8,  // lit_cand, lit_cnt, lit_flag
    (size_t)NA_BYTES + 8,                                              // lit_len
    sizeof(CallArgs),                                                  // args
};
constexpr size_t na_total() {
  size_t t = 0;
  for (size_t s : NA_SIZES) t += na_round(s);
  return t;
}

}  // namespace

// The fixed scratch.  In host code this name is only a stand-in for the
// device array: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char tt_noalloc_scratch[na_total()];

// writes the per-call arguments into the scratch (no host staging buffer)
static __global__ void k_noalloc_args(CallArgs a, CallArgs *dst) { *dst = a; }

// Device address of the scratch on the current device, looked up once per
// device (the first call on a device should precede any stream capture).
static tt_status noalloc_scratch_address(int dev, unsigned char **out) {
  static std::mutex mu;
  static std::map<int, unsigned char *> addr;
  std::lock_guard<std::mutex> lock(mu);
  auto it = addr.find(dev);
  if (it == addr.end()) {
    unsigned char *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress((void **)&p, tt_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      fprintf(stderr, "toktier: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(e));
      return TT_ERR_CUDA;
    }
    it = addr.emplace(dev, p).first;
  }
  *out = it->second;
  return TT_OK;
}

extern "C" tt_status tt_encode_batch_noalloc(tt_tokenizer *h, const uint8_t *d_utf8, const int64_t *d_byte_offsets,
                                             int64_t n_requests, int64_t max_total_bytes, int32_t *d_out_ids,
                                             int64_t *d_out_id_offsets, tt_stream_t stream_) {
  if (!h || n_requests < 0 || !d_byte_offsets || !d_out_id_offsets || max_total_bytes < 0) return TT_ERR_INVALID_ARG;
  if (max_total_bytes > NA_BYTES || n_requests > NA_REQS) {
    fprintf(stderr, "toktier: tt_encode_batch_noalloc: batch of up to %lld bytes / %lld requests exceeds the fixed "
            "scratch (%d bytes, %d requests)\n", (long long)max_total_bytes, (long long)n_requests,
            TT_NOALLOC_MAX_BYTES, TT_NOALLOC_MAX_REQUESTS);
    return TT_ERR_CAPACITY;
  }
  if (n_requests > 0 && max_total_bytes > 0 && (!d_utf8 || !d_out_ids)) return TT_ERR_INVALID_ARG;
  cudaStream_t stream = (cudaStream_t)stream_;
  int dev = -1;
  TT_CUDA(cudaGetDevice(&dev));
  if (dev != h->device) return TT_ERR_INVALID_ARG;
  if (n_requests == 0) {
    TT_CUDA(cudaMemsetAsync(d_out_id_offsets, 0, sizeof(int64_t), stream));
    return TT_OK;
  }
  unsigned char *base = nullptr;
  tt_status s = noalloc_scratch_address(dev, &base);
  if (s != TT_OK) return s;
  Work W{};
  void **dst[] = {(void **)&W.s1_sum,  (void **)&W.rq_sum,
                  (void **)&W.s2_agg,  (void **)&W.s2_inc,   (void **)&W.s2_flag,  (void **)&W.cnt_agg,
                  (void **)&W.cnt_inc, (void **)&W.cnt_flag, (void **)&W.ids_agg,  (void **)&W.ids_inc,
                  (void **)&W.counters, (void **)&W.piece_start, (void **)&W.n_ids,
                  (void **)&W.scratch,  (void **)&W.tmp_a,    (void **)&W.tmp_b,
                  (void **)&W.tmp_c,   (void **)&W.long_list, (void **)&W.huge_list, (void **)&W.bad,
                  (void **)&W.bad_pre, (void **)&W.req_piece, (void **)&W.lit_cand, (void **)&W.lit_cnt,
                  (void **)&W.lit_flag, (void **)&W.lit_len, (void **)&W.args};
  static_assert(sizeof(dst) / sizeof(dst[0]) == sizeof(NA_SIZES) / sizeof(NA_SIZES[0]), "layout");
  size_t off = 0;
  for (size_t i = 0; i < sizeof(NA_SIZES) / sizeof(NA_SIZES[0]); ++i) {
    *dst[i] = base + off;
    off += na_round(NA_SIZES[i]);
  }
  W.cap_bytes = NA_BYTES;
  W.cap_reqs = NA_REQS;
  W.cap_tiles = (int32_t)NA_TILES;
  W.status = h->d_status;
  Tables T;
  {
    // a consistent view of the tables and settings (tt_set_added_tokens and
    // tt_debug_lookback change them under this lock); the launches need no lock
    std::lock_guard<std::mutex> lock(h->mu);
    T = h->T;
    W.spin_limit = h->spin_limit;
    W.withhold_tile = h->withhold_tile;
  }
  const CallArgs args = {d_utf8, d_byte_offsets, n_requests, d_out_ids, d_out_id_offsets, nullptr, nullptr, nullptr,
                         nullptr, max_total_bytes};
  k_noalloc_args<<<1, 1, 0, stream>>>(args, W.args);
  // what must start at zero: the counters and the rejected-request flags
  // (look-back flags and ID chunk totals are reset by k_prepass)
  TT_CUDA(cudaMemsetAsync(W.counters, 0, 4 * 16, stream));
  TT_CUDA(cudaMemsetAsync(W.bad, 0, (size_t)NA_REQS + 1, stream));
  const int g_tiles = (int)((NA_BYTES + TILE - 1) / TILE);
  const int g_warp = (int)warp_grid(NA_BYTES);
  const int g_long = (int)std::min<int64_t>(std::max<int64_t>(NA_BYTES / (MID_MAX + 1), 1), 152 * 2);
  const int g_chunks = (int)((NA_BYTES + 1 + IDS_CHUNK - 1) / IDS_CHUNK);
  if (T.n_lit) {
    TT_CUDA(cudaMemsetAsync(W.lit_flag, 0, (size_t)NA_BYTES + 8, stream));
    launch_lit_find(T, W, g_tiles, stream);
    launch_lit_pick(T, W, (g_tiles + 7) / 8, stream);
  }
  launch_prepass(T, W, g_tiles, stream);
  launch_pretok(T, W, g_tiles, stream);
  launch_bpe_warp(T, W, g_warp, stream);
  launch_bpe_long(T, W, g_long, stream);
  launch_idscan(W, stream);
  launch_ids(T, W, g_chunks, stream);
  TT_CUDA(cudaGetLastError());
  h->launches += 7 + (T.n_lit ? 2 : 0);       // the encode's kernels and k_noalloc_args
  return TT_OK;
}
