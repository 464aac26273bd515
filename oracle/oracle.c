/*
 * CPU ORACLE for exact full-context BPE tokenization.  TEST INFRASTRUCTURE:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It shares no code with the CUDA path.
 *
 * What it computes (TokTier: Exact Stateful CPU+GPU Tokenization for Agentic
 * LLM Serving, §3.1: pre-tokenization, then BPE per piece; and the pipeline
 * definition F = E* o G of the summary page's §2.2): for every request
 * independently,
 *   1. decode the request as strict UTF-8 (a request that is not valid
 *      UTF-8 is rejected and yields no IDs);
 *   2. pre-tokenize it G: starting at position 0, try the pattern family's
 *      alternatives in order, take the first that matches (each alternative
 *      with the regex's own greedy-with-backtracking semantics), emit that
 *      match as one piece and continue at its end (§4.1: the GPT-family
 *      patterns are ordered alternatives tried leftmost-first, each with the
 *      usual backtracking);
 *   3. encode every piece E independently (§4.2): if the piece's bytes are a
 *      vocabulary entry emit that one ID (the ignore_merges shortcut), else
 *      start from single-byte IDs and repeatedly merge the LEFTMOST occurrence
 *      of the adjacent pair with the lowest merge rank until no adjacent pair
 *      has a rank;
 *   4. concatenate the IDs.
 * Nothing here is blocked, fused or reordered: one sequential matcher, one
 * single-merge loop per piece.
 *
 * Character classes come from the frozen table (probed from the regex engine,
 * §4.1 and §5.2); the caller passes it in as one uint16 mask per code point:
 *   bit 0 L, 1 Lu, 2 Ll, 3 Lt, 4 Lm, 5 Lo, 6 M, 7 N, 8 \s.
 *
 * Pattern families (the pages print neither pattern; these are this
 * project's own specifications of the two lineages the paper names):
 *   cl100k-style, alternatives in order:
 *     C1  '(?i:s|t|re|ve|m|ll|d)            (ASCII case folding)
 *     C2  [^\r\n\p{L}\p{N}]?\p{L}+
 *     C3  \p{N}{1,3}
 *     C4   ?[^\s\p{L}\p{N}]+[\r\n]*
 *     C5  \s*[\r\n]+
 *     C6  \s+(?!\S)
 *     C7  \s+
 *   o200k-style, alternatives in order (U = Lu Lt Lm Lo M, W = Ll Lm Lo M,
 *   K = an optional contraction suffix as in C1):
 *     O1  [^\r\n\p{L}\p{N}]?U*W+K?
 *     O2  [^\r\n\p{L}\p{N}]?U+W*K?
 *     O3..O7 as C3..C7
 *   deepseek-style (the paper, §4.1: DeepSeek-family tokenizers run three
 *   splitters one after another; each one re-splits every piece the one
 *   before it produced, and the text between two of its matches stays a
 *   piece of its own).  The three splitters:
 *     D1  \p{N}{1,3}
 *     D2  [\x{3040}-\x{30FF}\x{4E00}-\x{9FFF}]+   (Hiragana, Katakana and CJK
 *         Unified Ideographs blocks)
 *     D3  C1 | C2 | C4 | C5 | C6 | C7   (no digit alternative: a digit group
 *         left by D1 matches nothing and survives whole)
 *   A splitter applied to a piece sees that piece as its whole subject: the
 *   piece's end is the end of the text for C6's lookahead.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

enum { B_L = 1, B_LU = 2, B_LL = 4, B_LT = 8, B_LM = 16, B_LO = 32, B_M = 64, B_N = 128, B_S = 256 };
enum { FAM_CL100K = 1, FAM_O200K = 2, FAM_DEEPSEEK = 3 };
enum { OK = 0, ERR_ARG = 1, ERR_VOCAB = 2, ERR_FAMILY = 3, ERR_UTF8 = 4, ERR_CAPACITY = 5, ERR_OOM = 6 };

typedef struct {
  const uint16_t *cls;           /* 0x110000 masks, owned by the caller */
  int family;
  int64_t n_vocab;
  const uint8_t *vbytes;         /* copies */
  int64_t *voff;
  int64_t *vsorted;              /* vocab ids sorted by byte string */
  int64_t n_merges;
  int32_t *mleft, *mright;       /* by rank */
  int32_t *mresult;              /* result id by rank */
  int64_t *msorted;              /* ranks sorted by (left, right) */
  int64_t n_lit;                 /* added-token literals (copies) */
  uint8_t *lbytes;
  int64_t *loff;
  int32_t *lid;
} oracle_t;

/* ------------------------------------------------------------ classes */
static int mask(const oracle_t *o, uint32_t cp) { return cp < 0x110000 ? o->cls[cp] : 0; }
static int isL(const oracle_t *o, uint32_t c) { return mask(o, c) & B_L; }
static int isN(const oracle_t *o, uint32_t c) { return mask(o, c) & B_N; }
static int isS(const oracle_t *o, uint32_t c) { return mask(o, c) & B_S; }
static int isCRLF(uint32_t c) { return c == '\r' || c == '\n'; }
/* [^\r\n\p{L}\p{N}] */
static int isPrefix(const oracle_t *o, uint32_t c) { return !isCRLF(c) && !isL(o, c) && !isN(o, c); }
/* [^\s\p{L}\p{N}] */
static int isOther(const oracle_t *o, uint32_t c) { return !isS(o, c) && !isL(o, c) && !isN(o, c); }
/* o200k U = [\p{Lu}\p{Lt}\p{Lm}\p{Lo}\p{M}], W = [\p{Ll}\p{Lm}\p{Lo}\p{M}] */
static int isUpperSet(const oracle_t *o, uint32_t c) { return mask(o, c) & (B_LU | B_LT | B_LM | B_LO | B_M); }
static int isLowerSet(const oracle_t *o, uint32_t c) { return mask(o, c) & (B_LL | B_LM | B_LO | B_M); }
/* deepseek-style D2: the Hiragana, Katakana and CJK Unified Ideographs blocks */
static int isKanaHan(uint32_t c) { return (c >= 0x3040 && c <= 0x30FF) || (c >= 0x4E00 && c <= 0x9FFF); }

/* ------------------------------------------------------- strict UTF-8 */
/* RFC 3629: no overlongs, no surrogates, nothing above U+10FFFF, no stray or
 * missing continuation bytes.  Returns the number of code points or -1. */
static int64_t utf8_decode(const uint8_t *b, int64_t n, uint32_t *cp, int64_t *pos) {
  int64_t i = 0, k = 0;
  while (i < n) {
    uint32_t c = b[i];
    int len;
    uint32_t min;
    if (c < 0x80) { len = 1; min = 0; }
    else if (c >= 0xC2 && c <= 0xDF) { len = 2; c &= 0x1F; min = 0x80; }
    else if (c >= 0xE0 && c <= 0xEF) { len = 3; c &= 0x0F; min = 0x800; }
    else if (c >= 0xF0 && c <= 0xF4) { len = 4; c &= 0x07; min = 0x10000; }
    else return -1;
    if (i + len > n) return -1;
    for (int j = 1; j < len; ++j) {
      if ((b[i + j] & 0xC0) != 0x80) return -1;
      c = (c << 6) | (b[i + j] & 0x3F);
    }
    if (c < min || c > 0x10FFFF || (c >= 0xD800 && c <= 0xDFFF)) return -1;
    cp[k] = c; pos[k] = i; ++k;
    i += len;
  }
  pos[k] = n;
  return k;
}

/* ---------------------------------------------------- the alternatives */
/* each returns the match end (> p) or -1; c[0..n) are code points */

static int contraction_len(const uint32_t *c, int64_t n, int64_t p) {   /* '(?i:s|t|re|ve|m|ll|d) at p, or 0 */
  if (p >= n || c[p] != '\'') return 0;
  uint32_t a = p + 1 < n ? c[p + 1] : 0, b = p + 2 < n ? c[p + 2] : 0;
  if (a >= 'A' && a <= 'Z') a += 32;
  if (b >= 'A' && b <= 'Z') b += 32;
  if (a == 's' || a == 't') return 2;            /* alternatives tried in order: 's 't 're 've 'm 'll 'd */
  if (a == 'r' && b == 'e') return 3;
  if (a == 'v' && b == 'e') return 3;
  if (a == 'm') return 2;
  if (a == 'l' && b == 'l') return 3;
  if (a == 'd') return 2;
  return 0;
}

static int64_t count_while(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p, int (*pred)(const oracle_t *, uint32_t)) {
  int64_t q = p;
  while (q < n && pred(o, c[q])) ++q;
  return q - p;
}
static int isCRLFo(const oracle_t *o, uint32_t c) { (void)o; return isCRLF(c); }

/* C2: [^\r\n\p{L}\p{N}]?\p{L}+ */
static int64_t alt_letters(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p) {
  for (int pre = 1; pre >= 0; --pre) {                     /* greedy ? : with the char first */
    if (pre && !isPrefix(o, c[p])) continue;
    int64_t q = p + pre;
    int64_t k = count_while(o, c, n, q, isL);
    if (k >= 1) return q + k;
  }
  return -1;
}

/* C3: \p{N}{1,3} */
static int64_t alt_digits(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p) {
  int64_t k = 0;
  while (k < 3 && p + k < n && isN(o, c[p + k])) ++k;
  return k >= 1 ? p + k : -1;
}

/* C4:  ?[^\s\p{L}\p{N}]+[\r\n]* */
static int64_t alt_other(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p) {
  for (int sp = 1; sp >= 0; --sp) {
    if (sp && c[p] != ' ') continue;
    int64_t q = p + sp;
    int64_t k = count_while(o, c, n, q, isOther);
    if (k >= 1) { q += k; return q + count_while(o, c, n, q, isCRLFo); }
  }
  return -1;
}

/* C5: \s*[\r\n]+   (backtrack \s* from its longest) */
static int64_t alt_newlines(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p) {
  int64_t w = count_while(o, c, n, p, isS);
  for (int64_t k = w; k >= 0; --k) {
    int64_t r = count_while(o, c, n, p + k, isCRLFo);
    if (r >= 1) return p + k + r;
  }
  return -1;
}

/* C6: \s+(?!\S)   (backtrack \s+ from its longest) */
static int64_t alt_trailing_ws(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p) {
  int64_t w = count_while(o, c, n, p, isS);
  for (int64_t k = w; k >= 1; --k)
    if (p + k == n || isS(o, c[p + k])) return p + k;
  return -1;
}

/* C7: \s+ */
static int64_t alt_ws(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p) {
  int64_t w = count_while(o, c, n, p, isS);
  return w >= 1 ? p + w : -1;
}

/* O1: [^\r\n\p{L}\p{N}]?U*W+K?   (backtrack U* from its longest) */
static int64_t alt_case_lower(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p) {
  for (int pre = 1; pre >= 0; --pre) {
    if (pre && !isPrefix(o, c[p])) continue;
    int64_t q = p + pre;
    int64_t u = count_while(o, c, n, q, isUpperSet);
    for (int64_t k = u; k >= 0; --k) {
      int64_t w = count_while(o, c, n, q + k, isLowerSet);
      if (w >= 1) { int64_t e = q + k + w; return e + contraction_len(c, n, e); }
    }
  }
  return -1;
}

/* O2: [^\r\n\p{L}\p{N}]?U+W*K? */
static int64_t alt_case_upper(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p) {
  for (int pre = 1; pre >= 0; --pre) {
    if (pre && !isPrefix(o, c[p])) continue;
    int64_t q = p + pre;
    int64_t u = count_while(o, c, n, q, isUpperSet);
    if (u >= 1) {
      int64_t e = q + u + count_while(o, c, n, q + u, isLowerSet);
      return e + contraction_len(c, n, e);
    }
  }
  return -1;
}

/* one piece starting at p: the first alternative that matches */
static int64_t match_at(const oracle_t *o, const uint32_t *c, int64_t n, int64_t p) {
  int64_t e;
  if (o->family == FAM_CL100K) {
    int k = contraction_len(c, n, p);
    if (k) return p + k;
    if ((e = alt_letters(o, c, n, p)) > 0) return e;
  } else {
    if ((e = alt_case_lower(o, c, n, p)) > 0) return e;
    if ((e = alt_case_upper(o, c, n, p)) > 0) return e;
  }
  if ((e = alt_digits(o, c, n, p)) > 0) return e;
  if ((e = alt_other(o, c, n, p)) > 0) return e;
  if ((e = alt_newlines(o, c, n, p)) > 0) return e;
  if ((e = alt_trailing_ws(o, c, n, p)) > 0) return e;
  if ((e = alt_ws(o, c, n, p)) > 0) return e;
  return -1;   /* unreachable: every code point is L, N, \s or other */
}

/* deepseek-style: the end of a match of splitter `stage` (1 = D1, 2 = D2,
 * 3 = D3) at p inside the subject c[0..n), or -1 */
static int64_t ds_match(const oracle_t *o, int stage, const uint32_t *c, int64_t n, int64_t p) {
  int64_t e;
  if (stage == 1) return alt_digits(o, c, n, p);
  if (stage == 2) {
    e = p;
    while (e < n && isKanaHan(c[e])) ++e;
    return e > p ? e : -1;
  }
  int k = contraction_len(c, n, p);
  if (k) return p + k;
  if ((e = alt_letters(o, c, n, p)) > 0) return e;
  if ((e = alt_other(o, c, n, p)) > 0) return e;
  if ((e = alt_newlines(o, c, n, p)) > 0) return e;
  if ((e = alt_trailing_ws(o, c, n, p)) > 0) return e;
  return alt_ws(o, c, n, p);
}

static int64_t ds_split(const oracle_t *o, int stage, const uint32_t *c, int64_t a, int64_t b, int64_t *starts,
                        int64_t k);
/* a piece [a, b) that splitter `stage` produced: the last splitter's pieces
 * are final, the others go to the next splitter */
static int64_t ds_emit(const oracle_t *o, int stage, const uint32_t *c, int64_t a, int64_t b, int64_t *starts,
                       int64_t k) {
  if (stage == 3) { starts[k] = a; return k + 1; }
  return ds_split(o, stage + 1, c, a, b, starts, k);
}
/* Splitter `stage` over the piece c[a..b), which is its whole subject: scan
 * for the leftmost match from the end of the previous one; the stretch
 * skipped before a match (and the rest after the last match) is a piece too. */
static int64_t ds_split(const oracle_t *o, int stage, const uint32_t *c, int64_t a, int64_t b, int64_t *starts,
                        int64_t k) {
  int64_t p = a, q = a;   /* p: start of the unmatched stretch; q: where a match is tried */
  while (q < b) {
    const int64_t e = ds_match(o, stage, c + a, b - a, q - a);
    if (e < 0) { ++q; continue; }
    if (q > p) k = ds_emit(o, stage, c, p, q, starts, k);
    k = ds_emit(o, stage, c, q, a + e, starts, k);
    p = q = a + e;
  }
  if (b > p) k = ds_emit(o, stage, c, p, b, starts, k);
  return k;
}

/* pre-tokenize c[0..n): writes piece start indices (char indices); returns count */
static int64_t pretokenize_chars(const oracle_t *o, const uint32_t *c, int64_t n, int64_t *starts) {
  if (o->family == FAM_DEEPSEEK) return ds_split(o, 1, c, 0, n, starts, 0);
  int64_t p = 0, k = 0;
  while (p < n) {
    int64_t e = match_at(o, c, n, p);
    if (e <= p) return -1;
    starts[k++] = p;
    p = e;
  }
  return k;
}

/* ------------------------------------------------------------- vocab */
static const oracle_t *g_sort_ctx;
static int cmp_bytes(const uint8_t *a, int64_t la, const uint8_t *b, int64_t lb) {
  int64_t m = la < lb ? la : lb;
  int r = memcmp(a, b, (size_t)m);
  if (r) return r;
  return la < lb ? -1 : la > lb;
}
static int cmp_vid(const void *x, const void *y) {
  const oracle_t *o = g_sort_ctx;
  int64_t a = *(const int64_t *)x, b = *(const int64_t *)y;
  return cmp_bytes(o->vbytes + o->voff[a], o->voff[a + 1] - o->voff[a], o->vbytes + o->voff[b], o->voff[b + 1] - o->voff[b]);
}
static int cmp_rank(const void *x, const void *y) {
  const oracle_t *o = g_sort_ctx;
  int64_t a = *(const int64_t *)x, b = *(const int64_t *)y;
  if (o->mleft[a] != o->mleft[b]) return o->mleft[a] < o->mleft[b] ? -1 : 1;
  if (o->mright[a] != o->mright[b]) return o->mright[a] < o->mright[b] ? -1 : 1;
  return 0;
}

/* id of a byte string, or -1 (binary search over the sorted vocab) */
static int64_t vocab_find(const oracle_t *o, const uint8_t *b, int64_t len) {
  int64_t lo = 0, hi = o->n_vocab - 1;
  while (lo <= hi) {
    int64_t mid = (lo + hi) / 2, id = o->vsorted[mid];
    int r = cmp_bytes(o->vbytes + o->voff[id], o->voff[id + 1] - o->voff[id], b, len);
    if (r == 0) return id;
    if (r < 0) lo = mid + 1; else hi = mid - 1;
  }
  return -1;
}

/* rank of the pair (l, r), or -1 */
static int64_t merge_rank(const oracle_t *o, int32_t l, int32_t r) {
  int64_t lo = 0, hi = o->n_merges - 1;
  while (lo <= hi) {
    int64_t mid = (lo + hi) / 2, k = o->msorted[mid];
    int c = o->mleft[k] != l ? (o->mleft[k] < l ? -1 : 1) : o->mright[k] != r ? (o->mright[k] < r ? -1 : 1) : 0;
    if (c == 0) return k;
    if (c < 0) lo = mid + 1; else hi = mid - 1;
  }
  return -1;
}

static pthread_mutex_t g_sort_lock = PTHREAD_MUTEX_INITIALIZER;

/* Build the oracle.  Copies the vocab and merges; keeps the class-table
 * pointer.  Checks only what the oracle itself needs: every single byte is an
 * entry, entries are unique, and every merge's concatenation is an entry. */
int oracle_create(const uint16_t *cls, int family,
                  const int32_t *merges, int64_t n_merges,
                  const uint8_t *vbytes, const int64_t *voff, int64_t n_vocab, void **out) {
  if (!cls || !out || n_vocab < 256 || n_merges < 0 || (n_merges && !merges)) return ERR_ARG;
  if (family != FAM_CL100K && family != FAM_O200K && family != FAM_DEEPSEEK) return ERR_FAMILY;
  oracle_t *o = calloc(1, sizeof(oracle_t));
  o->cls = cls; o->family = family; o->n_vocab = n_vocab; o->n_merges = n_merges;
  int64_t nb = voff[n_vocab] - voff[0];
  uint8_t *vb = malloc((size_t)(nb ? nb : 1));
  memcpy(vb, vbytes + voff[0], (size_t)nb);
  o->vbytes = vb;
  o->voff = malloc(sizeof(int64_t) * (size_t)(n_vocab + 1));
  for (int64_t i = 0; i <= n_vocab; ++i) o->voff[i] = voff[i] - voff[0];
  o->vsorted = malloc(sizeof(int64_t) * (size_t)n_vocab);
  for (int64_t i = 0; i < n_vocab; ++i) o->vsorted[i] = i;
  o->mleft = malloc(sizeof(int32_t) * (size_t)(n_merges + 1));
  o->mright = malloc(sizeof(int32_t) * (size_t)(n_merges + 1));
  o->mresult = malloc(sizeof(int32_t) * (size_t)(n_merges + 1));
  o->msorted = malloc(sizeof(int64_t) * (size_t)(n_merges + 1));
  for (int64_t k = 0; k < n_merges; ++k) { o->mleft[k] = merges[2 * k]; o->mright[k] = merges[2 * k + 1]; o->msorted[k] = k; }
  pthread_mutex_lock(&g_sort_lock);
  g_sort_ctx = o;
  qsort(o->vsorted, (size_t)n_vocab, sizeof(int64_t), cmp_vid);
  qsort(o->msorted, (size_t)n_merges, sizeof(int64_t), cmp_rank);
  pthread_mutex_unlock(&g_sort_lock);
  int st = OK;
  for (int64_t i = 1; i < n_vocab && st == OK; ++i) {
    int64_t a = o->vsorted[i - 1], b = o->vsorted[i];
    if (!cmp_bytes(o->vbytes + o->voff[a], o->voff[a + 1] - o->voff[a], o->vbytes + o->voff[b], o->voff[b + 1] - o->voff[b])) st = ERR_VOCAB;
  }
  for (int v = 0; v < 256 && st == OK; ++v) { uint8_t b = (uint8_t)v; if (vocab_find(o, &b, 1) < 0) st = ERR_VOCAB; }
  for (int64_t k = 0; k < n_merges && st == OK; ++k) {
    int32_t l = o->mleft[k], r = o->mright[k];
    if (l < 0 || r < 0 || l >= n_vocab || r >= n_vocab) { st = ERR_VOCAB; break; }
    int64_t ll = o->voff[l + 1] - o->voff[l], lr = o->voff[r + 1] - o->voff[r];
    uint8_t *cat = malloc((size_t)(ll + lr));
    memcpy(cat, o->vbytes + o->voff[l], (size_t)ll);
    memcpy(cat + ll, o->vbytes + o->voff[r], (size_t)lr);
    int64_t id = vocab_find(o, cat, ll + lr);
    free(cat);
    if (id < 0) st = ERR_VOCAB; else o->mresult[k] = (int32_t)id;
  }
  *out = o;
  return st;
}

/* Added tokens (TokTier §4.4: literal strings the model reserves as single
 * IDs, extracted leftmost-longest before the family tokenizes the rest):
 * n literals, bytes[offs[k] .. offs[k+1]) with ID ids[k].  Replaces any
 * earlier set; n = 0 clears it.  Literals must be non-empty and distinct. */
int oracle_set_added_tokens(void *h, const uint8_t *bytes, const int64_t *offs, const int32_t *ids, int64_t n) {
  oracle_t *o = h;
  if (!o || n < 0 || (n > 0 && (!bytes || !offs || !ids))) return ERR_ARG;
  for (int64_t k = 0; k < n; ++k) {
    if (offs[k + 1] - offs[k] < 1) return ERR_ARG;
    for (int64_t q = 0; q < k; ++q)
      if (offs[q + 1] - offs[q] == offs[k + 1] - offs[k] &&
          memcmp(bytes + offs[q], bytes + offs[k], (size_t)(offs[k + 1] - offs[k])) == 0)
        return ERR_ARG;
  }
  free(o->lbytes); free(o->loff); free(o->lid);
  o->n_lit = n;
  const int64_t total = n > 0 ? offs[n] - offs[0] : 0;
  o->lbytes = malloc((size_t)(total ? total : 1));
  o->loff = malloc(sizeof(int64_t) * (size_t)(n + 1));
  o->lid = malloc(sizeof(int32_t) * (size_t)(n ? n : 1));
  if (total) memcpy(o->lbytes, bytes + offs[0], (size_t)total);
  o->loff[0] = 0;
  for (int64_t k = 0; k < n; ++k) { o->loff[k + 1] = offs[k + 1] - offs[0]; o->lid[k] = ids[k]; }
  return OK;
}

void oracle_destroy(void *h) {
  oracle_t *o = h;
  if (!o) return;
  free(o->lbytes); free(o->loff); free(o->lid);
  free((void *)o->vbytes); free(o->voff); free(o->vsorted);
  free(o->mleft); free(o->mright); free(o->mresult); free(o->msorted);
  free(o);
}

/* E: encode one piece's bytes.  ids must hold len entries; returns the count.
 * rank[] caches the rank of each adjacent pair; after a merge only the two
 * pairs next to it change, so only they are looked up again.
 * If sstart is not NULL it must hold len entries and receives, for every
 * emitted ID, the offset in the piece of the first byte that ID covers: each
 * symbol starts as one byte at its own offset, and a merge keeps the left
 * symbol's start (the byte range of a merged symbol is the union of the two
 * adjacent ranges it joins).  This provenance is tracked through the merges,
 * not derived from token lengths. */
static int64_t encode_piece_spans(const oracle_t *o, const uint8_t *b, int64_t len, int32_t *ids, int64_t *rank,
                                  int64_t *sstart) {
  int64_t whole = vocab_find(o, b, len);
  if (whole >= 0) {
    ids[0] = (int32_t)whole;
    if (sstart) sstart[0] = 0;
    return 1;
  }
  int64_t n = len;
  for (int64_t i = 0; i < n; ++i) ids[i] = (int32_t)vocab_find(o, b + i, 1);
  if (sstart) for (int64_t i = 0; i < n; ++i) sstart[i] = i;
  for (int64_t i = 0; i + 1 < n; ++i) rank[i] = merge_rank(o, ids[i], ids[i + 1]);
  for (;;) {
    int64_t best = -1, at = -1;
    for (int64_t i = 0; i + 1 < n; ++i)                 /* lowest rank, leftmost on ties */
      if (rank[i] >= 0 && (best < 0 || rank[i] < best)) { best = rank[i]; at = i; }
    if (best < 0) break;
    ids[at] = o->mresult[best];
    memmove(ids + at + 1, ids + at + 2, sizeof(int32_t) * (size_t)(n - at - 2));
    if (sstart) memmove(sstart + at + 1, sstart + at + 2, sizeof(int64_t) * (size_t)(n - at - 2));
    memmove(rank + at + 1, rank + at + 2, sizeof(int64_t) * (size_t)(n > at + 3 ? n - at - 3 : 0));
    --n;
    if (at > 0) rank[at - 1] = merge_rank(o, ids[at - 1], ids[at]);
    if (at + 1 < n) rank[at] = merge_rank(o, ids[at], ids[at + 1]);
  }
  return n;
}

static int64_t encode_piece(const oracle_t *o, const uint8_t *b, int64_t len, int32_t *ids, int64_t *rank) {
  return encode_piece_spans(o, b, len, ids, rank, NULL);
}

/* ---------------------------------------------------------- batch API */
typedef struct {
  const oracle_t *o;
  const uint8_t *bytes;
  const int64_t *offs;
  int64_t n_req;
  int64_t next;                  /* next request to take (shared, locked) */
  pthread_mutex_t lock;
  /* per request results, owned by the job */
  int32_t **ids; int64_t *nids;
  int64_t **spans;               /* per request: (start, end) per ID, relative to the request */
  int64_t **pieces; int64_t *npieces;
  int *status;
  int want_ids, want_spans;
} job_t;

/* The longest added-token literal that occurs at byte x of b[0..nb), as an
 * index, or -1. */
static int64_t literal_at(const oracle_t *o, const uint8_t *b, int64_t nb, int64_t x) {
  int64_t best = -1, best_len = 0;
  for (int64_t k = 0; k < o->n_lit; ++k) {
    const int64_t len = o->loff[k + 1] - o->loff[k];
    if (len > best_len && x + len <= nb && memcmp(b + x, o->lbytes + o->loff[k], (size_t)len) == 0) {
      best = k;
      best_len = len;
    }
  }
  return best;
}

/* G on the chars of bytes [from, to) of a valid request: appends the piece
 * starts (byte offsets relative to the request) to st, marks them unforced. */
static int64_t pretokenize_segment(const oracle_t *o, const uint8_t *b, int64_t from, int64_t to, int64_t *st,
                                   int64_t *forced, int64_t np) {
  if (to <= from) return np;
  uint32_t *cp = malloc(sizeof(uint32_t) * (size_t)(to - from + 1));
  int64_t *pos = malloc(sizeof(int64_t) * (size_t)(to - from + 2));
  int64_t *s = malloc(sizeof(int64_t) * (size_t)(to - from + 1));
  const int64_t nc = utf8_decode(b + from, to - from, cp, pos);     /* valid: the request passed */
  const int64_t k = pretokenize_chars(o, cp, nc, s);
  for (int64_t i = 0; i < k; ++i) { st[np] = from + pos[s[i]]; forced[np] = -1; ++np; }
  free(cp); free(pos); free(s);
  return np;
}

static void run_request(job_t *j, int64_t r) {
  const oracle_t *o = j->o;
  const uint8_t *b = j->bytes + j->offs[r];
  int64_t nb = j->offs[r + 1] - j->offs[r];
  uint32_t *cp = malloc(sizeof(uint32_t) * (size_t)(nb + 1));
  int64_t *pos = malloc(sizeof(int64_t) * (size_t)(nb + 2));
  int64_t nc = utf8_decode(b, nb, cp, pos);
  free(cp); free(pos);
  if (nc < 0) { j->status[r] = ERR_UTF8; return; }
  /* Added tokens first (TokTier §4.4): scanning left to right, the longest
   * literal at the leftmost position where one occurs is cut out as one piece
   * with its reserved ID; the segments between literals are pre-tokenized
   * separately, as documents of their own. */
  int64_t *st = malloc(sizeof(int64_t) * (size_t)(nb + 1));
  int64_t *forced = malloc(sizeof(int64_t) * (size_t)(nb + 1));   /* literal ID of a piece, or -1 */
  int64_t np = 0, seg = 0;
  for (int64_t x = 0; o->n_lit > 0 && x < nb;) {
    const int64_t k = literal_at(o, b, nb, x);
    if (k < 0) { ++x; continue; }
    np = pretokenize_segment(o, b, seg, x, st, forced, np);
    st[np] = x; forced[np] = o->lid[k]; ++np;
    x += o->loff[k + 1] - o->loff[k];
    seg = x;
  }
  np = pretokenize_segment(o, b, seg, nb, st, forced, np);
  st[np] = nb;
  j->pieces[r] = st; j->npieces[r] = np;
  if (j->want_ids) {
    int32_t *ids = malloc(sizeof(int32_t) * (size_t)(nb + 1));
    int64_t *rank = malloc(sizeof(int64_t) * (size_t)(nb + 1));
    int64_t *ss = malloc(sizeof(int64_t) * (size_t)(nb + 1));
    int64_t *sp = j->want_spans ? malloc(sizeof(int64_t) * 2 * (size_t)(nb + 1)) : NULL;
    int64_t t = 0;
    for (int64_t k = 0; k < np; ++k) {
      const int64_t plen = st[k + 1] - st[k];
      int64_t m;
      if (forced[k] >= 0) {                       /* a literal: its one reserved ID */
        ids[t] = (int32_t)forced[k];
        ss[0] = 0;
        m = 1;
      } else {
        m = encode_piece_spans(o, b + st[k], plen, ids + t, rank, ss);
      }
      for (int64_t i = 0; sp && i < m; ++i) {     /* an ID ends where the next one in its piece starts */
        sp[2 * (t + i)] = st[k] + ss[i];
        sp[2 * (t + i) + 1] = st[k] + (i + 1 < m ? ss[i + 1] : plen);
      }
      t += m;
    }
    free(rank); free(ss);
    j->ids[r] = ids; j->nids[r] = t;
    j->spans[r] = sp;
  }
  free(forced);
}

static void *worker(void *arg) {
  job_t *j = arg;
  for (;;) {
    pthread_mutex_lock(&j->lock);
    int64_t r = j->next++;
    pthread_mutex_unlock(&j->lock);
    if (r >= j->n_req) break;
    run_request(j, r);
  }
  return NULL;
}

/* Tokenize a batch.  bytes/offs describe the requests (offs[0..n_req]).
 * Outputs (any may be NULL):
 *   out_ids[cap_ids] + out_id_offsets[n_req+1]  IDs, concatenated per request
 *   out_piece_starts[cap_pieces] + out_piece_offsets[n_req+1]
 *        piece starts as absolute byte offsets into `bytes`
 *   out_status[n_req]   per-request status (ERR_UTF8 for invalid requests,
 *                       which contribute no pieces and no IDs)
 * threads: worker threads (>= 1).  Returns OK or ERR_CAPACITY. */
static int run_batch(void *h, const uint8_t *bytes, const int64_t *offs, int64_t n_req, int threads,
                     int32_t *out_ids, int64_t cap_ids, int64_t *out_id_offsets, int64_t *out_spans,
                     int64_t *out_piece_starts, int64_t cap_pieces, int64_t *out_piece_offsets,
                     int32_t *out_status) {
  job_t j;
  memset(&j, 0, sizeof(j));
  j.o = h; j.bytes = bytes; j.offs = offs; j.n_req = n_req;
  j.want_spans = out_spans != NULL;
  j.want_ids = out_ids != NULL || out_id_offsets != NULL || j.want_spans;
  pthread_mutex_init(&j.lock, NULL);
  j.ids = calloc((size_t)(n_req + 1), sizeof(int32_t *)); j.nids = calloc((size_t)(n_req + 1), sizeof(int64_t));
  j.spans = calloc((size_t)(n_req + 1), sizeof(int64_t *));
  j.pieces = calloc((size_t)(n_req + 1), sizeof(int64_t *)); j.npieces = calloc((size_t)(n_req + 1), sizeof(int64_t));
  j.status = calloc((size_t)(n_req + 1), sizeof(int));
  if (threads < 1) threads = 1;
  if (threads == 1 || n_req <= 1) {
    worker(&j);
  } else {
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)threads);
    for (int t = 0; t < threads; ++t) pthread_create(&th[t], NULL, worker, &j);
    for (int t = 0; t < threads; ++t) pthread_join(th[t], NULL);
    free(th);
  }
  int rc = OK;
  int64_t ti = 0, tp = 0;
  if (out_id_offsets) out_id_offsets[0] = 0;
  if (out_piece_offsets) out_piece_offsets[0] = 0;
  for (int64_t r = 0; r < n_req; ++r) {
    if (out_status) out_status[r] = j.status[r];
    if (j.want_ids) {
      if (out_ids) {
        if (ti + j.nids[r] > cap_ids) rc = ERR_CAPACITY;
        else memcpy(out_ids + ti, j.ids[r], sizeof(int32_t) * (size_t)j.nids[r]);
      }
      if (out_spans) {                            /* byte offsets from the batch start offs[0] */
        if (ti + j.nids[r] > cap_ids) rc = ERR_CAPACITY;
        else for (int64_t i = 0; i < 2 * j.nids[r]; ++i) out_spans[2 * ti + i] = offs[r] - offs[0] + j.spans[r][i];
      }
      ti += j.nids[r];
      if (out_id_offsets) out_id_offsets[r + 1] = ti;
    }
    if (out_piece_starts) {
      if (tp + j.npieces[r] > cap_pieces) rc = ERR_CAPACITY;
      else for (int64_t k = 0; k < j.npieces[r]; ++k) out_piece_starts[tp + k] = offs[r] + j.pieces[r][k];
    }
    tp += j.npieces[r];
    if (out_piece_offsets) out_piece_offsets[r + 1] = tp;
    free(j.ids[r]); free(j.spans[r]); free(j.pieces[r]);
  }
  free(j.ids); free(j.nids); free(j.spans); free(j.pieces); free(j.npieces); free(j.status);
  pthread_mutex_destroy(&j.lock);
  return rc;
}

int oracle_run_batch(void *h, const uint8_t *bytes, const int64_t *offs, int64_t n_req, int threads,
                     int32_t *out_ids, int64_t cap_ids, int64_t *out_id_offsets,
                     int64_t *out_piece_starts, int64_t cap_pieces, int64_t *out_piece_offsets,
                     int32_t *out_status) {
  return run_batch(h, bytes, offs, n_req, threads, out_ids, cap_ids, out_id_offsets, NULL, out_piece_starts,
                   cap_pieces, out_piece_offsets, out_status);
}

/* As oracle_run_batch with IDs and, for every ID, the source byte range it
 * covers: out_spans[2 * cap_ids] receives (start, end) per ID, byte offsets
 * from the batch start offs[0] (TokTier §3: the session state a repair step
 * edits holds IDs and byte spans; §4.4: the paper's GPU path does not return
 * them).  Tracked through the merges as described at encode_piece_spans. */
int oracle_run_batch_spans(void *h, const uint8_t *bytes, const int64_t *offs, int64_t n_req, int threads,
                           int32_t *out_ids, int64_t cap_ids, int64_t *out_id_offsets, int64_t *out_spans,
                           int32_t *out_status) {
  return run_batch(h, bytes, offs, n_req, threads, out_ids, cap_ids, out_id_offsets, out_spans, NULL, 0, NULL,
                   out_status);
}

/* E alone on one byte string (for the BPE pins): ids must hold len entries */
int64_t oracle_encode_bytes(void *h, const uint8_t *b, int64_t len, int32_t *ids) {
  if (len <= 0) return 0;
  int64_t *rank = malloc(sizeof(int64_t) * (size_t)(len + 1));
  int64_t n = encode_piece(h, b, len, ids, rank);
  free(rank);
  return n;
}

/* the same loop without the whole-piece shortcut (plain BPE), for pins that
 * compare the two */
int64_t oracle_encode_bytes_plain(void *h, const uint8_t *b, int64_t len, int32_t *ids) {
  const oracle_t *o = h;
  if (len <= 0) return 0;
  int64_t *rank = malloc(sizeof(int64_t) * (size_t)(len + 1));
  int64_t n = len;
  for (int64_t i = 0; i < n; ++i) ids[i] = (int32_t)vocab_find(o, b + i, 1);
  for (int64_t i = 0; i + 1 < n; ++i) rank[i] = merge_rank(o, ids[i], ids[i + 1]);
  for (;;) {
    int64_t best = -1, at = -1;
    for (int64_t i = 0; i + 1 < n; ++i)
      if (rank[i] >= 0 && (best < 0 || rank[i] < best)) { best = rank[i]; at = i; }
    if (best < 0) break;
    ids[at] = o->mresult[best];
    memmove(ids + at + 1, ids + at + 2, sizeof(int32_t) * (size_t)(n - at - 2));
    memmove(rank + at + 1, rank + at + 2, sizeof(int64_t) * (size_t)(n > at + 3 ? n - at - 3 : 0));
    --n;
    if (at > 0) rank[at - 1] = merge_rank(o, ids[at - 1], ids[at]);
    if (at + 1 < n) rank[at] = merge_rank(o, ids[at], ids[at + 1]);
  }
  free(rank);
  return n;
}
