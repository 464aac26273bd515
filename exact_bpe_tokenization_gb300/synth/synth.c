/*
 * Seeded synthetic inputs for the exact BPE tokenizer: transcript-shaped text,
 * adversarial long-run text, request-length samplers and a greedy byte-level
 * BPE merge trainer.
 *
 * This module produces INPUTS only (text and a merge list).  It holds none of
 * the tokenizer's own arithmetic: the trainer splits its corpus with a crude
 * chunker of its own (below), not with the pre-tokenizer, and it never encodes
 * text with a finished merge list.  Both the CUDA path and the CPU oracle read
 * what this module writes; neither shares code with it beyond that.
 *
 * Determinism: the same seed gives the same bytes on x86-64 and AArch64.  The
 * random stream is PCG64 (XSL-RR 128/64, O'Neill 2014) on unsigned __int128;
 * floating point is limited to IEEE basic operations (+ - * / and frexp/ldexp),
 * with exp/log written out below from their series, and the file is compiled
 * with -ffp-contract=off so no fused multiply-add changes a rounding.
 *
 * Workload shapes follow the TokTier paper's description of coding-agent
 * transcripts (section 2 workload study; ~4 chars per token on real session
 * text, section 5.3) with the profile mix stated in the configuration text:
 * profile 0 = ASCII code-like text; profile 1 = adds mixed case, contractions,
 * CJK runs, Latin-1 letters, emoji and long blank runs; profile 2 = profile 1
 * plus camelCase/PascalCase identifiers and combining-mark text.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* ------------------------------------------------------------------ PCG64 */
typedef struct { unsigned __int128 state, inc; } pcg64_t;

static const unsigned __int128 PCG_MULT =
    (((unsigned __int128)0x2360ED051FC65DA4ULL) << 64) | 0x4385DF649FCCF645ULL;

static uint64_t pcg_next(pcg64_t *r) {
  r->state = r->state * PCG_MULT + r->inc;
  uint64_t hi = (uint64_t)(r->state >> 64), lo = (uint64_t)r->state;
  unsigned rot = (unsigned)(r->state >> 122);
  uint64_t x = hi ^ lo;
  return (x >> rot) | (x << ((64u - rot) & 63u));
}

static void pcg_seed(pcg64_t *r, uint64_t seed, uint64_t stream) {
  r->state = 0;
  r->inc = (((unsigned __int128)stream) << 1) | 1u;
  pcg_next(r);
  r->state += seed;
  pcg_next(r);
}

/* uniform integer in [0, n) by multiply-shift */
static uint64_t rnd_below(pcg64_t *r, uint64_t n) {
  return (uint64_t)(((unsigned __int128)pcg_next(r) * n) >> 64);
}
/* uniform double in [0, 1) with 53 random bits */
static double rnd_unit(pcg64_t *r) { return (double)(pcg_next(r) >> 11) * (1.0 / 9007199254740992.0); }
static int rnd_chance(pcg64_t *r, double p) { return rnd_unit(r) < p; }

/* ------------------------------------------- exp / log from their series */
static const double LN2 = 0.69314718055994530942;

static double det_log(double x) {          /* x > 0 */
  int e;
  double m = frexp(x, &e);                 /* x = m * 2^e, m in [0.5, 1) */
  m *= 2.0; e -= 1;                        /* m in [1, 2) */
  double t = (m - 1.0) / (m + 1.0), t2 = t * t, term = t, sum = 0.0;
  for (int k = 1; k < 80; k += 2) { sum += term / (double)k; term *= t2; }
  return (double)e * LN2 + 2.0 * sum;
}

static double det_exp(double x) {
  double kf = x / LN2;
  long k = (long)(kf < 0 ? kf - 0.5 : kf + 0.5);
  double r = x - (double)k * LN2, term = 1.0, sum = 1.0;
  for (int i = 1; i < 30; ++i) { term *= r / (double)i; sum += term; }
  return ldexp(sum, (int)k);
}

/* ------------------------------------------------------------ UTF-8 out */
typedef struct { uint8_t *buf; int64_t len, cap, chars, limit; int full; } sink_t;

static void put_cp(sink_t *s, uint32_t cp) {
  if (s->chars >= s->limit) { s->full = 1; return; }
  uint8_t b[4]; int n;
  if (cp < 0x80) { b[0] = (uint8_t)cp; n = 1; }
  else if (cp < 0x800) { b[0] = 0xC0 | (cp >> 6); b[1] = 0x80 | (cp & 63); n = 2; }
  else if (cp < 0x10000) { b[0] = 0xE0 | (cp >> 12); b[1] = 0x80 | ((cp >> 6) & 63); b[2] = 0x80 | (cp & 63); n = 3; }
  else { b[0] = 0xF0 | (cp >> 18); b[1] = 0x80 | ((cp >> 12) & 63); b[2] = 0x80 | ((cp >> 6) & 63); b[3] = 0x80 | (cp & 63); n = 4; }
  if (s->buf && s->len + n <= s->cap) memcpy(s->buf + s->len, b, (size_t)n);
  s->len += n;
  s->chars += 1;
}

/* ------------------------------------------------------ lexicon + Zipf */
typedef struct {
  int n;
  char (*words)[11];
  uint8_t *lens;
  double *cdf;              /* cumulative Zipf(1.1) weights, normalised */
} lexicon_t;

static void zipf_cdf(double *cdf, int n, double s) {
  double tot = 0.0;
  for (int k = 1; k <= n; ++k) { tot += det_exp(-s * det_log((double)k)); cdf[k - 1] = tot; }
  for (int k = 0; k < n; ++k) cdf[k] /= tot;
}

static int zipf_draw(pcg64_t *r, const double *cdf, int n) {
  double u = rnd_unit(r);
  int lo = 0, hi = n - 1;
  while (lo < hi) { int mid = (lo + hi) >> 1; if (cdf[mid] > u) hi = mid; else lo = mid + 1; }
  return lo;
}

static void lexicon_build(lexicon_t *lx, int n, uint64_t seed) {
  pcg64_t r; pcg_seed(&r, seed, 0x1e71c0);
  lx->n = n;
  lx->words = malloc(sizeof(*lx->words) * (size_t)n);
  lx->lens = malloc((size_t)n);
  lx->cdf = malloc(sizeof(double) * (size_t)n);
  for (int i = 0; i < n; ++i) {
    int len = 2 + (int)rnd_below(&r, 9);
    for (int j = 0; j < len; ++j) lx->words[i][j] = (char)('a' + rnd_below(&r, 26));
    lx->lens[i] = (uint8_t)len;
  }
  zipf_cdf(lx->cdf, n, 1.1);
}

static void lexicon_free(lexicon_t *lx) { free(lx->words); free(lx->lens); free(lx->cdf); }

/* ------------------------------------------------------ profile tables */
typedef struct {
  int lexicon;              /* words in the lexicon */
  double p_digits, p_punct, p_cjk, p_emoji, p_marks;
  double p_title, p_upper, p_camel, p_contraction, p_latin1, p_blank_run, p_attach;
  double p_glue;            /* a token follows the previous one with no separator */
  double p_kana;            /* a CJK token is kana rather than ideographs */
} profile_t;

static const profile_t PROFILES[4] = {
  /* 0: ASCII code-like text */
  {5000, 0.07, 0.10, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.14, 0.0, 0.0},
  /* 1: mixed UTF-8 */
  {50000, 0.065, 0.09, 0.034, 0.085, 0.0, 0.12, 0.04, 0.05, 0.03, 0.035, 0.02, 0.13, 0.0, 0.0},
  /* 2: as 1, with camelCase/PascalCase identifiers and combining marks */
  {50000, 0.055, 0.08, 0.036, 0.09, 0.14, 0.08, 0.03, 0.30, 0.03, 0.035, 0.02, 0.13, 0.0, 0.0},
  /* 3: as 1, with kana and ideograph runs often glued to words, digits and punctuation */
  {50000, 0.08, 0.10, 0.30, 0.01, 0.0, 0.08, 0.03, 0.0, 0.03, 0.02, 0.02, 0.10, 0.35, 0.4},
};

static const char PUNCT[] = "()[]{};:,.=+-*/<>!&|\"#%@$^~?_'`\\";
static const char *CONTRACTIONS[] = {"'s", "'t", "'re", "'ve", "'m", "'ll", "'d"};
/* Latin-1 letters U+00C0..U+00FF without the two operators U+00D7 and U+00F7 */
static uint32_t latin1_letter(pcg64_t *r) {
  for (;;) { uint32_t c = 0xC0 + (uint32_t)rnd_below(r, 64); if (c != 0xD7 && c != 0xF7) return c; }
}

typedef struct {
  pcg64_t r;
  const profile_t *pf;
  lexicon_t lx;
  double cjk_cdf[3000];
} gen_t;

static void put_word_cased(gen_t *g, sink_t *s, int w, int mode /*0 lower 1 title 2 upper*/, int latin) {
  const char *p = g->lx.words[w];
  for (int j = 0; j < g->lx.lens[w]; ++j) {
    uint32_t c = (uint32_t)p[j];
    if (mode == 2 || (mode == 1 && j == 0)) c = c - 'a' + 'A';
    if (latin && rnd_chance(&g->r, g->pf->p_latin1)) c = latin1_letter(&g->r);
    put_cp(s, c);
  }
}

/* one token; returns nothing, writes into the sink */
static void put_token(gen_t *g, sink_t *s) {
  const profile_t *pf = g->pf;
  pcg64_t *r = &g->r;
  double u = rnd_unit(r);
  int latin = pf->p_latin1 > 0.0;
  if ((u -= pf->p_digits) < 0) {
    int n = 1 + (int)rnd_below(r, 12);
    for (int i = 0; i < n; ++i) put_cp(s, (uint32_t)('0' + rnd_below(r, 10)));
    return;
  }
  if ((u -= pf->p_punct) < 0) {
    int n = 1 + (int)rnd_below(r, 3);
    for (int i = 0; i < n; ++i) put_cp(s, (uint32_t)PUNCT[rnd_below(r, sizeof(PUNCT) - 1)]);
    return;
  }
  if ((u -= pf->p_cjk) < 0) {
    int n = 2 + (int)rnd_below(r, 39);
    if (pf->p_kana > 0.0 && rnd_chance(r, pf->p_kana)) {
      /* hiragana / katakana, with a few of the blocks' marks, long-vowel sign and middle dot */
      static const uint32_t extra[] = {0x30FC, 0x30FB, 0x3099, 0x309B, 0x30FC, 0x309D};
      for (int i = 0; i < n; ++i) {
        uint64_t k = rnd_below(r, 100);
        put_cp(s, k < 50 ? 0x3041u + (uint32_t)rnd_below(r, 86)
                  : k < 94 ? 0x30A1u + (uint32_t)rnd_below(r, 90) : extra[rnd_below(r, 6)]);
      }
      return;
    }
    for (int i = 0; i < n; ++i) put_cp(s, 0x4E00u + (uint32_t)zipf_draw(r, g->cjk_cdf, 3000));
    return;
  }
  if ((u -= pf->p_emoji) < 0) {
    int n = 1 + (int)rnd_below(r, 3);
    for (int i = 0; i < n; ++i) put_cp(s, 0x1F300u + (uint32_t)rnd_below(r, 0x1FB00 - 0x1F300));
    return;
  }
  if ((u -= pf->p_marks) < 0) {            /* base letters each followed by 1-2 combining marks */
    int w = zipf_draw(r, g->lx.cdf, g->lx.n);
    for (int j = 0; j < g->lx.lens[w]; ++j) {
      put_cp(s, (uint32_t)g->lx.words[w][j]);
      int m = 1 + (int)rnd_below(r, 2);
      for (int k = 0; k < m; ++k) put_cp(s, 0x300u + (uint32_t)rnd_below(r, 0x70));
    }
    return;
  }
  /* identifier */
  if (rnd_chance(r, pf->p_attach * 0.5)) put_cp(s, (uint32_t)PUNCT[rnd_below(r, 12)]);  /* leading ( [ { ... */
  if (rnd_chance(r, pf->p_camel)) {
    int parts = 2 + (int)rnd_below(r, 2), pascal = (int)rnd_below(r, 2);
    for (int k = 0; k < parts; ++k)
      put_word_cased(g, s, zipf_draw(r, g->lx.cdf, g->lx.n), (k == 0 && !pascal) ? 0 : 1, latin);
  } else {
    int mode = 0;
    double c = rnd_unit(r);
    if (c < pf->p_title) mode = 1; else if (c < pf->p_title + pf->p_upper) mode = 2;
    put_word_cased(g, s, zipf_draw(r, g->lx.cdf, g->lx.n), mode, latin);
  }
  if (rnd_chance(r, pf->p_contraction)) {
    const char *c = CONTRACTIONS[rnd_below(r, 7)];
    for (; *c; ++c) put_cp(s, (uint32_t)*c);
  }
  if (rnd_chance(r, pf->p_attach)) {
    int n = 1 + (int)rnd_below(r, 2);
    for (int i = 0; i < n; ++i) put_cp(s, (uint32_t)PUNCT[rnd_below(r, sizeof(PUNCT) - 1)]);
  }
}

static void gen_init(gen_t *g, uint64_t seed, int profile) {
  g->pf = &PROFILES[profile];
  pcg_seed(&g->r, seed, 0x7e47);
  /* the lexicon depends on the profile only, so training text and test text share it */
  lexicon_build(&g->lx, g->pf->lexicon, 0x5eed0000ULL + (uint64_t)g->pf->lexicon);
  zipf_cdf(g->cjk_cdf, 3000, 1.1);
}

static void gen_lines(gen_t *g, sink_t *s) {
  pcg64_t *r = &g->r;
  while (!s->full) {
    int64_t line_start = s->chars;
    int indent = 4 * (int)rnd_below(r, 4);
    int target = 20 + (int)rnd_below(r, 81);
    for (int i = 0; i < indent; ++i) put_cp(s, ' ');
    int first = 1;
    while (!s->full && s->chars - line_start < target) {
      /* measure the next separator + token into a scratch sink, then copy if it fits */
      uint8_t tmp[512];
      sink_t t = {tmp, 0, sizeof(tmp), 0, 1 << 30, 0};
      if (!first && !(g->pf->p_glue > 0.0 && rnd_chance(r, g->pf->p_glue))) {
        if (rnd_chance(r, g->pf->p_blank_run)) {
          int n = 1 + (int)rnd_below(r, 64);
          for (int i = 0; i < n; ++i) put_cp(&t, rnd_below(r, 4) ? ' ' : '\t');
        } else {
          put_cp(&t, ' ');
        }
      }
      put_token(g, &t);
      if (s->chars - line_start + t.chars > 100 && !first) break;
      /* copy char by char so the exact char limit is honoured */
      int64_t i = 0;
      while (i < t.len && !s->full) {
        uint8_t b0 = tmp[i];
        int n = b0 < 0x80 ? 1 : b0 < 0xE0 ? 2 : b0 < 0xF0 ? 3 : 4;
        uint32_t cp = n == 1 ? b0 : n == 2 ? (uint32_t)(b0 & 31) << 6 | (tmp[i + 1] & 63)
                    : n == 3 ? (uint32_t)(b0 & 15) << 12 | (uint32_t)(tmp[i + 1] & 63) << 6 | (tmp[i + 2] & 63)
                    : (uint32_t)(b0 & 7) << 18 | (uint32_t)(tmp[i + 1] & 63) << 12 | (uint32_t)(tmp[i + 2] & 63) << 6 | (tmp[i + 3] & 63);
        put_cp(s, cp);
        i += n;
      }
      first = 0;
    }
    if (rnd_chance(r, 0.05)) put_cp(s, '\r');
    put_cp(s, '\n');
  }
}

/* Transcript text of exactly n_chars code points.  Returns the byte length;
 * bytes are written only if they fit in cap (call with out=NULL to size). */
int64_t synth_transcript(uint64_t seed, int64_t n_chars, int profile, uint8_t *out, int64_t cap) {
  if (profile < 0 || profile > 3 || n_chars < 0) return -1;
  gen_t g; gen_init(&g, seed, profile);
  sink_t s = {out, 0, out ? cap : 0, 0, n_chars, n_chars == 0};
  gen_lines(&g, &s);
  lexicon_free(&g.lx);
  return s.len;
}

/* Adversarial long request: profile-1 text interleaved with pathological
 * blocks: 10K-digit runs, 50K-space runs ending in a letter, repeated
 * "\r\n\r\n \n", 5K-char punctuation runs and 10K-char "a a a ..."
 * alternations.  Exactly n_chars code points. */
int64_t synth_adversarial(uint64_t seed, int64_t n_chars, uint8_t *out, int64_t cap) {
  if (n_chars < 0) return -1;
  gen_t g; gen_init(&g, seed, 1);
  sink_t s = {out, 0, out ? cap : 0, 0, n_chars, n_chars == 0};
  int64_t block = 0;
  while (!s.full) {
    /* a stretch of ordinary text */
    int64_t stretch = 60000 + (int64_t)rnd_below(&g.r, 120000);
    int64_t lim = s.limit;
    s.limit = s.chars + stretch < lim ? s.chars + stretch : lim;
    gen_lines(&g, &s);
    s.full = 0;
    s.limit = lim;
    if (s.chars >= s.limit) { s.full = 1; break; }
    switch (block++ % 5) {
      case 0: for (int i = 0; i < 10000; ++i) put_cp(&s, (uint32_t)('0' + rnd_below(&g.r, 10))); break;
      case 1: for (int i = 0; i < 49999; ++i) put_cp(&s, ' '); put_cp(&s, 'x'); break;
      case 2: for (int i = 0; i < 400; ++i) { const char *p = "\r\n\r\n \n"; for (; *p; ++p) put_cp(&s, (uint32_t)*p); } break;
      case 3: for (int i = 0; i < 5000; ++i) put_cp(&s, (uint32_t)PUNCT[rnd_below(&g.r, 20)]); break;
      case 4: for (int i = 0; i < 5000; ++i) { put_cp(&s, 'a'); put_cp(&s, ' '); } break;
    }
  }
  lexicon_free(&g.lx);
  return s.len;
}

/* n lengths log-uniform in [lo, hi] */
void synth_lengths_loguniform(uint64_t seed, int64_t n, int64_t lo, int64_t hi, int64_t *out) {
  pcg64_t r; pcg_seed(&r, seed, 0x10c0);
  double a = det_log((double)lo), b = det_log((double)hi);
  for (int64_t i = 0; i < n; ++i) {
    int64_t v = (int64_t)det_exp(a + (b - a) * rnd_unit(&r));
    out[i] = v < lo ? lo : v > hi ? hi : v;
  }
}

/* n lengths lognormal with the given median and sigma, capped at cap.  The
 * normal deviate is the Box-Muller radius times a cosine built from the unit
 * circle by rejection (no trigonometric library call). */
void synth_lengths_lognormal(uint64_t seed, int64_t n, double median, double sigma, int64_t cap, int64_t *out) {
  pcg64_t r; pcg_seed(&r, seed, 0x10e0);
  double mu = det_log(median);
  for (int64_t i = 0; i < n; ++i) {
    double x, y, q;
    do { x = 2.0 * rnd_unit(&r) - 1.0; y = 2.0 * rnd_unit(&r) - 1.0; q = x * x + y * y; } while (q >= 1.0 || q == 0.0);
    double z = x * sqrt(-2.0 * det_log(q) / q);      /* Marsaglia polar method */
    int64_t v = (int64_t)det_exp(mu + sigma * z);
    out[i] = v < 1 ? 1 : v > cap ? cap : v;
  }
}

/* ================================================================ trainer */
/* Greedy byte-level BPE training.  The corpus is cut into chunks by a crude
 * splitter (letters with one leading blank, digits in threes, punctuation with
 * one leading blank, blank runs, newline runs); identical chunks are counted
 * once with a weight.  Each step merges the most frequent adjacent pair
 * (ties: smallest (left, right)); the new symbol is 256 + step.  Training stops
 * at n_merges or when the best count falls below 2. */

typedef struct { uint64_t *keys; int32_t *vals; int64_t cap, n; } map_t;   /* u64 -> i32, open addressing */

static uint64_t mix64(uint64_t x) {
  x ^= x >> 33; x *= 0xff51afd7ed558ccdULL; x ^= x >> 33; x *= 0xc4ceb9fe1a85ec53ULL; x ^= x >> 33; return x;
}
static void map_init(map_t *m, int64_t cap) {
  m->cap = cap; m->n = 0;
  m->keys = malloc(sizeof(uint64_t) * (size_t)cap);
  m->vals = malloc(sizeof(int32_t) * (size_t)cap);
  for (int64_t i = 0; i < cap; ++i) m->keys[i] = UINT64_MAX;
}
static void map_free(map_t *m) { free(m->keys); free(m->vals); }
static int32_t *map_slot(map_t *m, uint64_t key, int create);
static void map_grow(map_t *m) {
  map_t n2; map_init(&n2, m->cap * 2);
  for (int64_t i = 0; i < m->cap; ++i)
    if (m->keys[i] != UINT64_MAX) *map_slot(&n2, m->keys[i], 1) = m->vals[i];
  map_free(m); *m = n2;
}
static int32_t *map_slot(map_t *m, uint64_t key, int create) {
  if (create && (m->n + 1) * 2 > m->cap) map_grow(m);
  uint64_t h = mix64(key) & (uint64_t)(m->cap - 1);
  for (;;) {
    if (m->keys[h] == key) return &m->vals[h];
    if (m->keys[h] == UINT64_MAX) {
      if (!create) return NULL;
      m->keys[h] = key; m->vals[h] = -1; m->n++;
      return &m->vals[h];
    }
    h = (h + 1) & (uint64_t)(m->cap - 1);
  }
}

/* crude chunk classes, by code point */
enum { CK_LET, CK_DIG, CK_BLANK, CK_NL, CK_OTH };
static int ck_class(uint32_t cp) {
  if ((cp | 32) >= 'a' && (cp | 32) <= 'z') return CK_LET;
  if (cp >= '0' && cp <= '9') return CK_DIG;
  if (cp == ' ' || cp == '\t') return CK_BLANK;
  if (cp == '\n' || cp == '\r') return CK_NL;
  if (cp < 0x80) return CK_OTH;
  if (cp >= 0x1F000 && cp < 0x20000) return CK_OTH;     /* pictographs */
  return CK_LET;                                          /* other non-ASCII: treated as letters */
}
/* with han_split, kana / CJK ideograph runs are chunks of their own */
enum { CK_HAN = 5 };
static int ck_class2(uint32_t cp, int han_split) {
  if (han_split && ((cp >= 0x3040 && cp <= 0x30FF) || (cp >= 0x4E00 && cp <= 0x9FFF))) return CK_HAN;
  return ck_class(cp);
}
static int ck_upper(uint32_t cp) { return (cp >= 'A' && cp <= 'Z') || (cp >= 0xC0 && cp <= 0xDE); }

typedef struct { int64_t start, len; } span_t;

static int64_t utf8_decode_all(const uint8_t *t, int64_t n, uint32_t *cps, int64_t *pos) {
  int64_t k = 0;
  for (int64_t i = 0; i < n;) {
    uint8_t b0 = t[i];
    int len = b0 < 0x80 ? 1 : b0 < 0xE0 ? 2 : b0 < 0xF0 ? 3 : 4;
    if (i + len > n) len = 1;
    uint32_t cp = len == 1 ? b0 : len == 2 ? (uint32_t)(b0 & 31) << 6 | (t[i + 1] & 63)
                 : len == 3 ? (uint32_t)(b0 & 15) << 12 | (uint32_t)(t[i + 1] & 63) << 6 | (t[i + 2] & 63)
                 : (uint32_t)(b0 & 7) << 18 | (uint32_t)(t[i + 1] & 63) << 12 | (uint32_t)(t[i + 2] & 63) << 6 | (t[i + 3] & 63);
    cps[k] = cp; pos[k] = i; ++k; i += len;
  }
  pos[k] = n;
  return k;
}

/* split into chunks (byte spans); case_split also cuts lower->Upper inside letter runs
 * and keeps a following 's/'t/... on the word */
static int64_t crude_chunks(const uint8_t *t, int64_t n, int flags, span_t **out) {
  const int case_split = flags & 1, han = (flags >> 1) & 1;
  uint32_t *cp = malloc(sizeof(uint32_t) * (size_t)(n + 1));
  int64_t *pos = malloc(sizeof(int64_t) * (size_t)(n + 2));
  int64_t m = utf8_decode_all(t, n, cp, pos);
  int64_t cap = m + 16, k = 0;
  span_t *sp = malloc(sizeof(span_t) * (size_t)cap);
#define EMIT(a, b) do { sp[k].start = pos[a]; sp[k].len = pos[b] - pos[a]; ++k; } while (0)
  int64_t i = 0;
  while (i < m) {
    int c = ck_class2(cp[i], han);
    int64_t j = i;
    if (c == CK_BLANK) {
      while (j < m && ck_class2(cp[j], han) == CK_BLANK) ++j;
      int nx = j < m ? ck_class2(cp[j], han) : CK_NL;
      if ((nx == CK_LET || nx == CK_OTH) && j - i >= 2) { EMIT(i, j - 1); i = j - 1; continue; }
      if (nx == CK_LET || nx == CK_OTH) { /* single blank joins the next chunk */
        int64_t s = i; i = j; c = nx; j = i;
        if (c == CK_LET) {
          while (j < m && ck_class2(cp[j], han) == CK_LET && !(case_split && j > i && ck_upper(cp[j]) && !ck_upper(cp[j - 1]))) ++j;
        } else {
          while (j < m && ck_class2(cp[j], han) == CK_OTH) ++j;
        }
        EMIT(s, j); i = j; continue;
      }
      EMIT(i, j); i = j; continue;
    }
    if (c == CK_HAN) { while (j < m && ck_class2(cp[j], han) == CK_HAN) ++j; EMIT(i, j); i = j; continue; }
    if (c == CK_NL) { while (j < m && ck_class2(cp[j], han) == CK_NL) ++j; EMIT(i, j); i = j; continue; }
    if (c == CK_DIG) { while (j < m && j - i < 3 && ck_class2(cp[j], han) == CK_DIG) ++j; EMIT(i, j); i = j; continue; }
    if (c == CK_LET) {
      ++j;
      while (j < m && ck_class2(cp[j], han) == CK_LET && !(case_split && ck_upper(cp[j]) && !ck_upper(cp[j - 1]))) ++j;
      if (case_split && j + 1 < m && cp[j] == '\'' && ck_class2(cp[j + 1], han) == CK_LET) j += 2;
      EMIT(i, j); i = j; continue;
    }
    /* other */
    while (j < m && ck_class2(cp[j], han) == CK_OTH) ++j;
    EMIT(i, j); i = j;
  }
#undef EMIT
  free(cp); free(pos);
  *out = sp;
  return k;
}

/* max-heap of (count, pair) with lazy deletion */
typedef struct { int64_t count; uint64_t pair; } hent_t;
typedef struct { hent_t *a; int64_t n, cap; } heap_t;
static int hbetter(const hent_t *x, const hent_t *y) {   /* x before y ? */
  if (x->count != y->count) return x->count > y->count;
  return x->pair < y->pair;                              /* (left,right) packed left<<32|right */
}
static void hpush(heap_t *h, int64_t count, uint64_t pair) {
  if (h->n == h->cap) { h->cap = h->cap ? h->cap * 2 : 1024; h->a = realloc(h->a, sizeof(hent_t) * (size_t)h->cap); }
  int64_t i = h->n++;
  hent_t e = {count, pair};
  while (i > 0) { int64_t p = (i - 1) / 2; if (!hbetter(&e, &h->a[p])) break; h->a[i] = h->a[p]; i = p; }
  h->a[i] = e;
}
static hent_t hpop(heap_t *h) {
  hent_t top = h->a[0], last = h->a[--h->n];
  int64_t i = 0;
  for (;;) {
    int64_t l = 2 * i + 1, r = l + 1, b = i;
    const hent_t *bv = &last;
    if (l < h->n && hbetter(&h->a[l], bv)) { b = l; bv = &h->a[l]; }
    if (r < h->n && hbetter(&h->a[r], bv)) { b = r; bv = &h->a[r]; }
    if (b == i) break;
    h->a[i] = h->a[b]; i = b;
  }
  if (h->n) h->a[i] = last;
  return top;
}

typedef struct { int32_t *ids; int32_t len; int64_t count; int64_t stamp; } word_t;
typedef struct { int32_t *w; int32_t n, cap; } wlist_t;

typedef struct {
  map_t pidx;               /* pair -> index into counts/lists */
  int64_t *counts;
  wlist_t *lists;
  int64_t np, capp;
} pairs_t;

static int32_t pair_index(pairs_t *P, uint64_t pair) {
  int32_t *s = map_slot(&P->pidx, pair, 1);
  if (*s < 0) {
    if (P->np == P->capp) {
      P->capp = P->capp ? P->capp * 2 : 1 << 16;
      P->counts = realloc(P->counts, sizeof(int64_t) * (size_t)P->capp);
      P->lists = realloc(P->lists, sizeof(wlist_t) * (size_t)P->capp);
    }
    P->counts[P->np] = 0;
    P->lists[P->np].w = NULL; P->lists[P->np].n = 0; P->lists[P->np].cap = 0;
    *s = (int32_t)P->np++;
  }
  return *s;
}
static void wlist_add(wlist_t *l, int32_t w) {
  if (l->n && l->w[l->n - 1] == w) return;
  if (l->n == l->cap) { l->cap = l->cap ? l->cap * 2 : 4; l->w = realloc(l->w, sizeof(int32_t) * (size_t)l->cap); }
  l->w[l->n++] = w;
}
#define PAIR(a, b) (((uint64_t)(uint32_t)(a) << 32) | (uint32_t)(b))

int64_t synth_train_bpe(const uint8_t *text, int64_t len, int64_t n_merges, int flags, int32_t *out_pairs) {
  span_t *sp;
  int64_t nch = crude_chunks(text, len, flags, &sp);
  /* unique chunks with counts: hash of bytes -> word index (collisions resolved by compare) */
  map_t wmap; map_init(&wmap, 1 << 20);
  word_t *words = NULL; int64_t nw = 0, capw = 0;
  for (int64_t c = 0; c < nch; ++c) {
    const uint8_t *b = text + sp[c].start; int64_t L = sp[c].len;
    uint64_t h = 1469598103934665603ULL;
    for (int64_t i = 0; i < L; ++i) { h ^= b[i]; h *= 1099511628211ULL; }
    h ^= (uint64_t)L; if (h == UINT64_MAX) h = 0;
    for (;;) {                                   /* probe sequence over h, h+1, ... on collisions */
      int32_t *s = map_slot(&wmap, h, 1);
      if (*s < 0) {
        if (nw == capw) { capw = capw ? capw * 2 : 1 << 16; words = realloc(words, sizeof(word_t) * (size_t)capw); }
        words[nw].ids = malloc(sizeof(int32_t) * (size_t)L);
        for (int64_t i = 0; i < L; ++i) words[nw].ids[i] = b[i];
        words[nw].len = (int32_t)L; words[nw].count = 1; words[nw].stamp = -1;
        *s = (int32_t)nw++;
        break;
      }
      word_t *w = &words[*s];
      int same = w->len == L;
      for (int64_t i = 0; same && i < L; ++i) same = w->ids[i] == b[i];
      if (same) { w->count++; break; }
      h = h + 0x9E3779B97F4A7C15ULL; if (h == UINT64_MAX) h = 0;
    }
  }
  free(sp); map_free(&wmap);

  pairs_t P; memset(&P, 0, sizeof(P)); map_init(&P.pidx, 1 << 20);
  for (int64_t w = 0; w < nw; ++w)
    for (int32_t i = 0; i + 1 < words[w].len; ++i) {
      int32_t pi = pair_index(&P, PAIR(words[w].ids[i], words[w].ids[i + 1]));
      P.counts[pi] += words[w].count;
      wlist_add(&P.lists[pi], (int32_t)w);
    }
  heap_t H = {0};
  for (int64_t s = 0; s < P.pidx.cap; ++s)
    if (P.pidx.keys[s] != UINT64_MAX) hpush(&H, P.counts[P.pidx.vals[s]], P.pidx.keys[s]);

  int32_t *tmp = NULL; int64_t tmpcap = 0;
  int64_t done = 0;
  /* scratch for net deltas of one word */
  uint64_t *dk = NULL; int64_t *dv = NULL; int64_t dcap = 0;
  while (done < n_merges && H.n) {
    hent_t top = hpop(&H);
    int32_t *ps = map_slot(&P.pidx, top.pair, 0);
    if (!ps || P.counts[*ps] != top.count) continue;       /* stale */
    if (top.count < 2) break;
    int32_t a = (int32_t)(top.pair >> 32), b = (int32_t)(uint32_t)top.pair, X = 256 + (int32_t)done;
    out_pairs[2 * done] = a; out_pairs[2 * done + 1] = b;
    int32_t pidx = *ps;
    wlist_t lst = P.lists[pidx];
    P.lists[pidx].w = NULL; P.lists[pidx].n = P.lists[pidx].cap = 0;
    for (int32_t li = 0; li < lst.n; ++li) {
      word_t *w = &words[lst.w[li]];
      if (w->stamp == done) continue;
      w->stamp = done;
      int32_t L = w->len, has = 0;
      for (int32_t i = 0; i + 1 < L; ++i) if (w->ids[i] == a && w->ids[i + 1] == b) { has = 1; break; }
      if (!has) continue;
      if (tmpcap < L) { tmpcap = L * 2; tmp = realloc(tmp, sizeof(int32_t) * (size_t)tmpcap); }
      int32_t nl = 0;
      for (int32_t i = 0; i < L;) {
        if (i + 1 < L && w->ids[i] == a && w->ids[i + 1] == b) { tmp[nl++] = X; i += 2; }
        else tmp[nl++] = w->ids[i++];
      }
      /* net pair deltas: -old pairs, +new pairs */
      if (dcap < 2 * L) { dcap = 4 * L; dk = realloc(dk, sizeof(uint64_t) * (size_t)dcap); dv = realloc(dv, sizeof(int64_t) * (size_t)dcap); }
      int64_t nd = 0;
      for (int pass = 0; pass < 2; ++pass) {
        const int32_t *ids = pass ? tmp : w->ids; int32_t n = pass ? nl : L;
        for (int32_t i = 0; i + 1 < n; ++i) {
          uint64_t k = PAIR(ids[i], ids[i + 1]);
          int64_t j = 0; while (j < nd && dk[j] != k) ++j;
          if (j == nd) { dk[nd] = k; dv[nd] = 0; ++nd; }
          dv[j] += pass ? w->count : -w->count;
        }
      }
      memcpy(w->ids, tmp, sizeof(int32_t) * (size_t)nl);
      w->len = nl;
      for (int64_t j = 0; j < nd; ++j) {
        if (dv[j] == 0) continue;
        int32_t pi = pair_index(&P, dk[j]);
        P.counts[pi] += dv[j];
        if (dv[j] > 0) wlist_add(&P.lists[pi], (int32_t)(w - words));
        if (dk[j] != top.pair && P.counts[pi] > 0) hpush(&H, P.counts[pi], dk[j]);
      }
    }
    free(lst.w);
    P.counts[pidx] = 0;
    ++done;
  }
  free(tmp); free(dk); free(dv); free(H.a);
  for (int64_t p = 0; p < P.np; ++p) free(P.lists[p].w);
  free(P.lists); free(P.counts); map_free(&P.pidx);
  for (int64_t w = 0; w < nw; ++w) free(words[w].ids);
  free(words);
  return done;
}
