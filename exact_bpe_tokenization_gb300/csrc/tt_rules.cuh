// tt_rules.cuh - run-local piece-start rules of the pattern families.
//
// TokTier: Exact Stateful CPU+GPU Tokenization for Agentic LLM Serving, §4.1
// (the run decomposition): each character gets one of four classes (letter,
// number, whitespace, other); whether it begins a piece depends only on its
// offset in its maximal same-class run, at most four characters of lookback
// across the run boundary, and per-run aggregates (run start, first non-CRLF,
// last CRLF) that prefix scans provide.  The o200k lineage adds a case rule,
// a contraction path and a narrow fallback for combining marks.
//
// This file holds the rules as pure functions of a character's neighbourhood
// (`Nbr`) and of the scan results at that character (`Aggs`), plus the scan
// events each character contributes.  The kernels compute neighbourhoods and
// scans in parallel; the functions are also compiled for the host so the
// rules can be unit-tested in isolation.
//
// The rules were derived alternative by alternative from the families'
// definitions (see include/toktier.h for the families):
//   cl100k-style:  '(s|t|re|ve|m|ll|d) | [^\r\n L N]?L+ | N{1,3} |
//                   ?[^\s L N]+[\r\n]* | \s*[\r\n]+ | \s+(?!\S) | \s+
//   o200k-style:   [^\r\n L N]?U*W+K? | [^\r\n L N]?U+W*K? | (the rest as above)
//                  U = Lu Lt Lm Lo M,  W = Ll Lm Lo M,  K = optional contraction
//   deepseek-style: three splitters in sequence, each re-splitting every
//                   piece of the one before, the stretches between matches
//                   kept as pieces: N{1,3}, then runs of kana / CJK
//                   ideographs (U+3040-30FF, U+4E00-9FFF), then the
//                   cl100k-style alternatives without N{1,3}
//
// Derived rules (a "run" is a maximal stretch of one effective class inside
// one request; s = run start, e = run end):
//   number run:   starts at s, s+3, s+6, ...
//   other run:    starts at s unless the char before is U+0020 (it joins the
//                 blank's piece).  o200k: a lone apostrophe right after
//                 letters and followed by a contraction is absorbed too.
//                 The piece swallows the CR/LF chars that follow the run.
//   blank run:    r0 = first non-CRLF if the run follows an "other" run
//                 (the CR/LFs before it were swallowed), else s; r0 starts;
//                 lc+1 starts if lc (the run's last CR/LF) is >= r0 and
//                 lc+1 < e; e-1 starts if the non-CRLF tail has >= 2 chars
//                 and the run is not at the request end.
//   letter run:   s starts unless the char before is a non-CRLF blank or a
//                 one-char "other" run that itself starts a piece (it is the
//                 optional prefix).  After a one-char apostrophe run that
//                 takes a contraction, the first letter after the
//                 contraction letters starts.  o200k: an upper-case letter
//                 starts when the nearest preceding cased letter of its
//                 segment is lower-case, or when it follows a caseless letter
//                 (Lm/Lo/M) and only upper-case letters follow up to the run
//                 end (the U*W+ backtracking rule).
//   o200k marks:  a mark is a caseless letter, except inside a stretch of
//                 other/mark chars after the stretch has had two adjacent
//                 "other" chars or began with a blank-prefixed "other": from
//                 there on the "other" piece swallows marks.
//   o200k contraction chain: an apostrophe after letters is swallowed as the
//                 preceding piece's contraction suffix only if that piece
//                 ended with its letter part.  A letter run made up of exactly
//                 the letters of a swallowed contraction ends its piece with
//                 the contraction instead, so in x'd'd'd... the apostrophes
//                 alternate between swallowed and piece-starting.  The state
//                 "the last letter run ended with its letter part" is carried
//                 by a scan over the functions {identity, not, true, false}.
//   deepseek-style: the first two splitters cut a request into segments at
//                 every change between digits, kana/CJK chars and the rest,
//                 and into digit groups of three (the number-run rule).  A
//                 segment is the third splitter's whole subject, so its start
//                 acts exactly like a request start: the cl100k-style rules
//                 apply unchanged once segment starts are flagged like
//                 request starts (lookback and lookahead stop there, a blank
//                 run's lookahead sees the segment end as the text end).
//                 The paper (§4.1) names this composition property; the
//                 digit groups need no flag since digits only ever meet
//                 digits inside a segment.
#pragma once
#include <stdint.h>

#ifndef TT_HD
#if defined(__CUDACC__)
#define TT_HD __host__ __device__ __forceinline__
#else
#define TT_HD inline
#endif
#endif

namespace tt {

// raw / effective character kinds
enum : uint8_t { K_OTHER = 0, K_LU = 1, K_LL = 2, K_LB = 3, K_MARK = 4, K_NUM = 5, K_WS = 6, K_NONE = 7,
                 K_LIT = 8 };   // K_LIT: a char of an added-token literal after its first (never starts a piece)
// deepseek-style tables flag kana / CJK ideograph chars in the raw kind
enum : uint8_t { K_HAN_FLAG = 0x10, K_KIND_MASK = 0x0F };
enum : int { FAM_CL100K = 1, FAM_O200K = 2, FAM_DEEPSEEK = 3 };
// results of the "first char after i" queries
enum : uint8_t { R_END = 0, R_CRLF = 1, R_OTHER = 2, R_LETTER = 3 };

TT_HD bool is_letter(uint8_t k) { return k >= K_LU && k <= K_LB; }
TT_HD bool is_crlf(uint32_t c) { return c == 10u || c == 13u; }
TT_HD uint32_t lower_ascii(uint32_t c) { return (c >= 'A' && c <= 'Z') ? c + 32u : c; }
// contraction letters after an apostrophe, ASCII case folding:
// one-letter: s t m d ; two-letter: re ve ll
TT_HD bool contraction1(uint32_t a) {
  a = lower_ascii(a);
  return a == 's' || a == 't' || a == 'm' || a == 'd';
}
TT_HD bool contraction2(uint32_t a, uint32_t b) {
  a = lower_ascii(a); b = lower_ascii(b);
  return (a == 'r' && b == 'e') || (a == 'v' && b == 'e') || (a == 'l' && b == 'l');
}
// the contraction an apostrophe would take given the next two chars (0 = none)
TT_HD int contraction_after(uint32_t n1, uint32_t n2) {
  if (contraction1(n1)) return 1;
  if (contraction2(n1, n2)) return 2;
  return 0;
}

// Neighbourhood of char i inside its request.  Outside the request (or the
// batch) classes read K_NONE and code points read 0.
struct Nbr {
  uint8_t e0, e1, e2, e3, e4;      // effective kinds of i, i-1, .., i-4
  uint32_t c0, c1, c2, c3, c4;     // code points of i, i-1, .., i-4
  uint8_t en1, en2;                // effective kinds of i+1, i+2
  uint32_t cn1, cn2;               // code points of i+1, i+2
  bool rs;                         // i is the first char of its request
  bool l1, l2, l3;                 // o200k chain state after chars i-1, i-2, i-3:
                                   // "the last letter run ended with its letter part"
};

// Scan results at char i.
struct Aggs {
  int nidx3;          // (index of i inside its number run) mod 3
  bool w_start;       // i is the first char of its blank run
  bool w_prev_other;  // the char before i's blank run is "other"
  bool w_ncw_before;  // a non-CRLF blank precedes i inside its run
  int case_prev;      // o200k: last cased letter of i's segment before i: 0 none, 1 upper, 2 lower
  uint8_t rq_ws;      // first char after i that is not a non-CRLF blank: R_CRLF / R_END / R_OTHER
  uint8_t rq_up;      // first char after i that is not upper-case: R_LETTER / R_END / R_OTHER
};

// i ends a contraction that started right after an apostrophe which itself
// was a lone "other" char at a piece start (cl100k) / followed letters (o200k)
TT_HD bool contraction_end(int fam, const Nbr &n) {
  if (!is_letter(n.e1)) return false;
  if (fam != FAM_O200K) {   // cl100k-style and deepseek-style
    if (n.c2 == '\'' && n.e2 == K_OTHER && contraction1(n.c1) && n.e3 != K_OTHER && n.c3 != ' ') return true;
    if (n.c3 == '\'' && n.e3 == K_OTHER && is_letter(n.e2) && contraction2(n.c2, n.c1) && n.e4 != K_OTHER &&
        n.c4 != ' ')
      return true;
    return false;
  }
  if (n.c2 == '\'' && n.e2 == K_OTHER && contraction1(n.c1) && is_letter(n.e3) && n.l2) return true;
  if (n.c3 == '\'' && n.e3 == K_OTHER && is_letter(n.e2) && contraction2(n.c2, n.c1) && is_letter(n.e4) && n.l3)
    return true;
  return false;
}

// The piece-start predicate.  Requires: char i belongs to a valid request.
TT_HD bool piece_start(int fam, const Nbr &n, const Aggs &a) {
  if (n.rs) return true;
  const uint8_t e = n.e0;
  if (e == K_LIT) return false;
  if (e == K_NUM) return a.nidx3 == 0;
  if (e == K_WS) {
    const bool crlf0 = is_crlf(n.c0);
    if (a.w_start) return !(a.w_prev_other && crlf0);
    if (crlf0) return false;
    if (a.w_prev_other && !a.w_ncw_before) return true;                 // r0 after swallowed CR/LFs
    if (is_crlf(n.c1) && a.rq_ws != R_CRLF) return true;                 // lc + 1
    if (n.en1 != K_WS && n.en1 != K_NONE && !is_crlf(n.c1)) return true; // e - 1 (lookahead)
    return false;
  }
  if (e == K_OTHER) {
    if (n.e1 == K_OTHER) return false;
    if (n.c1 == ' ') return false;
    if (fam == FAM_O200K && n.c0 == '\'' && is_letter(n.e1) && n.l1 && contraction_after(n.cn1, n.cn2)) return false;
    return true;
  }
  // letters
  if (!is_letter(n.e1)) {
    const bool absorbed = (n.e1 == K_WS && !is_crlf(n.c1)) || (n.e1 == K_OTHER && n.e2 != K_OTHER && n.c2 != ' ');
    return !absorbed;
  }
  if (contraction_end(fam, n)) return true;
  if (fam == FAM_O200K && e == K_LU) {
    // the second letter of a swallowed two-letter contraction belongs to the previous piece
    if (n.c2 == '\'' && n.e2 == K_OTHER && is_letter(n.e3) && n.l2 && contraction2(n.c1, n.c0)) return false;
    if (a.case_prev == 2) return true;
    if (n.e1 == K_LB && a.rq_up != R_LETTER) return true;
  }
  return false;
}

// The families without a case rule: the predicate reads of a char's
// neighbourhood only rs, e0, e1, c0, c1, en1 and cn1, except for a letter
// after an "other" char (the optional-prefix rule reads e2 and c2) or after
// a letter (the contraction rules read two to four chars back).  Where this
// is false, a neighbourhood holding just those fields decides exactly.
TT_HD bool needs_far_nbr(uint8_t e0, uint8_t e1) { return is_letter(e0) && (e1 == K_OTHER || is_letter(e1)); }

// ---------------------------------------------------------------- events
// o200k mark resolution ("scan 1"), on raw kinds.  An other/mark stretch
// starts at j; a trigger at j switches the rest of its stretch to "other".
TT_HD bool om_kind(uint8_t raw) { return raw == K_OTHER || raw == K_MARK; }
TT_HD bool region_start(uint8_t raw0, uint8_t raw_prev /*K_NONE at request start*/) {
  return om_kind(raw0) && !om_kind(raw_prev);
}
TT_HD bool trigger(uint8_t raw0, uint8_t raw_prev, uint32_t cp_prev, uint8_t raw_next) {
  if (raw0 != K_OTHER) return false;
  if (raw_next == K_OTHER) return true;
  return region_start(raw0, raw_prev) && cp_prev == ' ';
}
// effective kind of a char from its raw kind and (for marks) the resolution
TT_HD uint8_t effective(int fam, uint8_t raw, bool mark_is_other) {
  raw &= K_KIND_MASK;
  if (raw != K_MARK) return raw;
  return (fam == FAM_O200K && !mark_is_other) ? K_LB : K_OTHER;
}

// o200k contraction chain.  A function on the chain state is two bits:
// bit 0 = f(false), bit 1 = f(true).
enum : uint8_t { CH_FALSE = 0, CH_NOT = 1, CH_ID = 2, CH_TRUE = 3 };
TT_HD uint8_t chain_apply(uint8_t f, bool x) { return (f >> (x ? 1 : 0)) & 1; }
TT_HD uint8_t chain_then(uint8_t f, uint8_t g) {   // g after f
  return (uint8_t)(chain_apply(g, chain_apply(f, false)) | (chain_apply(g, chain_apply(f, true)) << 1));
}
// the transition char i applies: at the start of a letter run that is made up
// of exactly the letters of a contraction after an apostrophe that follows
// letters, the state flips (the run's piece ends with the contraction iff
// the apostrophe was swallowed); at any other letter-run start it becomes
// true; elsewhere nothing changes.
TT_HD uint8_t chain_event(int fam, const Nbr &n) {
  if (fam != FAM_O200K || !is_letter(n.e0) || is_letter(n.e1)) return CH_ID;
  if (n.e1 == K_OTHER && n.c1 == '\'' && is_letter(n.e2)) {
    const int k = contraction_after(n.c0, n.cn1);
    if ((k == 1 && !is_letter(n.en1)) || (k == 2 && !is_letter(n.en2))) return CH_NOT;
  }
  return CH_TRUE;
}

// ------------------------------------------------------------ scan 2
// One associative scan carries every forward aggregate the predicate needs:
//   number runs: segmented count (reset at a run start), mod 3;
//   blank runs:  latest run start, packed (pos << 1 | "after an other run"),
//                and the latest non-CRLF blank position (max-scans);
//   o200k:       the contraction chain as a function f on its bit, and the
//                latest case event (pos << 2 | 0 segment start, 1 upper,
//                2 lower) as a max for each incoming chain bit.
// A char's element depends only on the state just before it, so prefixes
// compose: combine(a, b) = "a, then b".
struct S2 {
  int32_t wst, ncw;        // max-scans, -1 = none
  int32_t case0, case1;    // case max given chain bit false / true on entry
  uint8_t nflag, ncount;   // number runs: a reset happened; count since it (mod 3)
  uint8_t chain, pad;      // chain function (CH_*)
};
// Positions are byte offsets below 2^29, so pos * 4 + type fits an int32.
constexpr int64_t S2_MAX_POS = (int64_t)1 << 29;

TT_HD S2 s2_identity() {
  S2 r;
  r.wst = r.ncw = r.case0 = r.case1 = -1;
  r.nflag = r.ncount = 0;
  r.chain = CH_ID;
  r.pad = 0;
  return r;
}
TT_HD int32_t max32(int32_t a, int32_t b) { return a > b ? a : b; }
TT_HD S2 s2_combine(const S2 &a, const S2 &b) {
  S2 r;
  r.nflag = a.nflag | b.nflag;
  r.ncount = b.nflag ? b.ncount : (uint8_t)((a.ncount + b.ncount) % 3);
  r.wst = max32(a.wst, b.wst);
  r.ncw = max32(a.ncw, b.ncw);
  r.chain = chain_then(a.chain, b.chain);
  r.case0 = max32(a.case0, chain_apply(a.chain, false) ? b.case1 : b.case0);
  r.case1 = max32(a.case1, chain_apply(a.chain, true) ? b.case1 : b.case0);
  r.pad = 0;
  return r;
}

// The element of char i.  pos: byte position of i; pos1 / pos2: byte
// positions of chars i+1 / i+2 (used only when they exist).
TT_HD S2 s2_element(int fam, const Nbr &n, int32_t pos, int32_t pos1, int32_t pos2) {
  S2 r = s2_identity();
  if (n.e0 == K_NUM) {
    r.nflag = n.e1 != K_NUM;
    r.ncount = 1;
  }
  if (n.e0 == K_WS) {
    if (n.e1 != K_WS) r.wst = pos * 2 + (n.e1 == K_OTHER ? 1 : 0);
    if (!is_crlf(n.c0)) r.ncw = pos;
  }
  if (fam == FAM_O200K && is_letter(n.e0)) {
    const bool run_start = !is_letter(n.e1);
    const int t = n.e0 == K_LU ? 1 : n.e0 == K_LL ? 2 : 0;
    const int32_t ev = (run_start || t) ? pos * 4 + t : -1;
    r.case0 = r.case1 = ev;
    if (run_start) {
      r.chain = CH_TRUE;
      if (n.e1 == K_OTHER && n.c1 == '\'' && is_letter(n.e2)) {
        const int k = contraction_after(n.c0, n.cn1);
        const uint8_t ek = k == 1 ? n.en1 : n.en2;
        if (k && !is_letter(ek)) {
          r.chain = CH_NOT;                       // the run is exactly the contraction letters
        } else if (k) {
          // if the apostrophe is swallowed (chain bit true), a new segment
          // starts after the contraction letters
          const int tk = ek == K_LU ? 1 : ek == K_LL ? 2 : 0;
          r.case1 = max32(ev, (k == 1 ? pos1 : pos2) * 4 + tk);
        }
      }
    }
  }
  return r;
}

// True when char i's element is the identity (most chars): nothing to combine.
TT_HD bool s2_trivial(int fam, const Nbr &n) {
  return n.e0 != K_NUM && n.e0 != K_WS && !(fam == FAM_O200K && is_letter(n.e0));
}

// Per-char aggregates from the state before char i and the state after it
// (before combined with i's element).  The chain bit is true before the
// first char of the batch.
TT_HD void s2_values(const S2 &before, const S2 &after, int32_t pos, Aggs &a, bool &chain_after) {
  a.nidx3 = (after.ncount + 2) % 3;
  const int32_t s = after.wst >> 1;
  a.w_start = s == pos;
  a.w_prev_other = (after.wst & 1) != 0;
  a.w_ncw_before = before.ncw >= s;
  const int32_t ce = before.case1;                 // exclusive, chain bit true on entry
  a.case_prev = ce >= 0 ? (int)(ce & 3) : 0;
  chain_after = chain_apply(after.chain, true) != 0;
}

// The forward aggregates of the families without a case rule (cl100k- and
// deepseek-style): S2 without its o200k fields, in 12 bytes.
struct S2L {
  int32_t wst, ncw;        // as in S2
  uint32_t num;            // number runs: bit 2 = a reset happened, bits 0..1 = count since it (mod 3)
};
TT_HD S2L s2l_identity() {
  S2L r;
  r.wst = r.ncw = -1;
  r.num = 0;
  return r;
}
TT_HD S2L s2l_combine(const S2L &a, const S2L &b) {
  S2L r;
  r.wst = max32(a.wst, b.wst);
  r.ncw = max32(a.ncw, b.ncw);
  if (b.num & 4u) {
    r.num = b.num;
  } else {
    const uint32_t c = (a.num & 3u) + (b.num & 3u);
    r.num = (a.num & 4u) | (c >= 3u ? c - 3u : c);
  }
  return r;
}
// the element of char i from its effective kind e0, its predecessor's e1
// (K_NONE at a request start), its code point c0 and byte position pos;
// the identity unless i is a digit or a blank
TT_HD S2L s2l_element(uint8_t e0, uint8_t e1, uint32_t c0, int32_t pos) {
  S2L r = s2l_identity();
  if (e0 == K_NUM) r.num = (e1 != K_NUM ? 4u : 0u) | 1u;
  if (e0 == K_WS) {
    if (e1 != K_WS) r.wst = pos * 2 + (e1 == K_OTHER ? 1 : 0);
    if (!is_crlf(c0)) r.ncw = pos;
  }
  return r;
}
// the aggregates s2_values gives, from S2L states (no case rule, chain true)
TT_HD void s2l_values(const S2L &before, const S2L &after, int32_t pos, Aggs &a) {
  a.nidx3 = (int)(((after.num & 3u) + 2u) % 3u);
  const int32_t s = after.wst >> 1;
  a.w_start = s == pos;
  a.w_prev_other = (after.wst & 1) != 0;
  a.w_ncw_before = before.ncw >= s;
  a.case_prev = 0;
}

// deepseek-style segments: 0 the rest, 1 digits, 2 kana / CJK ideographs
// (raw kinds; an added-token literal's inner chars are never cut)
TT_HD int ds_segment_class(uint8_t raw) {
  return (raw & K_HAN_FLAG) ? 2 : (raw == K_NUM ? 1 : 0);
}
// char j (raw kind raw_j, not the first of its request) starts a segment
TT_HD bool ds_segment_start(uint8_t raw_prev, uint8_t raw_j) {
  return raw_j != K_LIT && ds_segment_class(raw_prev) != ds_segment_class(raw_j);
}

// reverse-query events: what a char at j means to queries from before j.
// deepseek-style: a digit or kana/CJK char met by a blank run's lookahead
// starts a segment (the blank run's piece ends with its segment), so it reads
// as the end; elsewhere those chars are never the first event a blank sees.
// Bit k (k < 4) = the top bit of byte k of w (little-endian): the four top
// bits, shifted down to bits 0, 8, 16, 24, are gathered by one multiply whose
// partial products (at 0/7/14/21 + 8k) never overlap, so nothing carries.
TT_HD uint32_t top_bits4(uint32_t w) { return (((w & 0x80808080u) >> 7) * 0x204081u) >> 21 & 0xFu; }

TT_HD uint8_t rq_ws_event(int fam, bool rs_j, uint8_t raw_j, uint32_t cp_j) {  // 0xFF = not an event
  if (rs_j) return R_END;
  if (fam == FAM_DEEPSEEK && ds_segment_class(raw_j) != 0) return R_END;
  if (raw_j != K_WS) return R_OTHER;
  return is_crlf(cp_j) ? R_CRLF : 0xFF;
}
TT_HD uint8_t rq_up_event(bool rs_j, uint8_t raw_j) {
  if (rs_j) return R_END;
  if (raw_j == K_LU) return 0xFF;
  return (raw_j == K_LL || raw_j == K_LB || raw_j == K_MARK) ? R_LETTER : R_OTHER;
}

}  // namespace tt
