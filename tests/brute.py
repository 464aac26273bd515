"""Independent brute-force checkers for the oracle (test infrastructure).

1. A generic backtracking regex matcher over a small AST, written here from
   the textbook semantics of ordered alternation, greedy quantifiers with
   backtracking and negative lookahead.  The two pattern families are written
   as ASTs; pieces are found the way a leftmost-first regex scanner finds
   them (TokTier, §4.1: the patterns are ordered alternatives tried
   leftmost-first, with backtracking).  It shares nothing with oracle.c but
   the frozen class table.
2. The textbook BPE definition: every step rescans all adjacent pairs, takes
   the lowest rank and merges its leftmost occurrence (TokTier, §4.2).
3. The same pattern families as pattern strings for the installed `regex`
   module (a library run, used as a second cross-check where installed).
4. The deepseek-style family's three splitters, run one after another by a
   plain split driver over either matcher.
"""
import sys

sys.setrecursionlimit(100000)

B_L, B_LU, B_LL, B_LT, B_LM, B_LO, B_M, B_N, B_S = (1 << i for i in range(9))


# ----------------------------------------------------------------- AST nodes
class Node:
    pass


class Cls(Node):            # one char satisfying pred(cp)
    def __init__(self, pred):
        self.pred = pred


class Lit(Node):            # literal string, optionally ASCII case-insensitive
    def __init__(self, s, ci=False):
        self.s, self.ci = s, ci


class Seq(Node):
    def __init__(self, *items):
        self.items = items


class Alt(Node):            # ordered alternation
    def __init__(self, *items):
        self.items = items


class Rep(Node):            # greedy {lo, hi}; hi None = unbounded
    def __init__(self, item, lo, hi):
        self.item, self.lo, self.hi = item, lo, hi


class NegLook(Node):        # (?!item)
    def __init__(self, item):
        self.item = item


def _m(node, s, i, k):
    """Try node at s[i:]; call k(j) for each way it can end at j, in the
    regex's priority order; return the first non-None result."""
    if isinstance(node, Cls):
        return k(i + 1) if i < len(s) and node.pred(ord(s[i])) else None
    if isinstance(node, Lit):
        t = s[i:i + len(node.s)]
        ok = (t.lower() == node.s.lower()) if node.ci else (t == node.s)
        # ASCII-only folding
        if node.ci and ok and any(ord(c) > 127 for c in t):
            ok = False
        return k(i + len(node.s)) if ok and len(t) == len(node.s) else None
    if isinstance(node, Seq):
        def run(idx, pos):
            if idx == len(node.items):
                return k(pos)
            return _m(node.items[idx], s, pos, lambda j: run(idx + 1, j))
        return run(0, i)
    if isinstance(node, Alt):
        for it in node.items:
            r = _m(it, s, i, k)
            if r is not None:
                return r
        return None
    if isinstance(node, Rep):
        def rep(count, pos):
            if node.hi is None or count < node.hi:          # greedy: one more first
                r = _m(node.item, s, pos, lambda j: rep(count + 1, j) if j > pos else None)
                if r is not None:
                    return r
            return k(pos) if count >= node.lo else None
        return rep(0, i)
    if isinstance(node, NegLook):
        return None if _m(node.item, s, i, lambda j: j) is not None else k(i)
    raise TypeError(node)


def Opt(x):
    return Rep(x, 0, 1)


def Star(x):
    return Rep(x, 0, None)


def Plus(x):
    return Rep(x, 1, None)


def family_ast(family, masks):
    """The pattern family as an AST over the frozen class masks."""
    def m(c):
        return int(masks[c]) if c < len(masks) else 0
    isL = lambda c: m(c) & B_L
    isN = lambda c: m(c) & B_N
    isS = lambda c: m(c) & B_S
    crlf = lambda c: c in (10, 13)
    pre = Cls(lambda c: not crlf(c) and not isL(c) and not isN(c))
    other = Cls(lambda c: not isS(c) and not isL(c) and not isN(c))
    contraction = Seq(Lit("'"), Alt(*(Lit(x, ci=True) for x in ("s", "t", "re", "ve", "m", "ll", "d"))))
    tail = [
        Rep(Cls(isN), 1, 3),
        Seq(Opt(Lit(" ")), Plus(other), Star(Cls(crlf))),
        Seq(Star(Cls(isS)), Plus(Cls(crlf))),
        Seq(Plus(Cls(isS)), NegLook(Cls(lambda c: not isS(c)))),
        Plus(Cls(isS)),
    ]
    if family == 1:
        return Alt(contraction, Seq(Opt(pre), Plus(Cls(isL))), *tail)
    up = Cls(lambda c: m(c) & (B_LU | B_LT | B_LM | B_LO | B_M))
    lo = Cls(lambda c: m(c) & (B_LL | B_LM | B_LO | B_M))
    return Alt(Seq(Opt(pre), Star(up), Plus(lo), Opt(contraction)),
               Seq(Opt(pre), Plus(up), Star(lo), Opt(contraction)),
               *tail)


def is_kana_han(c):
    """deepseek-style D2 set: the Hiragana, Katakana and CJK Unified
    Ideographs blocks."""
    return 0x3040 <= c <= 0x30FF or 0x4E00 <= c <= 0x9FFF


def deepseek_asts(masks):
    """The three splitters of the deepseek-style family, in order, as ASTs:
    digit groups, kana/CJK runs, then the cl100k-style alternatives without
    the digit alternative."""
    def m(c):
        return int(masks[c]) if c < len(masks) else 0
    isL = lambda c: m(c) & B_L
    isN = lambda c: m(c) & B_N
    isS = lambda c: m(c) & B_S
    crlf = lambda c: c in (10, 13)
    pre = Cls(lambda c: not crlf(c) and not isL(c) and not isN(c))
    other = Cls(lambda c: not isS(c) and not isL(c) and not isN(c))
    contraction = Seq(Lit("'"), Alt(*(Lit(x, ci=True) for x in ("s", "t", "re", "ve", "m", "ll", "d"))))
    third = Alt(contraction, Seq(Opt(pre), Plus(Cls(isL))),
                Seq(Opt(Lit(" ")), Plus(other), Star(Cls(crlf))),
                Seq(Star(Cls(isS)), Plus(Cls(crlf))),
                Seq(Plus(Cls(isS)), NegLook(Cls(lambda c: not isS(c)))),
                Plus(Cls(isS)))
    return [Rep(Cls(isN), 1, 3), Plus(Cls(is_kana_han)), third]


def split_pieces(ast, s):
    """One splitter over the subject s: the leftmost match from the end of
    the previous one is a piece, and so is each stretch between matches."""
    out, p, q = [], 0, 0
    while q < len(s):
        e = _m(ast, s, q, lambda j: j)
        if e is None:
            q += 1
            continue
        assert e > q
        if q > p:
            out.append(s[p:q])
        out.append(s[q:e])
        p = q = e
    if p < len(s):
        out.append(s[p:])
    return out


def split_sequence(splitters, s, split=split_pieces):
    """Splitters in sequence: each re-splits every piece of the one before."""
    pieces = [s] if s else []
    for sp in splitters:
        pieces = [x for piece in pieces for x in split(sp, piece)]
    return pieces


def brute_pieces(ast, s):
    """Leftmost-first scan: the first alternative matching at p is the piece."""
    out, p = [], 0
    while p < len(s):
        e = _m(ast, s, p, lambda j: j)
        assert e is not None and e > p, (s, p)
        out.append(s[p:e])
        p = e
    return out


# ------------------------------------------------------------ textbook BPE
def textbook_bpe(data, ranks, results, whole=None):
    """ranks: {(l, r): rank}; results: {(l, r): id}; whole: {bytes: id} for
    the whole-piece shortcut (None = plain BPE).  Every step rescans all
    adjacent pairs."""
    if whole is not None and bytes(data) in whole:
        return [whole[bytes(data)]]
    ids = list(data)
    while True:
        best = None
        for i in range(len(ids) - 1):
            r = ranks.get((ids[i], ids[i + 1]))
            if r is not None and (best is None or r < best[0]):
                best = (r, i)
        if best is None:
            return ids
        i = best[1]
        ids[i:i + 2] = [results[(ids[i], ids[i + 1])]]


# ------------------------------------------------------- `regex` patterns
_K = r"(?i:'s|'t|'re|'ve|'m|'ll|'d)"
TAIL = r"\p{N}{1,3}| ?[^\s\p{L}\p{N}]+[\r\n]*|\s*[\r\n]+|\s+(?!\S)|\s+"
REGEX_PATTERNS = {
    1: _K + r"|[^\r\n\p{L}\p{N}]?\p{L}+|" + TAIL,
    2: (r"[^\r\n\p{L}\p{N}]?[\p{Lu}\p{Lt}\p{Lm}\p{Lo}\p{M}]*[\p{Ll}\p{Lm}\p{Lo}\p{M}]+" + _K + "?|"
        r"[^\r\n\p{L}\p{N}]?[\p{Lu}\p{Lt}\p{Lm}\p{Lo}\p{M}]+[\p{Ll}\p{Lm}\p{Lo}\p{M}]*" + _K + "?|" + TAIL),
}


DEEPSEEK_REGEX_SPLITTERS = [
    r"\p{N}{1,3}",
    r"[\u3040-\u30FF\u4E00-\u9FFF]+",
    _K + r"|[^\r\n\p{L}\p{N}]?\p{L}+| ?[^\s\p{L}\p{N}]+[\r\n]*|\s*[\r\n]+|\s+(?!\S)|\s+",
]


def regex_split(pat, s):
    """One splitter run by the regex engine: its matches over s, with the
    stretches between them kept as pieces."""
    out, p = [], 0
    for mt in pat.finditer(s):
        if mt.start() > p:
            out.append(s[p:mt.start()])
        out.append(mt.group())
        p = mt.end()
    if p < len(s):
        out.append(s[p:])
    return out


def all_strings(alphabet, max_len):
    """Every string over `alphabet` of length 1..max_len (shortest first)."""
    cur = [""]
    for _ in range(max_len):
        cur = [s + a for s in cur for a in alphabet]
        yield from cur


def family_pieces_chunk(args):
    """(family, strings) -> the AST matcher's pieces of each string; a
    worker for process pools (each process builds its own AST from the frozen
    class table).  family 3 runs the deepseek-style splitters in sequence."""
    family, strings = args
    import oracle
    masks = oracle.class_table()
    if family == 3:
        asts = deepseek_asts(masks)
        return [split_sequence(asts, s) for s in strings]
    ast = family_ast(family, masks)
    return [brute_pieces(ast, s) for s in strings]


def pieces_in_pool(family, strings, chunk=4096):
    """family_pieces_chunk over many strings, in a pool of spawned processes."""
    import multiprocessing
    import os
    parts = [(family, strings[i:i + chunk]) for i in range(0, len(strings), chunk)]
    with multiprocessing.get_context("spawn").Pool(min(8, os.cpu_count() or 1)) as pool:
        out = []
        for r in pool.map(family_pieces_chunk, parts):
            out.extend(r)
    return out
