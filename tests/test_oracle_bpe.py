"""Pins of the oracle's piece encoder E (TokTier §4.2: rank-ordered merges
per piece; the ignore_merges whole-piece shortcut) against things other than
itself: the textbook definition on every short string, hand-worked results,
the zero-merge closed form, losslessness and the fixpoint property, the
round-equivalence the GPU schedule relies on (with the counterexample that
shows why the vocabulary must be well-ordered), and the equivalence of the
GPU's rounds with safe pairs merged early (with a planted mistake that the
comparison catches)."""
import random

import numpy as np
import pytest

import brute
import oracle
from exact_bpe_tokenization_gb300 import synth

A, Bc, C, D = ord("a"), ord("b"), ord("c"), ord("d")

# hand-made vocabulary with overlapping merges; id 256+k is merge k's result
HAND = [("a", "a"), ("a", "b"), ("b", "a"), ("aa", "b"), ("c", "d"), ("ab", "a"), ("d", "c"), ("b", "b"),
        ("cd", "cd"), ("aa", "aa"), ("ba", "d"), ("a", "bb")]


def hand_vocab():
    toks = [bytes([i]) for i in range(256)]
    ids = {t: i for i, t in enumerate(toks)}
    merges = []
    for l, r in HAND:
        merges.append((ids[l.encode()], ids[r.encode()]))
        t = (l + r).encode()
        ids[t] = len(toks)
        toks.append(t)
    vo = np.zeros(len(toks) + 1, dtype=np.int64)
    np.cumsum([len(t) for t in toks], out=vo[1:])
    return np.array(merges, dtype=np.int32), np.frombuffer(b"".join(toks), dtype=np.uint8), vo, toks


def tables(merges, toks):
    ranks = {(int(l), int(r)): k for k, (l, r) in enumerate(merges)}
    index = {t: i for i, t in enumerate(toks)}
    results = {(int(l), int(r)): index[toks[l] + toks[r]] for l, r in merges}
    return ranks, results, index


@pytest.fixture(scope="module")
def hand():
    m, vb, vo, toks = hand_vocab()
    return oracle.Oracle(m, vb, vo, 1), m, toks


def test_hand_worked_examples(hand):
    o, _, _ = hand
    # worked by hand from the merge table above (plain BPE, no shortcut)
    cases = {"aaa": [256, A], "aaaa": [265], "aab": [259], "aba": [261], "bad": [266], "cdcd": [264],
             "dcd": [D, 260], "abb": [257, Bc], "ddd": [D, D, D], "abab": [257, 257], "baba": [Bc, 261],
             "aaaaa": [265, A], "": []}
    for s, want in cases.items():
        assert o.encode_bytes(s.encode(), plain=True) == want, s
    # the whole-piece shortcut differs from plain BPE exactly where the piece
    # is a vocabulary entry that plain BPE does not reach
    assert o.encode_bytes(b"abb") == [267]
    assert o.encode_bytes(b"aba") == [261]


def test_exhaustive_against_textbook(hand):
    """Every string of length <= 6 over {a,b,c,d}: plain and shortcut."""
    o, m, toks = hand
    ranks, results, index = tables(m, toks)
    for s in brute.all_strings("abcd", 6):
        b = s.encode()
        assert o.encode_bytes(b, plain=True) == brute.textbook_bpe(b, ranks, results), s
        assert o.encode_bytes(b) == brute.textbook_bpe(b, ranks, results, whole=index), s


def test_zero_merges_is_utf8_bytes():
    o = oracle.pretokenizer(1)
    text = synth.transcript(3, 20000, 1).decode()
    assert o.encode(text) == list(text.encode("utf-8"))


@pytest.mark.parametrize("family", [1, 2])
def test_lossless_and_fixpoint(family, small_vocabs):
    m, vb, vo = small_vocabs[family]
    o = oracle.Oracle(m, vb, vo, family)
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    ranks = {(int(l), int(r)) for l, r in m}
    text = synth.transcript(5, 60000, 2 if family == 2 else 1)
    ids = o.encode(text)
    assert b"".join(toks[i] for i in ids) == text
    # plain BPE ends at a fixpoint: no adjacent pair of the output has a rank
    for piece in oracle.pretokenizer(family).pieces(text.decode())[:3000]:
        out = o.encode_bytes(piece.encode(), plain=True)
        assert not any((out[i], out[i + 1]) in ranks for i in range(len(out) - 1))


def round_parallel(b, ranks, results):
    """One round = lowest rank present, then every leftmost non-overlapping
    occurrence of that pair merged in one sweep (TokTier §4.2)."""
    ids = list(b)
    while True:
        rs = [ranks.get((ids[i], ids[i + 1])) for i in range(len(ids) - 1)]
        live = [r for r in rs if r is not None]
        if not live:
            return ids
        r = min(live)
        out, i = [], 0
        while i < len(ids):
            if i + 1 < len(ids) and rs[i] == r:
                out.append(results[(ids[i], ids[i + 1])])
                i += 2
            else:
                out.append(ids[i])
                i += 1
        ids = out


def test_round_equivalence_well_ordered(hand, small_vocabs):
    o, m, toks = hand
    ranks, results, _ = tables(m, toks)
    for s in brute.all_strings("abcd", 6):
        assert round_parallel(s.encode(), ranks, results) == o.encode_bytes(s.encode(), plain=True)
    m, vb, vo = small_vocabs[1]
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    ranks, results, _ = tables(m, toks)
    o = oracle.Oracle(m, vb, vo, 1)
    rng = random.Random(3)
    text = synth.transcript(9, 100000, 1).decode()
    pieces = oracle.pretokenizer(1).pieces(text)
    for p in rng.sample(pieces, 3000) + [" " * 300, "a a " * 50]:
        b = p.encode()
        assert round_parallel(b, ranks, results) == o.encode_bytes(b, plain=True), p


def test_round_equivalence_needs_well_ordering():
    """Counterexample: 'aba' is merged (rank 0) from 'ab', which is created
    only at rank 1.  Sequential merging and rounds disagree on 'abab'."""
    toks = [bytes([i]) for i in range(256)] + [b"ab", b"aba"]
    m = np.array([[256, A], [A, Bc]], dtype=np.int32)
    vo = np.zeros(len(toks) + 1, dtype=np.int64)
    np.cumsum([len(t) for t in toks], out=vo[1:])
    o = oracle.Oracle(m, np.frombuffer(b"".join(toks), dtype=np.uint8), vo, 1)
    ranks, results, _ = tables(m, toks)
    assert o.encode_bytes(b"abab", plain=True) == [257, Bc]
    assert round_parallel(b"abab", ranks, results) == [256, 256]


def safe_rounds(b, merges, toks, ranks, results, wrong_minimum=False):
    """The rounds with safe pairs that the warp and block BPE run.  A pair
    x.y of rank q is safe when no merge of lower rank can take x from the left
    (a merge (X, x) whose X ends with the text byte before x) or y from the
    right (a merge (y, Z) whose Z starts with the byte after y).  A round
    merges every safe pair and the leftmost non-overlapping occurrences of
    the lowest rank of all pairs.  wrong_minimum: take the round minimum over
    the pairs that are not safe only (a planted mistake)."""
    take_left, take_right = {}, {}
    for k, (l, r) in enumerate(merges.tolist()):
        take_left.setdefault((r, toks[l][-1]), k)
        take_right.setdefault((l, toks[r][0]), k)
    ids, start = list(b), list(range(len(b)))
    while True:
        n = len(ids)
        rs = [ranks.get((ids[i], ids[i + 1])) for i in range(n - 1)]
        if all(r is None for r in rs):
            return ids
        safe = []
        for i in range(n - 1):
            q = rs[i]
            end = start[i + 2] if i + 2 < n else len(b)
            before = b[start[i] - 1] if start[i] > 0 else None
            after = b[end] if end < len(b) else None
            safe.append(q is not None and
                        (before is None or take_left.get((ids[i], before), q + 1) > q) and
                        (after is None or take_right.get((ids[i + 1], after), q + 1) > q))
        pool = [r for i, r in enumerate(rs) if r is not None and not (wrong_minimum and safe[i])]
        r = min(pool) if pool else None
        sel = list(safe)
        i = 0
        while i < n - 1:
            if not safe[i] and rs[i] is not None and rs[i] == r:
                if wrong_minimum and ((i > 0 and sel[i - 1]) or (i + 2 < n and sel[i + 1])):
                    i += 1
                    continue
                sel[i] = True
                i += 2
            else:
                i += 1
        assert not any(sel[i] and sel[i + 1] for i in range(n - 2)), "merges overlap"
        out, i = [], 0
        while i < n:
            if i + 1 < n and sel[i]:
                out.append(results[(ids[i], ids[i + 1])])
                i += 2
            else:
                out.append(ids[i])
                i += 1
        ids, start = out, _starts(out, toks)


def _starts(ids, toks):
    st, x = [], 0
    for t in ids:
        st.append(x)
        x += len(toks[t])
    return st


def small_alphabet_case():
    """Letter runs over two- and three-symbol alphabets with a vocabulary of
    3,000 merges trained on the same text: many overlapping merges."""
    rng = random.Random(5)
    words = []
    for _ in range(600):
        alpha = rng.choice(["ab", "abc", "ab\u65e5", "a\u00e9", "a"])
        words.append("".join(rng.choice(alpha) for _ in range(rng.randint(17, 90))))
    text = " ".join(words)
    merges = synth.train_merges(text.encode(), 3000)
    vb, vo = synth.vocab_from_merges(merges)
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    return merges, vb, vo, toks, [w.encode() for w in words]


def test_safe_pair_rounds_equal_sequential_merging(hand, small_vocabs):
    """Merging safe pairs out of rank order (the GPU rounds) gives the
    sequential result: every string of length <= 6 over 'abcd' with the
    hand-made vocabulary, 2,000 pieces of generated text with 8,000 merges,
    and small-alphabet letter runs with a vocabulary trained on them."""
    o, m, toks = hand
    ranks, results, _ = tables(m, toks)
    for s in brute.all_strings("abcd", 6):
        assert safe_rounds(s.encode(), m, toks, ranks, results) == o.encode_bytes(s.encode(), plain=True), s
    m, vb, vo = small_vocabs[1]
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    ranks, results, _ = tables(m, toks)
    o = oracle.Oracle(m, vb, vo, 1)
    text = synth.transcript(11, 60000, 1).decode()
    pieces = oracle.pretokenizer(1).pieces(text)
    for p in random.Random(4).sample(pieces, 2000):
        b = p.encode()
        assert safe_rounds(b, m, toks, ranks, results) == o.encode_bytes(b, plain=True), p
    m, vb, vo, toks, words = small_alphabet_case()
    ranks, results, _ = tables(m, toks)
    o = oracle.Oracle(m, vb, vo, 1)
    for w in words:
        assert safe_rounds(w, m, toks, ranks, results) == o.encode_bytes(w, plain=True), w


def test_safe_pair_rounds_planted_minimum_mistake_is_caught():
    """The comparison above discriminates: taking the round minimum over the
    pairs that are not safe lets a lower-ranked safe pair lose a token to a
    merge it precedes, and changes the result of some small-alphabet run."""
    m, vb, vo, toks, words = small_alphabet_case()
    ranks, results, _ = tables(m, toks)
    o = oracle.Oracle(m, vb, vo, 1)
    assert any(safe_rounds(w, m, toks, ranks, results, wrong_minimum=True) != o.encode_bytes(w, plain=True)
               for w in words)


def test_renumbered_token_ids(small_vocabs):
    """Token IDs are names: renumbering every ID (byte tokens included, the
    rank order kept) renames the output and changes nothing else."""
    from conftest import permute_vocab
    m, vb, vo = small_vocabs[1]
    pm, pvb, pvo, perm = permute_vocab(m, vb, vo, 21)
    o, po = oracle.Oracle(m, vb, vo, 1), oracle.Oracle(pm, pvb, pvo, 1)
    text = synth.transcript(13, 40000, 1)
    assert po.encode(text) == [int(perm[i]) for i in o.encode(text)]


def test_seam_example():
    """tok(A) || tok(B) != tok(A || B) with A = ' pipe', B = 'line' on a
    vocabulary that holds ' pipe', 'line' and ' pipeline' (TokTier §3.1,
    Figure 4, restated on a synthetic vocabulary)."""
    text = (" pipeline" * 3000 + " pipe" * 4000 + " (line" * 4000 + "\n").encode()
    merges = synth.train_merges(text, 40)
    vb, vo = synth.vocab_from_merges(merges)
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    for t in (b" pipe", b"line", b" pipeline"):
        assert t in toks
    o = oracle.Oracle(merges, vb, vo, 1)
    a, b = o.encode(" pipe"), o.encode("line")
    ab = o.encode(" pipeline")
    assert a == [toks.index(b" pipe")] and b == [toks.index(b"line")] and ab == [toks.index(b" pipeline")]
    assert a + b != ab


@pytest.mark.parametrize("family", [1, 2])
def test_splice_invariants(family, small_vocabs):
    """E*(U || V) = E*(U) || E*(V) when U, V are whole pieces (summary page
    §2.2): the batch output equals per-piece encodings concatenated at every
    piece boundary.  Cutting the text itself is different: cutting at an
    arbitrary position changes G (the seam), and the test records where."""
    m, vb, vo = small_vocabs[family]
    o = oracle.Oracle(m, vb, vo, family)
    pt = oracle.pretokenizer(family)
    text = synth.transcript(21, 4000, 1).decode()
    pieces = pt.pieces(text)
    full = o.encode(text)
    per_piece = [o.encode_bytes(p.encode()) for p in pieces]
    assert sum(per_piece, []) == full
    # G(S[:b]) || G(S[b:]) == G(S) holds at some positions and fails at others
    ok = bad = 0
    for b in range(1, len(text)):
        if pt.pieces(text[:b]) + pt.pieces(text[b:]) == pieces:
            ok += 1
        else:
            bad += 1
    assert ok > 0 and bad > 0
    # named hazards: digit grouping, whitespace lookahead, newline absorption
    assert pt.pieces("12") + pt.pieces("34") != pt.pieces("1234")
    assert pt.pieces("a  ") + pt.pieces("b") != pt.pieces("a  b")
    assert pt.pieces(";") + pt.pieces("\n") != pt.pieces(";\n")
