"""Pins for the oracle's added-token extraction (TokTier §4.4: added and
special tokens are literal strings the model reserves as single IDs; a
leftmost-longest literal pass extracts them before the tokenizer family
handles the remaining segments).  Checked against hand-worked cases and, on
every short string over a small alphabet with overlapping literals, against
an independent reference: a plain leftmost-longest splitter written here and
the family tokenizer run on each remaining segment as a document of its own
(the oracle without literals, pinned separately)."""
import numpy as np
import pytest

import brute
import oracle
from exact_bpe_tokenization_gb300 import synth


@pytest.fixture(scope="module")
def vocab():
    return synth.make_vocab(synth.PROFILE_ASCII, 1 << 20, 4096)


def split_leftmost_longest(data, literals):
    """[(start, end, literal id or None)] covering data."""
    out, seg, x = [], 0, 0
    while x < len(data):
        best = None
        for lit, i in literals.items():
            if data.startswith(lit, x) and (best is None or len(lit) > len(best[0])):
                best = (lit, i)
        if best is None:
            x += 1
            continue
        if x > seg:
            out.append((seg, x, None))
        out.append((x, x + len(best[0]), best[1]))
        x += len(best[0])
        seg = x
    if seg < len(data):
        out.append((seg, len(data), None))
    return out


def reference(plain, data, literals):
    pieces, ids = [], []
    for a, b, lid in split_leftmost_longest(data, literals):
        if lid is not None:
            pieces.append(a)
            ids.append(lid)
            continue
        r = plain.run(data[a:b], np.array([0, b - a], dtype=np.int64))
        pieces += [a + int(s) for s in r["piece_starts"]]
        ids += r["ids"].tolist()
    return pieces, ids


def run(o, data):
    r = o.run(data, np.array([0, len(data)], dtype=np.int64))
    return r["piece_starts"].tolist(), r["ids"].tolist()


def test_hand_worked_leftmost_longest(vocab):
    m, vb, vo = vocab
    o = oracle.Oracle(m, vb, vo, 1)
    n = len(vo) - 1
    A, B, C, E = n + 10, n + 11, n + 12, n + 13
    o.set_added_tokens({b"ab": A, b"abc": B, b"bcd": C, b"<|e|>": E})
    assert run(o, b"abcd")[1][0] == B and run(o, b"abcd")[0] == [0, 3]          # longest at the leftmost start
    assert run(o, b"xbcd")[0] == [0, 1] and run(o, b"xbcd")[1][1] == C          # leftmost first
    assert run(o, b"aab")[0] == [0, 1] and run(o, b"aab")[1][1] == A
    assert run(o, b"<|e|><|e|>") == ([0, 5], [E, E])
    assert run(o, b"abab")[1] == [A, A]
    # runs are cut at a literal: "1<|e|>2" is two one-digit pieces around it
    assert run(o, b"12<|e|>34")[0] == [0, 2, 7]
    o.set_added_tokens({})
    assert run(o, b"abcd")[0] == [0]                                             # cleared: plain text


def test_every_short_string_against_split_then_tokenize(vocab):
    m, vb, vo = vocab
    n = len(vo) - 1
    literals = {b"<a>": n + 1, b"<a>b": n + 2, b"a>": n + 3, b" <": n + 4, b"b b": n + 5, b"1\n": n + 6}
    o = oracle.Oracle(m, vb, vo, 1)
    o.set_added_tokens(literals)
    plain = oracle.Oracle(m, vb, vo, 1)
    checked = 0
    for s in brute.all_strings(["a", "b", "<", ">", " ", "1", "\n"], 5):
        data = s.encode()
        assert run(o, data) == reference(plain, data, literals), repr(s)
        checked += 1
    assert checked == 19607            # lengths 1..5


def test_literals_in_generated_batches_and_spans(vocab):
    m, vb, vo = vocab
    n = len(vo) - 1
    literals = {b"<|endoftext|>": n + 1, b"<|im_start|>": n + 2, b"<|im_end|>": n + 3, b"<|im": n + 4}
    o = oracle.Oracle(m, vb, vo, 1)
    o.set_added_tokens(literals)
    plain = oracle.Oracle(m, vb, vo, 1)
    rng = np.random.default_rng(3)
    reqs = []
    for i in range(12):
        t = synth.transcript(500 + i, 400, synth.PROFILE_ASCII)
        cuts = sorted(rng.integers(0, len(t), 4).tolist())
        parts, prev = [], 0
        for c in cuts:
            parts += [t[prev:c], [b"<|endoftext|>", b"<|im_start|>", b"<|im_end|>", b"<|im"][c % 4]]
            prev = c
        reqs.append(b"".join(parts) + t[prev:])
    data, offs = synth.batch(reqs)
    got = o.run_spans(data, offs)
    ref_ids = []
    for r in range(len(reqs)):
        ref_ids += reference(plain, reqs[r], literals)[1]
    assert got["ids"].tolist() == ref_ids
    # every literal ID spans exactly its literal's bytes
    inv = {v: k for k, v in literals.items()}
    for i, (a, b) in zip(got["ids"].tolist(), got["spans"].tolist()):
        if i in inv:
            assert data[a:b].tobytes() == inv[i]
