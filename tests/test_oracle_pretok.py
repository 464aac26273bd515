"""Pins of the oracle's pre-tokenizer G against things other than itself:
brute force over every short string of two reduced alphabets (an independent
backtracking matcher, and the `regex` engine where installed), generated
text through the `regex` engine, and hand-derived closed forms for the hazard
classes the paper names (digit grouping, whitespace lookahead, newline
absorption: TokTier §3.1; the run-head / contraction / case rules: §4.1)."""
import importlib.util
import random

import numpy as np
import pytest

import brute
import oracle
from conftest import concat_requests
from exact_bpe_tokenization_gb300 import synth

ALPHABETS = {
    1: ["a", "s", "1", " ", "\t", "\n", "\r", "'", ".", "é"],
    2: ["a", "B", "1", " ", "\n", "'", ".", "か", "́", "\U0001F642"],
    # o200k contractions, case and marks together
    3: ["s", "T", "'", "a", "か", "́", " ", ".", "E", "r"],
}
HAVE_REGEX = importlib.util.find_spec("regex") is not None


def oracle_pieces_batch(o, strings):
    data, offs = concat_requests(strings)
    r = o.run(data, offs, ids=False)
    ps, po = r["piece_starts"], r["piece_offsets"]
    out = []
    for i, s in enumerate(strings):
        b = s.encode("utf-8")
        st = [int(x - offs[i]) for x in ps[po[i]:po[i + 1]]] + [len(b)]
        out.append([b[st[k]:st[k + 1]].decode("utf-8") for k in range(len(st) - 1)])
    return out


@pytest.mark.parametrize("family,alphabet", [(1, 1), (2, 2), (2, 3)])
def test_brute_force_matcher_short_strings(family, alphabet, masks):
    """Independent AST backtracking matcher: every string of length <= 4 and
    a seeded sample of 3000 strings of length 5-8."""
    ast = brute.family_ast(family, masks)
    alpha = ALPHABETS[alphabet]
    strings = list(brute.all_strings(alpha, 4))
    rng = random.Random(family)
    strings += ["".join(rng.choice(alpha) for _ in range(rng.randint(5, 8))) for _ in range(3000)]
    got = oracle_pieces_batch(oracle.pretokenizer(family), strings)
    for s, g in zip(strings, got):
        assert g == brute.brute_pieces(ast, s), repr(s)


# Seven symbols each, so that every string of length <= 6 (137,256 of them)
# goes through the independent AST matcher in seconds.
AST6 = [
    (1, ["a", "s", "1", " ", "\n", "'", "."]),       # contractions, digit groups, blank runs, newline absorption
    (1, ["r", "e", "'", " ", "\t", "\r", "é"]),       # two-letter contractions, tab / CR look-ahead, a 2-byte letter
    (2, ["s", "T", "'", "a", "\u0301", " ", "."]),     # case splits, a combining mark, contraction suffixes
    (2, ["B", "b", "か", "1", "\n", "'", "\U0001F642"]),  # caseless letters, digits, newline, a 4-byte symbol
]


@pytest.mark.slow
@pytest.mark.parametrize("family,alpha", AST6)
def test_brute_force_matcher_all_strings_up_to_6(family, alpha):
    """Independent AST backtracking matcher on every string of length <= 6
    over a 7-symbol alphabet that holds the hazards of the family (§3.1:
    digit grouping, whitespace look-ahead, newline absorption; §4.1: case,
    marks, contractions)."""
    strings = list(brute.all_strings(alpha, 6))
    assert len(strings) == 137256
    want = brute.pieces_in_pool(family, strings)
    got = oracle_pieces_batch(oracle.pretokenizer(family), strings)
    bad = [s for s, g, w in zip(strings, got, want) if g != w]
    assert not bad, [repr(s) for s in bad[:10]]


@pytest.mark.skipif(not HAVE_REGEX, reason="regex engine not installed")
@pytest.mark.parametrize("family,alphabet", [(1, 1), (2, 2), (2, 3)])
def test_regex_engine_all_strings_up_to_6(family, alphabet):
    """Library run: the regex engine on every string of length <= 6 over the
    reduced alphabet (1,111,110 strings), fed to the oracle as one batch of
    tiny requests."""
    import regex
    pat = regex.compile(brute.REGEX_PATTERNS[family])
    strings = list(brute.all_strings(ALPHABETS[alphabet], 6))
    got = oracle_pieces_batch(oracle.pretokenizer(family), strings)
    bad = [s for s, g in zip(strings, got) if g != pat.findall(s)]
    assert not bad, [repr(s) for s in bad[:10]]


@pytest.mark.skipif(not HAVE_REGEX, reason="regex engine not installed")
@pytest.mark.parametrize("family,profile,n", [(1, 0, 200_000), (1, 1, 300_000), (2, 2, 300_000), (1, 2, 100_000),
                                              (2, 1, 100_000)])
def test_regex_engine_generated_text(family, profile, n):
    import regex
    pat = regex.compile(brute.REGEX_PATTERNS[family])
    text = synth.transcript(11, n, profile).decode("utf-8")
    assert oracle.pretokenizer(family).pieces(text) == pat.findall(text)


@pytest.mark.skipif(not HAVE_REGEX, reason="regex engine not installed")
def test_regex_engine_adversarial_text():
    import regex
    pat = regex.compile(brute.REGEX_PATTERNS[1])
    text = synth.adversarial(7, 400_000).decode("utf-8")
    assert oracle.pretokenizer(1).pieces(text) == pat.findall(text)


# ---------------------------------------------------------- closed forms
@pytest.mark.parametrize("family", [1, 2])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 10, 100, 1000])
def test_digit_run_groups_of_three(family, n):
    s = "".join(str((7 * i) % 10) for i in range(n))
    p = oracle.pretokenizer(family).pieces(s)
    assert len(p) == -(-n // 3) and all(len(x) == 3 for x in p[:-1]) and "".join(p) == s


@pytest.mark.parametrize("family", [1, 2])
@pytest.mark.parametrize("n", [2, 3, 5, 64, 5000])
def test_whitespace_lookahead(family, n):
    # a + n blanks + b -> "a", (n-1) blanks, " b"
    assert oracle.pretokenizer(family).pieces("a" + " " * n + "b") == ["a", " " * (n - 1), " b"]
    # at the end of the request the blank run stays whole
    assert oracle.pretokenizer(family).pieces("a" + " " * n) == ["a", " " * n]


@pytest.mark.parametrize("family", [1, 2])
def test_newline_absorption_and_blocks(family):
    pt = oracle.pretokenizer(family)
    assert pt.pieces("x;\n\n  y") == ["x", ";\n\n", " ", " y"]
    assert pt.pieces("\r\n\r\n \n") == ["\r\n\r\n \n"]
    assert pt.pieces("a\r\n\r\n \nb") == ["a", "\r\n\r\n \n", "b"]
    assert pt.pieces("a  \n  b") == ["a", "  \n", " ", " b"]
    assert pt.pieces("}\n\n") == ["}\n\n"]
    assert pt.pieces("} \n") == ["}", " \n"]
    assert pt.pieces(" .\n\tx") == [" .\n", "\tx"]


def test_cl100k_contractions_and_letters():
    pt = oracle.pretokenizer(1)
    assert pt.pieces("don't") == ["don", "'t"]
    assert pt.pieces("we'RE here") == ["we", "'RE", " here"]
    assert pt.pieces("it'sa") == ["it", "'s", "a"]
    assert pt.pieces("'llama") == ["'ll", "ama"]
    assert pt.pieces(" 's") == [" '", "s"]
    assert pt.pieces("camelCase HTMLParser") == ["camelCase", " HTMLParser"]
    assert pt.pieces("(foo") == ["(foo"]
    assert pt.pieces("((foo") == ["((", "foo"]
    assert pt.pieces("\tfoo") == ["\tfoo"]
    assert pt.pieces("\nfoo") == ["\n", "foo"]
    assert pt.pieces("1abc") == ["1", "abc"]
    assert pt.pieces("a\u0301b") == ["a", "\u0301b"]   # a mark is "other" here: a one-char prefix


def test_o200k_case_contraction_marks():
    pt = oracle.pretokenizer(2)
    assert pt.pieces("don't") == ["don't"]
    assert pt.pieces("don'tx") == ["don't", "x"]
    assert pt.pieces("camelCase") == ["camel", "Case"]
    assert pt.pieces("HTMLParser") == ["HTMLParser"]
    assert pt.pieces("getHTTPResponse") == ["get", "HTTPResponse"]
    assert pt.pieces("aBC") == ["a", "BC"]
    assert pt.pieces("ABc") == ["ABc"]
    assert pt.pieces("かA") == ["か", "A"]
    assert pt.pieces("かAB") == ["か", "AB"]
    assert pt.pieces("かAb") == ["かAb"]
    assert pt.pieces("a'sかBc") == ["a's", "かBc"]
    assert pt.pieces("1'st") == ["1", "'st"]
    assert pt.pieces("áb") == ["áb"]                  # marks attach to letters
    assert pt.pieces(".́a") == [".́a"]
    assert pt.pieces("..́a") == ["..́", "a"]           # after two others a mark stays "other"
    assert pt.pieces(" .́a") == [" .́", "a"]
    assert pt.pieces("́.́..") == ["́", ".́", ".."]
    # contraction chain: letters used up by a contraction do not take another
    assert pt.pieces("a'd'd") == ["a'd", "'d"]
    assert pt.pieces("a'd'd'd") == ["a'd", "'d'd"]
    assert pt.pieces("s'rE") == ["s'rE"]


def test_request_boundaries_cut_runs():
    pt = oracle.pretokenizer(1)
    data, offs = concat_requests(["ab", "cd", "12", "34", "  ", " x"])
    r = pt.run(data, offs, ids=False)
    assert r["piece_offsets"].tolist() == [0, 1, 2, 3, 4, 5, 6]
    assert r["piece_starts"].tolist() == offs[:-1].tolist()


def test_empty_and_invalid_requests():
    pt = oracle.pretokenizer(1)
    data, offs = concat_requests([b"", b"ok", b"\xff", b"", b"a\xc3", b"fine"])
    r = pt.run(data, offs)
    assert r["status"].tolist() == [0, 0, oracle.ERR_UTF8, 0, oracle.ERR_UTF8, 0]
    assert r["id_offsets"].tolist() == [0, 0, 2, 2, 2, 2, 6]
    assert r["piece_offsets"].tolist() == [0, 0, 1, 1, 1, 1, 2]


def test_utf8_validation_matches_strict_decode():
    """Random byte strings biased towards UTF-8 edge bytes: the oracle rejects
    exactly what Python's strict decoder rejects."""
    rng = random.Random(5)
    edge = [0x00, 0x41, 0x7F, 0x80, 0xBF, 0xC0, 0xC1, 0xC2, 0xDF, 0xE0, 0xED, 0xEF, 0xF0, 0xF4, 0xF5, 0xFF, 0xA0, 0x9F, 0x8F, 0x90]
    reqs = []
    for _ in range(20000):
        n = rng.randint(1, 6)
        reqs.append(bytes(rng.choice(edge) if rng.random() < 0.8 else rng.randrange(256) for _ in range(n)))
    reqs += ["퟿".encode(), b"\xed\xa0\x80", "\U0010ffff".encode(), b"\xf4\x90\x80\x80", b"\xe0\x80\x80"]
    data, offs = concat_requests(reqs)
    st = oracle.pretokenizer(1).run(data, offs, ids=False)["status"]
    for b, s in zip(reqs, st):
        try:
            b.decode("utf-8", "strict")
            ok = True
        except UnicodeDecodeError:
            ok = False
        assert (s == 0) == ok, b
