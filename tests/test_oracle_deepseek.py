"""Pins of the oracle's deepseek-style pre-tokenizer (three splitters in
sequence, each re-splitting every piece of the one before, the stretches
between matches kept as pieces: TokTier §4.1, on DeepSeek-family tokenizers)
against things other than itself: an independent split driver over the
backtracking AST matcher on every short string of a reduced alphabet, the
`regex` engine's own splitting (where installed) on short strings and on
generated kana/CJK-mixed text, and hand-derived cases."""
import importlib.util
import random

import pytest

import brute
import oracle
from exact_bpe_tokenization_gb300 import synth
from test_oracle_pretok import oracle_pieces_batch

FAM = oracle.FAMILY_DEEPSEEK_STYLE
# digits, letters, kana (ideograph, hiragana, katakana middle dot: other
# inside D2's set), blanks, CR/LF, apostrophe and punctuation
ALPHABET = ["a", "s", "1", " ", "\n", "'", ".", "日", "か", "・"]
ALPHABET2 = ["B", "2", "\t", "\r", "ー", "゙", "'", "t", "x", "\U0001F642"]
HAVE_REGEX = importlib.util.find_spec("regex") is not None


@pytest.mark.parametrize("alpha", [ALPHABET, ALPHABET2])
def test_brute_force_splitters_short_strings(alpha, masks):
    """Every string of length <= 4 and 3000 seeded strings of length 5-9:
    oracle pieces == the three AST splitters run one after another."""
    asts = brute.deepseek_asts(masks)
    strings = list(brute.all_strings(alpha, 4))
    rng = random.Random(3)
    strings += ["".join(rng.choice(alpha) for _ in range(rng.randint(5, 9))) for _ in range(3000)]
    got = oracle_pieces_batch(oracle.pretokenizer(FAM), strings)
    for s, g in zip(strings, got):
        assert g == brute.split_sequence(asts, s), repr(s)


@pytest.mark.slow
@pytest.mark.parametrize("alpha", [
    ["a", "1", " ", "\n", "日", "か", "・"],     # letters, digit groups, blanks, kana / ideographs, middle dot
    ["s", "'", "2", "\t", "ー", ".", "x"],      # contractions, digits, tab look-ahead, long-vowel sign, other
])
def test_brute_force_splitters_all_strings_up_to_6(alpha):
    """The three AST splitters run one after another, on every string of
    length <= 6 over a 7-symbol alphabet (137,256 strings)."""
    strings = list(brute.all_strings(alpha, 6))
    want = brute.pieces_in_pool(FAM, strings)
    got = oracle_pieces_batch(oracle.pretokenizer(FAM), strings)
    bad = [s for s, g, w in zip(strings, got, want) if g != w]
    assert not bad, [repr(s) for s in bad[:10]]


@pytest.mark.skipif(not HAVE_REGEX, reason="regex engine not installed")
def test_regex_engine_splitters_all_strings_up_to_5():
    import regex
    pats = [regex.compile(p) for p in brute.DEEPSEEK_REGEX_SPLITTERS]
    strings = list(brute.all_strings(ALPHABET, 5))
    got = oracle_pieces_batch(oracle.pretokenizer(FAM), strings)
    bad = [s for s, g in zip(strings, got) if g != brute.split_sequence(pats, s, brute.regex_split)]
    assert not bad, [repr(s) for s in bad[:10]]


@pytest.mark.skipif(not HAVE_REGEX, reason="regex engine not installed")
@pytest.mark.parametrize("profile,n", [(3, 300_000), (1, 100_000), (2, 100_000)])
def test_regex_engine_splitters_generated_text(profile, n):
    import regex
    pats = [regex.compile(p) for p in brute.DEEPSEEK_REGEX_SPLITTERS]
    text = synth.transcript(12, n, profile).decode("utf-8")
    assert oracle.pretokenizer(FAM).pieces(text) == brute.split_sequence(pats, text, brute.regex_split)


# ---------------------------------------------------------- hand-derived
CASES = [
    # D1 cuts digit groups out first, from the start of each digit run
    ("x1234", ["x", "123", "4"]),
    ("ab12cd", ["ab", "12", "cd"]),
    # the blank run before a digit group ends its piece: C6 sees the piece end
    ("a  1", ["a", "  ", "1"]),
    ("a  b", ["a", " ", " b"]),          # (same text without the splitter: C6 backtracks)
    # D2 isolates kana / ideograph runs: no prefix char, no letters glued on
    ("abc日本語def", ["abc", "日本語", "def"]),
    (" 日本", [" ", "日本"]),
    (",日本", [",", "日本"]),
    ("日本's", ["日本", "'s"]),
    # inside a D2 run the third splitter still cuts: the middle dot is "other"
    ("カ・ナ", ["カ", "・ナ"]),
    ("カナ・", ["カナ", "・"]),
    # a digit group inside kana text
    ("第3章", ["第", "3", "章"]),
    # newline absorption stops at the piece end
    (";\n\n日", [";\n\n", "日"]),
    ("x\n日", ["x", "\n", "日"]),
    ("a \n1", ["a", " \n", "1"]),
    ("", []),
]


@pytest.mark.parametrize("text,pieces", CASES)
def test_hand_derived_cases(text, pieces):
    assert oracle.pretokenizer(FAM).pieces(text) == pieces


def test_same_as_cl100k_style_without_digits_or_kana():
    """On text with no digits and no D2 chars, D1 and D2 leave the request
    whole, so the three splitters reduce to the cl100k-style pattern."""
    text = synth.transcript(21, 200_000, 0).decode("utf-8")
    text = "".join(ch for ch in text if not ch.isdigit())
    assert oracle.pretokenizer(FAM).pieces(text) == oracle.pretokenizer(1).pieces(text)
