"""GPU parity for the deepseek-style family (three splitters in sequence,
folded into the per-character predicate: TokTier §4.1 on DeepSeek-family
tokenizers): the CUDA path against the oracle, per piece boundary, per ID and
per byte span, on every short string of two reduced alphabets as tiny
requests, random strings, segment edges at every alignment to the tiles,
pieces around the execution-unit thresholds, added-token literals, and the
64-request kana/CJK-mixed batch at full size."""
import os
import random

import numpy as np
import pytest

import brute
from exact_bpe_tokenization_gb300 import synth
from test_gpu_literals import parity as literal_parity
from test_gpu_literals import sprinkle
from test_gpu_parity import check
from test_gpu_spans import spans_parity

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
NCPU = os.cpu_count() or 1
FAM = 3
ALPHABETS = [["a", "s", "1", " ", "\n", "'", ".", "日", "か", "・"],
             ["B", "2", "\t", "\r", "ー", "゙", "'", "t", " ", "\U0001F642"]]


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from exact_bpe_tokenization_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def small3():
    return synth.make_vocab(synth.PROFILE_KANA_HAN, 1 << 20, 8000)


@pytest.fixture(scope="module")
def d1():
    return synth.make_vocab(synth.PROFILE_KANA_HAN, 8 << 20, 100000)


@pytest.mark.parametrize("alphabet", [0, 1])
def test_all_short_strings_as_tiny_requests(cuda, small3, alphabet):
    """Every string of length <= 5 (111,110 requests in one batch)."""
    check(cuda, small3, FAM, list(brute.all_strings(ALPHABETS[alphabet], 5)))


def test_random_mixed_strings(cuda, small3):
    alpha = ALPHABETS[0] + ALPHABETS[1] + ["A", "e", "r", "l", "́", "　", "٣", "0", "_", "(", "一", "゠", "ヿ",
                                           "぀", "鿿", "ゟ", "゠", "䷿", "ꀀ"]
    rng = random.Random(41)
    reqs = ["".join(rng.choice(alpha) for _ in range(rng.randint(1, 40))) for _ in range(60000)]
    check(cuda, small3, FAM, reqs)


PATHOLOGICAL = [
    "日" * 5000, "a日" * 3000, "1日" * 3000, " 日" * 3000, "カ・" * 3000, "123456789" * 1000, "  1" * 2000,
    " " * 9000 + "日", " " * 9000 + "7", "\n" * 5000 + "か", "x" * 6000 + "ー" * 6000, "'s日" * 2000,
    ";\n\n日" * 2000, "7" * 10000 + "日本", "a 1 b 2 " * 2000,
]


def test_segments_straddling_tiles_at_every_alignment(cuda, small3):
    """Each run is preceded by 0..47 filler bytes, so segment starts and
    ends fall at every offset relative to the tiles and the per-thread
    byte groups."""
    reqs = []
    for k, run in enumerate(PATHOLOGICAL):
        for pad in range(0, 48, 3 if k % 2 else 1):
            reqs.append("q" * pad + " " + run + " tail")
    check(cuda, small3, FAM, reqs)
    check(cuda, small3, FAM, ["z".join(reqs[::7])])


@pytest.mark.parametrize("n", [1, 2, 16, 17, 32, 33, 48, 49, 256, 257, 4096, 8193, 50000])
def test_piece_lengths_around_unit_thresholds(cuda, d1, n):
    reqs = ["日" * (n // 3 + 1), "か" * (n // 3 + 1) + "a", " " * n + "1", " " * n + "日", "a" * n + "日本",
            "(" * n + "か", "1" * n]
    check(cuda, d1, FAM, reqs)


def test_kana_han_batch_scaled(cuda, d1):
    check(cuda, d1, FAM, synth.workload("deepseek_64_loguniform", scale=0.1))


def test_deepseek_64_loguniform_full(cuda, d1):
    check(cuda, d1, FAM, synth.workload("deepseek_64_loguniform"))


def test_spans_kana_han_batch(cuda, d1):
    spans_parity(cuda, d1, FAM, synth.workload("deepseek_64_loguniform", scale=0.05))


def test_added_tokens_with_kana_literals(cuda, d1):
    n = len(d1[2]) - 1
    lits = {b"<|endoftext|>": n + 1, "<|ユーザー|>".encode(): n + 2, "日本".encode(): n + 3, b"12": n + 4,
            "aか".encode(): n + 5}
    reqs = sprinkle(synth.workload("deepseek_64_loguniform", scale=0.02), lits, seed=5, every=300)
    literal_parity(cuda, d1, FAM, lits, reqs)
