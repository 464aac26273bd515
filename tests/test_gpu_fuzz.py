"""Fuzzing the CUDA path against the oracle, per piece boundary and per ID:
requests of code points drawn from the whole Unicode range (every class the
frozen table knows, marks, kana/CJK, non-BMP), mixed with ASCII runs, blank
and CR/LF runs, apostrophes, digits, invalid byte sequences and empty
requests, for all three pattern families, in one batch that spans many
tiles."""
import random

import pytest

from exact_bpe_tokenization_gb300 import synth
from test_gpu_parity import check

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from exact_bpe_tokenization_gb300 import binding
    return binding


def random_request(rng):
    parts = []
    for _ in range(rng.randint(0, 40)):
        kind = rng.random()
        if kind < 0.35:                                   # any scalar value
            cp = rng.randint(0x20, 0x10FFFF)
            if 0xD800 <= cp <= 0xDFFF:
                cp = 0xFFFD
            parts.append(chr(cp).encode())
        elif kind < 0.55:
            parts.append("".join(rng.choice("aZé'sT tの日1 \n\r\t.,") for _ in range(rng.randint(1, 12))).encode())
        elif kind < 0.65:                                 # blank runs before what ends them
            parts.append((" " * rng.randint(1, 70) + rng.choice(["", "\n", "x", "1", "日", "́"])).encode())
        elif kind < 0.75:
            parts.append(str(rng.randint(0, 10 ** rng.randint(1, 14))).encode())
        elif kind < 0.85:
            parts.append(("'" + rng.choice(["s", "T", "re", "LL", "d", "x", ""])).encode())
        else:                                             # combining marks after letters and punctuation
            parts.append((rng.choice("aB.,か") + "".join(chr(0x300 + rng.randint(0, 0x6F))
                                                         for _ in range(rng.randint(1, 3)))).encode())
    if parts and rng.random() < 0.1:                      # one request in ten carries an invalid sequence
        parts.insert(rng.randrange(len(parts) + 1),
                     rng.choice([b"\xff", b"\xc3(", b"\xe0\x80\x80", b"\xed\xa0\x80", b"\xf4\x90\x80\x80",
                                 b"\x80", b"\xe4\xb8"]))
    return b"".join(parts)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("family", [1, 2, 3])
def test_fuzz_batch_against_the_oracle(cuda, family, seed):
    rng = random.Random(1000 * seed + family)
    reqs = [random_request(rng) for _ in range(6000)] + [b"", b"", b" "]
    profile = {1: synth.PROFILE_MIXED, 2: synth.PROFILE_CAMEL_MARKS, 3: synth.PROFILE_KANA_HAN}[family]
    vocab = synth.make_vocab(profile, 1 << 20, 8000)
    check(cuda, vocab, family, reqs)
