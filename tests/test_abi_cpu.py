"""The C ABI without a GPU: the library builds and loads, exports every
function include/toktier.h declares, embeds the pinned class table, and
tt_create rejects malformed vocabularies before any device call (the
well-ordering rule is what makes round-parallel merging equal to single
merges, TokTier §4.2)."""
import ctypes

import numpy as np
import pytest

from exact_bpe_tokenization_gb300 import binding, build, synth
from test_class_table import PINNED_SHA


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def test_exports_every_declared_symbol(lib):
    names = binding.declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    raw = ctypes.CDLL(binding.LIB_PATH)
    for n in names:
        getattr(raw, n)


def test_status_strings_and_digest(lib):
    assert binding.status_string(0) == "ok"
    assert "UTF-8" in binding.status_string(4)
    assert binding.tt_table_digest() == PINNED_SHA


def vocab_of(tokens, merges):
    vb = np.frombuffer(b"".join(tokens), dtype=np.uint8).copy()
    vo = np.zeros(len(tokens) + 1, dtype=np.int64)
    np.cumsum([len(t) for t in tokens], out=vo[1:])
    return np.array(merges, dtype=np.int32).reshape(-1, 2), vb, vo


BYTES = [bytes([i]) for i in range(256)]
A, B = ord("a"), ord("b")


@pytest.mark.parametrize("case,tokens,merges,status", [
    ("bad family", BYTES, [], binding.TT_ERR_BAD_FAMILY),
    ("missing byte", BYTES[:-1] + [b"ab"], [], binding.TT_ERR_BAD_VOCAB),
    ("duplicate string", BYTES + [b"a"], [], binding.TT_ERR_BAD_VOCAB),
    ("empty token", BYTES + [b""], [], binding.TT_ERR_BAD_VOCAB),
    ("result not a token", BYTES, [(A, B)], binding.TT_ERR_BAD_VOCAB),
    ("operand out of range", BYTES + [b"ab"], [(A, 999)], binding.TT_ERR_BAD_VOCAB),
    ("duplicate pair", BYTES + [b"ab"], [(A, B), (A, B)], binding.TT_ERR_BAD_VOCAB),
    ("two merges one result", BYTES + [b"ab", b"abb", b"bb"], [(A, B), (B, B), (256, B), (A, 258)],
     binding.TT_ERR_BAD_VOCAB),
    ("not well-ordered", BYTES + [b"ab", b"aba"], [(256, A), (A, B)], binding.TT_ERR_BAD_VOCAB),
])
def test_create_rejects(lib, case, tokens, merges, status):
    m, vb, vo = vocab_of(tokens, merges)
    fam = 9 if case == "bad family" else 1
    with pytest.raises(binding.TokTierError) as e:
        binding.tt_create(m, vb, vo, fam)
    assert e.value.status == status, case


def test_trained_vocabularies_are_well_ordered():
    """The greedy trainer only merges existing symbols, so its lists pass the
    create-time checks (checked here on the host with the same rule)."""
    for prof, nm in ((0, 4096), (1, 8000), (2, 8000)):
        m, vb, vo = synth.make_vocab(prof, 1 << 20, nm)
        created = {}
        for k, (l, r) in enumerate(m.tolist()):
            for x in (l, r):
                assert created.get(x, -1) < k
            created[256 + k] = k
