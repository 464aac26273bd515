"""Pins of the frozen character-class table (TokTier, §4.1 and §5.2: class
tables are probed out of the reference engine and pinned by hash)."""
import importlib.util
import os

import numpy as np
import pytest

import oracle

B_L, B_LU, B_LL, B_LT, B_LM, B_LO, B_M, B_N, B_S = (1 << i for i in range(9))
PINNED_SHA = "e33e988ffe174bb40b6295e9a421d4acdc09011e9eb242ea6f01b1daec359fd5"


def test_recorded_hash_is_pinned():
    with open(oracle.oracle.CLASS_TABLE) as f:
        head = [l for l in f if l.startswith("# body-sha256")]
    assert head and head[0].split()[2] == PINNED_SHA


def test_classes_are_disjoint(masks):
    m = masks.astype(np.int64)
    top = [(m & b) != 0 for b in (B_L, B_M, B_N, B_S)]
    for i in range(4):
        for j in range(i + 1, 4):
            assert not np.any(top[i] & top[j])
    subs = [(m & b) != 0 for b in (B_LU, B_LL, B_LT, B_LM, B_LO)]
    total = sum(s.astype(np.int64) for s in subs)
    # every letter is in exactly one letter subclass and nothing else is
    assert np.array_equal(total, ((m & B_L) != 0).astype(np.int64))


@pytest.mark.parametrize("ch,bits", [
    ("a", B_L | B_LL), ("A", B_L | B_LU), ("1", B_N), (" ", B_S), ("\t", B_S), ("\n", B_S), ("\r", B_S),
    ("́", B_M), ("か", B_L | B_LO), ("ǅ", B_L | B_LT), ("ʰ", B_L | B_LM), (".", 0), ("'", 0),
    ("\x1c", 0), ("\u0085", B_S), ("　", B_S), ("½", B_N), (" ", B_S), ("é", B_L | B_LL),
    ("\U0001F642", 0), ("一", B_L | B_LO), ("_", 0),
])
def test_spot_values(masks, ch, bits):
    assert int(masks[ord(ch)]) == bits


@pytest.mark.skipif(importlib.util.find_spec("regex") is None, reason="regex engine not installed")
def test_table_matches_a_fresh_probe(masks, tmp_path):
    """Re-probe the engine and compare every code point (library run)."""
    import sys
    sys.path.insert(0, os.path.dirname(oracle.oracle.CLASS_TABLE))
    import probe_char_classes
    fresh, version = probe_char_classes.probe_masks()
    assert np.array_equal(np.array(fresh, dtype=np.uint16), masks), "regex %s disagrees with the table" % version
