"""The CUDA path's piece-start rules (csrc/tt_rules.cuh), compiled for the
host with sequential scans, against the oracle's pre-tokenizer: every short
string over the reduced alphabets, generated text of every profile and the
adversarial blocks.  This isolates the rule derivation (TokTier §4.1) from
the parallel scans, which the GPU parity tests cover."""
import ctypes
import os
import random
import subprocess

import numpy as np
import pytest

import brute
import oracle
from conftest import concat_requests
from exact_bpe_tokenization_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
K_OTHER, K_LU, K_LL, K_LB, K_MARK, K_NUM, K_WS = range(7)


@pytest.fixture(scope="module")
def rules_lib(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("rules") / "librules_host.so")
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-o", so,
                           os.path.join(HERE, "rules_host.cpp")])
    lib = ctypes.CDLL(so)
    lib.rules_host_starts.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_void_p]
    lib.rules_host_top_bits4.argtypes = [ctypes.c_uint32]
    lib.rules_host_top_bits4.restype = ctypes.c_uint32
    return lib


def test_top_bit_gather_matches_the_bytes(rules_lib):
    # the UTF-8 check visits only bytes with the top bit set; the gather that
    # finds them must give bit k = top bit of byte k for every pattern of top
    # bits under any low bits
    rng = random.Random(5)
    words = [rng.getrandbits(32) for _ in range(20000)]
    words += [sum(((p >> k & 1) << (8 * k + 7)) | (low << (8 * k)) for k in range(4))
              for p in range(16) for low in (0x00, 0x7F, 0x55)]
    for w in words:
        want = sum(((w >> (8 * k + 7)) & 1) << k for k in range(4))
        assert rules_lib.rules_host_top_bits4(w) == want, hex(w)


K_HAN_FLAG = 0x10


def raw_kinds(masks, family=1):
    """Raw kinds per code point as the CUDA path's class table holds them
    (deepseek-style: kana / CJK ideographs flagged)."""
    m = masks.astype(np.int64)
    k = np.full(len(m), K_OTHER, dtype=np.uint8)
    k[(m & 64) != 0] = K_MARK
    k[(m & (16 | 32)) != 0] = K_LB
    k[(m & 4) != 0] = K_LL
    k[(m & (2 | 8)) != 0] = K_LU
    k[(m & 128) != 0] = K_NUM
    k[(m & 256) != 0] = K_WS
    if family == 3:
        k[0x3040:0x3100] |= K_HAN_FLAG
        k[0x4E00:0xA000] |= K_HAN_FLAG
    return k


def rule_starts(lib, family, kinds, strings):
    """Piece starts per request (as byte offsets within the request)."""
    cps, rs, char_pos = [], [], []
    for s in strings:
        b = s.encode("utf-8")
        pos = 0
        for i, ch in enumerate(s):
            cps.append(ord(ch))
            rs.append(1 if i == 0 else 0)
            char_pos.append(pos)
            pos += len(ch.encode("utf-8"))
    cp = np.array(cps, dtype=np.uint32)
    raw = kinds[cp] if len(cp) else np.zeros(0, dtype=np.uint8)
    rsa = np.array(rs, dtype=np.uint8)
    out = np.zeros(len(cp), dtype=np.uint8)
    if len(cp):
        lib.rules_host_starts(family, cp.ctypes.data, np.ascontiguousarray(raw).ctypes.data, rsa.ctypes.data,
                              len(cp), out.ctypes.data)
    # 2 marks a char where the 12-byte scan state of the families without a
    # case rule and the general 20-byte one give different aggregates
    assert not (out == 2).any(), "the two forms of the forward scan disagree"
    assert not (out == 3).any(), "a char decided from its near neighbourhood alone differs"
    res, k = [], 0
    for s in strings:
        n = len(s)
        res.append([char_pos[k + i] for i in range(n) if out[k + i]])
        k += n
    return res


def oracle_starts(family, strings):
    data, offs = concat_requests(strings)
    r = oracle.pretokenizer(family).run(data, offs, ids=False)
    ps, po = r["piece_starts"], r["piece_offsets"]
    return [[int(x - offs[i]) for x in ps[po[i]:po[i + 1]]] for i in range(len(strings))]


ALPHABETS = {
    1: ["a", "s", "1", " ", "\t", "\n", "\r", "'", ".", "é"],
    2: ["a", "B", "1", " ", "\n", "'", ".", "か", "́", "\U0001F642"],
    # o200k contractions, case and marks together
    3: ["s", "T", "'", "a", "か", "́", " ", ".", "E", "r"],
    # deepseek-style segments: digits, kana / ideographs (one of them "other")
    4: ["a", "s", "1", " ", "\n", "'", ".", "日", "か", "・"],
    5: ["B", "2", "\t", "\r", "ー", "゙", "'", "t", " ", "\U0001F642"],
}
EXTRA = {
    1: ["A", "t", "e", "r", "l", "m", "d", "v", "́", " ", "　", "٣"],
    2: ["s", "t", "r", "e", "l", "d", "\t", "\r", "ʰ", "ǅ", "é", "Ü"],
    3: ["A", "t", "e", "r", "\t", "\r", "́", "　", "٣", "カ", "ー", "゛", "\U0001F642"],
}
FAMILY_ALPHABET = {1: 1, 2: 2, 3: 4}


@pytest.mark.parametrize("family,alphabet", [(1, 1), (2, 2), (2, 3), (1, 3), (3, 4), (3, 5)])
def test_rules_all_short_strings(rules_lib, masks, family, alphabet):
    kinds = raw_kinds(masks, family)
    strings = list(brute.all_strings(ALPHABETS[alphabet], 6))
    got = rule_starts(rules_lib, family, kinds, strings)
    exp = oracle_starts(family, strings)
    bad = [(s, g, e) for s, g, e in zip(strings, got, exp) if g != e]
    assert not bad, bad[:5]


@pytest.mark.parametrize("family", [1, 2, 3])
def test_rules_mixed_alphabet_random(rules_lib, masks, family):
    kinds = raw_kinds(masks, family)
    alpha = ALPHABETS[FAMILY_ALPHABET[family]] + EXTRA[family]
    rng = random.Random(17 + family)
    strings = ["".join(rng.choice(alpha) for _ in range(rng.randint(1, 14))) for _ in range(200000)]
    got = rule_starts(rules_lib, family, kinds, strings)
    exp = oracle_starts(family, strings)
    bad = [(s, g, e) for s, g, e in zip(strings, got, exp) if g != e]
    assert not bad, bad[:5]


@pytest.mark.parametrize("family,profile", [(1, 0), (1, 1), (1, 2), (2, 1), (2, 2), (3, 3), (3, 1)])
def test_rules_generated_text(rules_lib, masks, family, profile):
    kinds = raw_kinds(masks, family)
    strings = [synth.transcript(100 + i, 20000, profile).decode() for i in range(8)]
    strings.append(synth.adversarial(7, 300000).decode())
    assert rule_starts(rules_lib, family, kinds, strings) == oracle_starts(family, strings)
