"""Plant plausible mistakes in copies of the oracle (compiled on the CPU) and
check that the pins catch every one; plant ID faults into an oracle output
and check that the parity comparator flags each (cf. TokTier §5.7: the
verifier is validated by injecting substitution, deletion, duplication,
adjacent-swap and same-length tail-resplit faults)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import brute
import oracle
from compare import compare_segmented
from test_oracle_bpe import hand_vocab, tables

SRC = os.path.join(os.path.dirname(oracle.oracle.__file__), "oracle.c")

MUTANTS = {
    # (original text, replacement, which pin catches it)
    "digits_up_to_4": ("while (k < 3 && p + k < n && isN", "while (k < 4 && p + k < n && isN", "pretok"),
    "no_whitespace_lookahead": ("for (int64_t k = w; k >= 1; --k)\n    if (p + k == n || isS",
                                "for (int64_t k = w; k >= w; --k)\n    if (p + k == n || isS", "pretok"),
    "no_newline_absorption": ("q += k; return q + count_while(o, c, n, q, isCRLFo);", "q += k; return q;", "pretok"),
    "contraction_ll_missing": ("if (a == 'l' && b == 'l') return 3;", "", "pretok"),
    "prefix_allows_newline": ("return !isCRLF(c) && !isL(o, c) && !isN(o, c); }",
                              "return !isL(o, c) && !isN(o, c); }", "pretok"),
    "o200k_lower_set_without_marks": ("(B_LL | B_LM | B_LO | B_M); }", "(B_LL | B_LM | B_LO); }", "pretok2"),
    "bpe_rightmost_on_ties": ("if (rank[i] >= 0 && (best < 0 || rank[i] < best)) { best = rank[i]; at = i; }\n    if (best < 0) break;\n    ids[at] = o->mresult[best];\n    memmove(ids + at + 1, ids + at + 2, sizeof(int32_t) * (size_t)(n - at - 2));\n    if (sstart)",
                              "if (rank[i] >= 0 && (best < 0 || rank[i] <= best)) { best = rank[i]; at = i; }\n    if (best < 0) break;\n    ids[at] = o->mresult[best];\n    memmove(ids + at + 1, ids + at + 2, sizeof(int32_t) * (size_t)(n - at - 2));\n    if (sstart)", "bpe"),
    "no_whole_piece_shortcut": ("  if (whole >= 0) {\n    ids[0] = (int32_t)whole;",
                                "  if (0 && whole >= 0) {\n    ids[0] = (int32_t)whole;", "bpe"),
    "stale_left_rank": ("    if (at > 0) rank[at - 1] = merge_rank(o, ids[at - 1], ids[at]);\n    if (at + 1 < n) rank[at] = merge_rank(o, ids[at], ids[at + 1]);\n  }\n  return n;\n}\n\nstatic int64_t encode_piece(",
                        "    if (at + 1 < n) rank[at] = merge_rank(o, ids[at], ids[at + 1]);\n  }\n  return n;\n}\n\nstatic int64_t encode_piece(", "bpe"),
    "span_keeps_right_start": ("if (sstart) memmove(sstart + at + 1, sstart + at + 2,", "if (sstart) memmove(sstart + at, sstart + at + 1,",
                               "spans"),
    "literal_shortest": ("    if (len > best_len && x + len <= nb", "    if ((best < 0 || len < best_len) && x + len <= nb", "literals"),
    "surrogates_accepted": ("(c >= 0xD800 && c <= 0xDFFF)", "(0)", "utf8"),
    "deepseek_katakana_missing": ("(c >= 0x3040 && c <= 0x30FF) || (c >= 0x4E00", "(c >= 0x3040 && c <= 0x309F) || (c >= 0x4E00",
                                  "pretok3"),
    "deepseek_gap_dropped": ("    if (q > p) k = ds_emit(o, stage, c, p, q, starts, k);\n", "", "pretok3"),
    "deepseek_no_rescan_of_pieces": ("  if (stage == 3) { starts[k] = a; return k + 1; }",
                                     "  if (stage >= 2) { starts[k] = a; return k + 1; }", "pretok3"),
}


def build_mutant(name, tmp_path):
    old, new, _ = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / ("oracle_%s.c" % name)
    path.write_text(src.replace(old, new))
    so = tmp_path / ("liboracle_%s.so" % name)
    subprocess.check_call(["gcc", "-O1", "-std=gnu11", "-shared", "-fPIC", "-pthread", "-o", str(so), str(path)])
    return oracle.oracle.load_lib(str(so))


def pretok_pin_fails(lib, family, masks):
    ast = brute.family_ast(family, masks)
    alpha = {1: ["a", "s", "1", " ", "\t", "\n", "\r", "'", ".", "l"],
             2: ["a", "B", "1", " ", "\n", "'", ".", "か", "́", "\U0001F642"]}[family]
    pt = oracle.pretokenizer(family, lib=lib)
    for s in brute.all_strings(alpha, 4):
        if pt.pieces(s) != brute.brute_pieces(ast, s):
            return True
    return False


def deepseek_pin_fails(lib, masks):
    asts = brute.deepseek_asts(masks)
    pt = oracle.pretokenizer(3, lib=lib)
    for s in brute.all_strings(["a", "1", " ", "\n", "'", ".", "日", "・", "s"], 4):
        if pt.pieces(s) != brute.split_sequence(asts, s):
            return True
    return False


def spans_pin_fails(lib):
    from test_oracle_spans import textbook_spans
    m, vb, vo, toks = hand_vocab()
    o = oracle.Oracle(m, vb, vo, 1, lib=lib)
    ranks, results, index = tables(m, toks)
    for s in brute.all_strings("abcd", 6):
        b = s.encode()
        got = o.run_spans(b, np.array([0, len(b)], dtype=np.int64))
        if [tuple(x) for x in got["spans"].tolist()] != textbook_spans(b, ranks, results, index, toks)[1]:
            return True
    return False


def literals_pin_fails(lib):
    from exact_bpe_tokenization_gb300 import synth
    m, vb, vo = synth.make_vocab(synth.PROFILE_ASCII, 1 << 20, 4096)
    o = oracle.Oracle(m, vb, vo, 1, lib=lib)
    n = len(vo) - 1
    o.set_added_tokens({b"ab": n + 1, b"abc": n + 2})
    r = o.run(b"abcd", np.array([0, 4], dtype=np.int64))
    return r["ids"].tolist()[:1] != [n + 2]


def bpe_pin_fails(lib):
    m, vb, vo, toks = hand_vocab()
    o = oracle.Oracle(m, vb, vo, 1, lib=lib)
    ranks, results, index = tables(m, toks)
    for s in brute.all_strings("abcd", 6):
        if o.encode_bytes(s.encode()) != brute.textbook_bpe(s.encode(), ranks, results, whole=index):
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_oracle_fault_is_caught(name, tmp_path, masks):
    lib = build_mutant(name, tmp_path)
    kind = MUTANTS[name][2]
    if kind == "pretok":
        assert pretok_pin_fails(lib, 1, masks)
    elif kind == "pretok2":
        assert pretok_pin_fails(lib, 2, masks)
    elif kind == "pretok3":
        assert deepseek_pin_fails(lib, masks)
    elif kind == "bpe":
        assert bpe_pin_fails(lib)
    elif kind == "spans":
        assert spans_pin_fails(lib)
    elif kind == "literals":
        assert literals_pin_fails(lib)
    else:
        pt = oracle.pretokenizer(1, lib=lib)
        bad = b"\xed\xa0\x80"
        assert pt.run(bad, np.array([0, 3]), ids=False)["status"][0] == 0   # mutant accepts
        with pytest.raises(UnicodeDecodeError):
            bad.decode("utf-8")                                            # the pin rejects


def test_unmutated_oracle_passes_the_same_pins(masks):
    lib = oracle.oracle._get()
    assert not pretok_pin_fails(lib, 1, masks)
    assert not pretok_pin_fails(lib, 2, masks)
    assert not deepseek_pin_fails(lib, masks)
    assert not bpe_pin_fails(lib)
    assert not spans_pin_fails(lib)
    assert not literals_pin_fails(lib)


@pytest.mark.parametrize("fault", ["substitute", "delete", "duplicate", "swap", "tail_resplit"])
def test_comparator_catches_planted_id_faults(fault, small_vocabs):
    from exact_bpe_tokenization_gb300 import synth
    m, vb, vo = small_vocabs[1]
    o = oracle.Oracle(m, vb, vo, 1)
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    reqs = [synth.transcript(40 + i, 3000, 1) for i in range(4)]
    data, offs = synth.batch(reqs)
    r = o.run(data, offs)
    ids, io = r["ids"].copy(), r["id_offsets"].copy()
    assert compare_segmented(r["ids"], r["id_offsets"], ids, io) == []
    got = ids.tolist()
    k = int(io[2]) + 17
    if fault == "substitute":
        got[k] = (got[k] + 1) % len(toks)
    elif fault == "delete":
        del got[k]
        io[3:] -= 1
    elif fault == "duplicate":
        got.insert(k, got[k])
        io[3:] += 1
    elif fault == "swap":
        j = next(j for j in range(k, len(got) - 1) if got[j] != got[j + 1])
        got[j], got[j + 1] = got[j + 1], got[j]
    else:   # same-length tail resplit: two tokens re-cut into two others with the same bytes
        index = {t: i for i, t in enumerate(toks)}
        for j in range(int(io[2]), int(io[3]) - 1):
            both = toks[got[j]] + toks[got[j + 1]]
            alt = [(index.get(both[:c]), index.get(both[c:])) for c in range(1, len(both))]
            alt = [a for a in alt if None not in a and a != (got[j], got[j + 1])]
            if alt:
                got[j], got[j + 1] = alt[0]
                break
        else:
            pytest.fail("no resplit found")
    assert compare_segmented(r["ids"], r["id_offsets"], np.array(got), io)
