"""Pins for the oracle's byte spans: for every ID, the half-open range of
source bytes it encodes (TokTier §3: the session state a repair step edits
holds IDs and byte spans; §4.4: the paper's GPU path returns IDs without
them).  The oracle tracks each symbol's start through the merges; here that
is checked against what fixes it independently: a textbook every-pair BPE
whose token byte lengths, laid end to end, give the spans (every string of
length <= 6 over a hand vocabulary), the vocabulary bytes of each ID equal to
the source bytes of its span, spans that tile each request in order without
crossing a piece boundary, and no spans for a rejected request."""
import numpy as np

import brute
import oracle
from exact_bpe_tokenization_gb300 import synth
from test_oracle_bpe import hand_vocab, tables


def textbook_spans(data, ranks, results, index, toks):
    ids = brute.textbook_bpe(data, ranks, results, whole=index)
    spans, p = [], 0
    for i in ids:
        spans.append((p, p + len(toks[i])))
        p += len(toks[i])
    return ids, spans


def test_spans_equal_textbook_token_lengths_on_every_short_string():
    m, vb, vo, toks = hand_vocab()
    o = oracle.Oracle(m, vb, vo, 1)
    ranks, results, index = tables(m, toks)
    for s in brute.all_strings("abcd", 6):            # letters only: one piece per string
        b = s.encode()
        got = o.run_spans(b, np.array([0, len(b)], dtype=np.int64))
        want_ids, want_spans = textbook_spans(b, ranks, results, index, toks)
        assert got["ids"].tolist() == want_ids, s
        assert [tuple(x) for x in got["spans"].tolist()] == want_spans, s


def check_batch(o, vb, vo, reqs):
    data, offs = synth.batch(reqs)
    got = o.run_spans(data, offs, threads=4)
    ref = o.run(data, offs, threads=4)
    assert np.array_equal(got["ids"], ref["ids"]) and np.array_equal(got["id_offsets"], ref["id_offsets"])
    io, ps, po = got["id_offsets"], ref["piece_starts"], ref["piece_offsets"]
    base = int(offs[0])
    for r in range(len(offs) - 1):
        sp = got["spans"][io[r]:io[r + 1]]
        if got["status"][r] != 0:
            assert len(sp) == 0
            continue
        lo, hi = int(offs[r]) - base, int(offs[r + 1]) - base
        if hi == lo:
            assert len(sp) == 0
            continue
        assert sp[0, 0] == lo and sp[-1, 1] == hi
        assert np.array_equal(sp[1:, 0], sp[:-1, 1]) and np.all(sp[:, 1] > sp[:, 0])
        # every piece start is the start of some ID's span
        assert set((ps[po[r]:po[r + 1]] - base).tolist()) <= set(sp[:, 0].tolist())
    for i, (a, b) in zip(got["ids"].tolist(), got["spans"].tolist()):
        assert bytes(vb[vo[i]:vo[i + 1]]) == data[a:b].tobytes()


def test_spans_tile_requests_and_match_vocabulary_bytes():
    for profile, family, name, scale in ((synth.PROFILE_MIXED, 1, "single_1m_mixed", 0.01),
                                         (synth.PROFILE_MIXED, 1, "adversarial_4_4m", 0.004),
                                         (synth.PROFILE_CAMEL_MARKS, 2, "o200k_256_lognormal", 0.0005)):
        m, vb, vo = synth.make_vocab(profile, 1 << 20, 8000)
        o = oracle.Oracle(m, vb, vo, family)
        reqs = synth.workload(name, scale=scale)
        # an empty request, a rejected one (a lone continuation byte) and a one-byte one
        reqs = reqs[:3] + [b"", b"ab\x80cd", b"x"] + reqs[3:]
        check_batch(o, vb, vo, reqs)
