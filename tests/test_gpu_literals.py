"""Added-token literal extraction on the GPU (tt_set_added_tokens) against
the oracle, per piece boundary, per ID and per byte span (TokTier §4.4:
added and special tokens are literal strings reserved as single IDs,
extracted leftmost-longest before the tokenizer family handles the remaining
segments).  Covers literals in generated text, dense overlapping literals
across tile edges, literals at request edges, rejected and empty requests,
both pattern families, a full-size request, removing the set and invalid
sets (the allocation-free entry point with literals: test_zz_no_alloc.py)."""
import os

import numpy as np
import pytest

import oracle
from compare import compare_segmented
from exact_bpe_tokenization_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
NCPU = os.cpu_count() or 1


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from exact_bpe_tokenization_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def c1_vocab():
    return synth.make_vocab(synth.PROFILE_MIXED, 8 << 20, 100000)


def special(vocab):
    n = len(vocab[2]) - 1
    return {b"<|endoftext|>": n + 7, b"<|im_start|>": n + 8, b"<|im_end|>": n + 9, b"<|im": n + 10,
            "<|ユーザー|>".encode(): n + 11}


def sprinkle(texts, literals, seed, every=700):
    rng = np.random.default_rng(seed)
    keys = list(literals)
    out = []
    for t in texts:
        parts, prev = [], 0
        for c in sorted(rng.integers(0, max(len(t), 1), max(len(t) // every, 1)).tolist()):
            while c < len(t) and (t[c] & 0xC0) == 0x80:     # cut on a char boundary
                c += 1
            parts += [t[prev:c], keys[int(rng.integers(len(keys)))]]
            prev = c
        out.append(b"".join(parts) + t[prev:])
    return out


def parity(binding, vocab, family, literals, reqs):
    merges, vb, vo = vocab
    data, offs = synth.batch(reqs)
    orc = oracle.Oracle(merges, vb, vo, family)
    orc.set_added_tokens(literals)
    ref = orc.run(data, offs, threads=NCPU)
    refs = orc.run_spans(data, offs, threads=NCPU)
    tok = binding.Tokenizer(merges, vb, vo, family)
    tok.set_added_tokens(literals)
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    for rep in range(2):
        ids, io, sp = tok.encode_spans(d, o)
        starts, po = tok.pretokenize(d, o)
        torch.cuda.synchronize()
        io, po = io.cpu().numpy(), po.cpu().numpy()
        errs = compare_segmented(ref["piece_starts"], ref["piece_offsets"], starts[:int(po[-1])].cpu().numpy(), po,
                                 "pieces")
        errs += compare_segmented(ref["ids"], ref["id_offsets"], ids[:int(io[-1])].cpu().numpy(), io, "ids")
        assert not errs, "\n".join(errs)
        assert np.array_equal(sp[:int(io[-1])].cpu().numpy().astype(np.int64), refs["spans"]), rep
    st, bad = tok.status()
    bad_ref = np.nonzero(ref["status"])[0]
    assert (st == 0) if not len(bad_ref) else (st == binding.TT_ERR_INVALID_UTF8 and bad == int(bad_ref[0]))
    tok.close()


def test_literals_in_generated_text(cuda, c1_vocab):
    lits = special(c1_vocab)
    parity(cuda, c1_vocab, 1, lits, sprinkle(synth.workload("burst_64_loguniform", scale=0.02), lits, 1))


def test_dense_overlapping_literals_across_tiles(cuda, c1_vocab):
    n = len(c1_vocab[2]) - 1
    lits = {b"<a>": n + 1, b"<a>b": n + 2, b"a>": n + 3, b" <": n + 4, b"b b": n + 5, b"1\n": n + 6, b"  ": n + 7}
    rng = np.random.default_rng(5)
    frags = [b"<a>", b"<a>b", b"a>", b" <", b"b b", b"1\n", b"x", b" ", b"<", b">", b"b", b"a"]
    reqs = [b"".join(frags[int(i)] for i in rng.integers(0, len(frags), size)) for size in (60000, 7, 1, 2000)]
    parity(cuda, c1_vocab, 1, lits, reqs)


def test_literals_at_request_edges_rejected_and_empty(cuda, c1_vocab):
    lits = special(c1_vocab)
    reqs = [b"<|endoftext|>", b"", b"abc<|im_end|>", b"<|im_start|>user\n hi", b"bad \xff <|im", b"<|im<|im_end|>",
            b"<|endoftext|><|endoftext|>", b"", "x<|ユーザー|>y".encode()]
    parity(cuda, c1_vocab, 1, lits, reqs)


def test_literals_o200k(cuda):
    vocab = synth.make_vocab(synth.PROFILE_CAMEL_MARKS, 1 << 20, 8000)
    lits = special(vocab)
    parity(cuda, vocab, 2, lits, sprinkle(synth.workload("o200k_256_lognormal", scale=0.002), lits, 2, every=300))


def test_literals_full_size_request(cuda, c1_vocab):
    lits = special(c1_vocab)
    parity(cuda, c1_vocab, 1, lits, sprinkle(synth.workload("single_1m_mixed", seed=9), lits, 3, every=2000))


def test_removing_the_set_restores_plain_output(cuda, c1_vocab):
    merges, vb, vo = c1_vocab
    lits = special(c1_vocab)
    data, offs = synth.batch(sprinkle(synth.workload("single_1m_mixed", seed=4, scale=0.02), lits, 4))
    ref = oracle.Oracle(merges, vb, vo, 1).run(data, offs)
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    d, o = torch.from_numpy(data).cuda(), torch.from_numpy(offs).cuda()
    tok.set_added_tokens(lits)
    tok.encode(d, o)
    tok.set_added_tokens({})
    ids, io = tok.encode(d, o)
    torch.cuda.synchronize()
    assert np.array_equal(ids[:int(io[-1].item())].cpu().numpy(), ref["ids"])
    tok.close()


@pytest.mark.parametrize("case", ["duplicate", "id_in_vocab", "invalid_utf8", "empty", "too_long", "duplicate_id"])
def test_invalid_literal_sets_are_rejected(cuda, c1_vocab, case):
    merges, vb, vo = c1_vocab
    n = len(vo) - 1
    lits = {"duplicate": [(b"<a>", n + 1), (b"<a>", n + 2)], "id_in_vocab": [(b"<a>", 5)],
            "invalid_utf8": [(b"<\xc3>", n + 1)], "empty": [(b"", n + 1)], "too_long": [(b"x" * 256, n + 1)],
            "duplicate_id": [(b"<a>", n + 1), (b"<b>", n + 1)]}[case]
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    data = np.frombuffer(b"".join(k for k, _ in lits) + b"\0", dtype=np.uint8).copy()   # never a NULL pointer
    offs = np.zeros(len(lits) + 1, dtype=np.int64)
    np.cumsum([len(k) for k, _ in lits], out=offs[1:])
    ids = np.array([v for _, v in lits], dtype=np.int32)
    rc = cuda.lib().tt_set_added_tokens(tok.h, data.ctypes.data, offs.ctypes.data, ids.ctypes.data, len(lits))
    assert rc == cuda.TT_ERR_BAD_VOCAB
    tok.close()
