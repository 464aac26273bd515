"""GPU span export (tt_encode_batch_spans) against the oracle's tracked byte
spans, element by element, with the IDs and ID offsets: the paper's GPU path
returns IDs without spans, so a state miss that must build session state
falls back to the CPU (TokTier §4.4); these tests hold the GPU spans to the
oracle on every workload shape, including the block paths for long pieces
(shared-memory lists up to 8 KiB, global memory beyond), rejected and empty
requests, and graph replay mixed with the plain entry point."""
import os

import numpy as np
import pytest

import oracle
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


def spans_parity(binding, vocab, family, reqs, plain_between=False):
    merges, vb, vo = vocab
    data, offs = synth.batch(reqs)
    ref = oracle.Oracle(merges, vb, vo, family).run_spans(data, offs, threads=NCPU)
    tok = binding.Tokenizer(merges, vb, vo, family)
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    for rep in range(2):                               # capture, then replay
        ids, io, sp = tok.encode_spans(d, o)
        if plain_between:
            tok.encode(d, o)                           # same graph, no spans requested
        torch.cuda.synchronize()
        io = io.cpu().numpy()
        t = int(io[-1])
        assert np.array_equal(io, ref["id_offsets"]), rep
        assert np.array_equal(ids[:t].cpu().numpy(), ref["ids"]), rep
        got = sp[:t].cpu().numpy().astype(np.int64)
        bad = np.nonzero(np.any(got != ref["spans"], axis=1))[0]
        assert len(bad) == 0, "first span mismatch at ID %d: got %s want %s" % (
            bad[0], got[bad[0]].tolist(), ref["spans"][bad[0]].tolist())
    tok.close()


@pytest.fixture(scope="module")
def c1_vocab():
    return synth.make_vocab(synth.PROFILE_MIXED, 8 << 20, 100000)


def test_spans_tiny_ascii(cuda):
    spans_parity(cuda, synth.make_vocab(synth.PROFILE_ASCII, 1 << 20, 4096), 1, synth.workload("tiny_ascii_64k"))


def test_spans_single_1m_mixed_full_size(cuda, c1_vocab):
    spans_parity(cuda, c1_vocab, 1, synth.workload("single_1m_mixed", seed=3), plain_between=True)


def test_spans_burst_scaled(cuda, c1_vocab):
    spans_parity(cuda, c1_vocab, 1, synth.workload("burst_64_loguniform", scale=0.05))


def test_spans_adversarial_full_size(cuda, c1_vocab):
    # 50K-blank pieces (global-memory block path), 5K punctuation runs (shared memory)
    spans_parity(cuda, c1_vocab, 1, synth.workload("adversarial_4_4m"))


def test_spans_o200k_scaled(cuda):
    vocab = synth.make_vocab(synth.PROFILE_CAMEL_MARKS, 16 << 20, 200000)
    spans_parity(cuda, vocab, 2, synth.workload("o200k_256_lognormal", scale=0.02))


def test_spans_rejected_and_empty_requests(cuda, c1_vocab):
    base = synth.workload("single_1m_mixed", seed=5, scale=0.01)[0]
    reqs = [b"", base[:500], b"ok \xc3(", b"", base[500:3000], b"\xf0\x9f\x98", b"x", b""]
    spans_parity(cuda, c1_vocab, 1, reqs)
