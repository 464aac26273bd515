import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def masks():
    import oracle
    return oracle.class_table()


@pytest.fixture(scope="session")
def small_vocabs():
    """Vocabularies small enough to train in a second, per family:
    {family: (merges, vocab_bytes, vocab_offsets)}."""
    from exact_bpe_tokenization_gb300 import synth
    return {
        1: synth.make_vocab(synth.PROFILE_MIXED, 1 << 20, 8000),
        2: synth.make_vocab(synth.PROFILE_CAMEL_MARKS, 1 << 20, 8000),
    }


def concat_requests(strings):
    """bytes + int64 offsets of a list of str/bytes requests."""
    bs = [s.encode("utf-8") if isinstance(s, str) else bytes(s) for s in strings]
    offs = np.zeros(len(bs) + 1, dtype=np.int64)
    np.cumsum([len(b) for b in bs], out=offs[1:])
    return b"".join(bs), offs


def permute_vocab(merges, vb, vo, seed):
    """The same vocabulary under a random renumbering of all its token IDs
    (byte tokens included): returns (merges, vocab_bytes, vocab_offsets,
    perm) with old ID i renamed perm[i].  Rank order is unchanged."""
    n = len(vo) - 1
    perm = np.random.default_rng(seed).permutation(n).astype(np.int64)
    inv = np.empty(n, dtype=np.int64)
    inv[perm] = np.arange(n)
    toks = [bytes(vb[vo[inv[j]]:vo[inv[j] + 1]]) for j in range(n)]
    offs = np.zeros(n + 1, dtype=np.int64)
    np.cumsum([len(t) for t in toks], out=offs[1:])
    m = perm[np.asarray(merges, dtype=np.int64)].astype(np.int32)
    return m, np.frombuffer(b"".join(toks), dtype=np.uint8).copy(), offs, perm
