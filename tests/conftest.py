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
