"""Values the pages print, stored under tests/golden/ with their citations,
checked against the oracle (and, where a GPU is present, the CUDA path)."""
import json
import os

import numpy as np
import pytest

import oracle
from exact_bpe_tokenization_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        g = json.load(f)
    assert g["cite"]
    return g


def seam_vocab():
    """A synthetic vocabulary holding the three strings of the example."""
    text = (" pipeline" * 3000 + " pipe" * 4000 + " (line" * 4000 + "\n").encode()
    merges = synth.train_merges(text, 40)
    vb, vo = synth.vocab_from_merges(merges)
    toks = [bytes(vb[vo[i]:vo[i + 1]]) for i in range(len(vo) - 1)]
    return merges, vb, vo, toks


@pytest.mark.parametrize("family", [1, 2, 3])
def test_seam_example_pieces(family):
    g = load("seam_pipeline.json")
    pt = oracle.pretokenizer(family)
    assert pt.pieces(g["left"] + g["right"]) == g["whole_pieces"]
    assert pt.pieces(g["left"]) == g["left_pieces"]
    assert pt.pieces(g["right"]) == g["right_pieces"]


@pytest.mark.parametrize("family", [1, 2, 3])
def test_seam_example_token_counts(family):
    g = load("seam_pipeline.json")
    merges, vb, vo, toks = seam_vocab()
    o = oracle.Oracle(merges, vb, vo, family)
    whole = o.encode(g["left"] + g["right"])
    parts = [o.encode(g["left"]), o.encode(g["right"])]
    assert len(whole) == g["whole_token_count"]
    assert [len(p) for p in parts] == g["separate_token_counts"]
    assert parts[0] + parts[1] != whole
    assert [toks[i] for i in whole] == [x.encode() for x in g["whole_pieces"]]


@pytest.mark.gpu
@pytest.mark.parametrize("family", [1, 2, 3])
def test_seam_example_on_the_gpu(family):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from exact_bpe_tokenization_gb300 import binding
    g = load("seam_pipeline.json")
    merges, vb, vo, _ = seam_vocab()
    reqs = [(g["left"] + g["right"]).encode(), g["left"].encode(), g["right"].encode()]
    data, offs = synth.batch(reqs)
    ref = oracle.Oracle(merges, vb, vo, family).run(data, offs)
    tok = binding.Tokenizer(merges, vb, vo, family)
    ids, io = tok.encode(torch.from_numpy(data).cuda(), torch.from_numpy(offs).cuda())
    io = io.cpu().numpy()
    assert np.array_equal(io, ref["id_offsets"])
    assert np.array_equal(ids[:int(io[-1])].cpu().numpy(), ref["ids"])
    assert list(np.diff(io)) == [g["whole_token_count"]] + g["separate_token_counts"]
    tok.close()
