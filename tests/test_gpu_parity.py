"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle,
bit-exact per piece boundary and per token ID (TokTier §4.1: both levels,
because the ID level can hide a boundary fault), on the same seeded inputs.

Covers the five workloads at full size, brute-force batches of tiny
requests (document-boundary cuts, §4.3), runs straddling tiles at every
alignment, long-piece lengths around the execution-unit thresholds, empty
and invalid requests, graph replay, the host-buffer entry point, several
streams and the status contract."""
import os
import random

import numpy as np
import pytest

import brute
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
def vocabs():
    return {
        "tiny": synth.make_vocab(synth.PROFILE_ASCII, 1 << 20, 4096),
        "small1": synth.make_vocab(synth.PROFILE_MIXED, 1 << 20, 8000),
        "small2": synth.make_vocab(synth.PROFILE_CAMEL_MARKS, 1 << 20, 8000),
        "c1": synth.make_vocab(synth.PROFILE_MIXED, 8 << 20, 100000),
    }


def run_gpu(binding, tok, data, offs, stream=None, graph_repeats=1):
    d = torch.from_numpy(np.ascontiguousarray(data)).cuda()
    o = torch.from_numpy(np.ascontiguousarray(offs)).cuda()
    for _ in range(graph_repeats):
        ids, io = tok.encode(d, o, stream=stream)
    starts, po = tok.pretokenize(d, o, stream=stream)
    torch.cuda.synchronize()
    status, bad = tok.status(stream)
    io = io.cpu().numpy()
    po = po.cpu().numpy()
    return {"ids": ids[:int(io[-1])].cpu().numpy(), "id_offsets": io,
            "piece_starts": starts[:int(po[-1])].cpu().numpy(), "piece_offsets": po,
            "status": status, "bad": bad}


def check(binding, vocab, family, reqs, threads=NCPU, expect_status=0):
    merges, vb, vo = vocab
    data, offs = synth.batch([r.encode() if isinstance(r, str) else r for r in reqs])
    tok = binding.Tokenizer(merges, vb, vo, family)
    got = run_gpu(binding, tok, data, offs)
    ref = oracle.Oracle(merges, vb, vo, family).run(data, offs, threads=threads)
    errs = compare_segmented(ref["piece_starts"], ref["piece_offsets"], got["piece_starts"], got["piece_offsets"],
                             "pieces")
    errs += compare_segmented(ref["ids"], ref["id_offsets"], got["ids"], got["id_offsets"], "ids")
    assert not errs, "\n".join(errs)
    bad_ref = np.nonzero(ref["status"])[0]
    if len(bad_ref):
        assert got["status"] == binding.TT_ERR_INVALID_UTF8 and got["bad"] == int(bad_ref[0])
    else:
        assert got["status"] == expect_status
    tok.close()
    return got


# ------------------------------------------------------------ brute force
ALPHABETS = {
    1: ["a", "s", "1", " ", "\t", "\n", "\r", "'", ".", "é"],
    2: ["a", "B", "1", " ", "\n", "'", ".", "か", "́", "\U0001F642"],
    3: ["s", "T", "'", "a", "か", "́", " ", ".", "E", "r"],
}


@pytest.mark.parametrize("family,alphabet", [(1, 1), (2, 2), (2, 3), (1, 3)])
def test_all_short_strings_as_tiny_requests(cuda, vocabs, family, alphabet):
    """Every string of length <= 5 (111,110 requests in one batch)."""
    reqs = list(brute.all_strings(ALPHABETS[alphabet], 5))
    check(cuda, vocabs["small%d" % family], family, reqs)


@pytest.mark.parametrize("family", [1, 2])
def test_random_mixed_strings(cuda, vocabs, family):
    alpha = ALPHABETS[family] + ["A", "t", "e", "r", "l", "m", "d", "v", "́", " ", "　", "٣", "ʰ", "ǅ", "Ü", "\t",
                                 "\r", "0", "_", "(", "一"]
    rng = random.Random(31 + family)
    reqs = ["".join(rng.choice(alpha) for _ in range(rng.randint(1, 40))) for _ in range(60000)]
    check(cuda, vocabs["small%d" % family], family, reqs)


# ------------------------------------------------------------ workloads
def test_tiny_ascii_64k(cuda, vocabs):
    check(cuda, vocabs["tiny"], 1, synth.workload("tiny_ascii_64k"))


@pytest.mark.parametrize("seed", [1, 2, 17])
def test_single_1m_mixed(cuda, vocabs, seed):
    check(cuda, vocabs["c1"], 1, synth.workload("single_1m_mixed", seed=seed))


def test_burst_64_loguniform_full(cuda, vocabs):
    check(cuda, vocabs["c1"], 1, synth.workload("burst_64_loguniform"))


def test_adversarial_4_4m_full(cuda, vocabs):
    check(cuda, vocabs["c1"], 1, synth.workload("adversarial_4_4m"))


def test_o200k_256_lognormal_full(cuda):
    vocab = synth.make_vocab(synth.PROFILE_CAMEL_MARKS, 16 << 20, 200000)
    check(cuda, vocab, 2, synth.workload("o200k_256_lognormal"))


# ------------------------------------------------------------ tiles and lengths
PATHOLOGICAL = [
    "7" * 10000, " " * 20000 + "x", "\r\n\r\n \n" * 900, ".,;:!" * 1200, "a " * 5000, "一" * 3000,
    "x'd" + "'d" * 3000, "a" + "か" * 4000 + "B", "a" + "か" * 4000 + "Bc", "..́" + ".́" * 3000 + "a",
    "\t" * 9000 + "\n" * 9000 + "y", "aB" * 3000, "ǅ" * 5000, "1 " * 4000,
]


@pytest.mark.parametrize("family", [1, 2])
def test_runs_straddling_tiles_at_every_alignment(cuda, vocabs, family):
    """Each pathological run is preceded by 0..47 filler bytes, so its start,
    end and internal events fall at every offset mod 16 relative to the
    4016-byte tiles and the 16-byte lanes."""
    reqs = []
    for k, run in enumerate(PATHOLOGICAL):
        for pad in range(0, 48, 3 if k % 2 else 1):
            reqs.append("q" * pad + " " + run + " tail")
    check(cuda, vocabs["small%d" % family], family, reqs)
    # and as one single request (runs cut only by content, not by documents)
    check(cuda, vocabs["small%d" % family], family, ["z".join(reqs[::7])])


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 34, 64, 127, 128, 129, 1000, 4095, 4096, 4097, 50000])
def test_piece_lengths_around_unit_thresholds(cuda, vocabs, n):
    reqs = [" " * n + "x", "(" * n + "a", "a" * n, "é" * (n // 2 + 1), "一" * (n // 3 + 1), "b" * n + " ",
            "\U0001F642" * (n // 4 + 1)]
    check(cuda, vocabs["c1"], 1, reqs)


def test_pieces_merged_two_to_a_warp_in_large_batches(cuda, vocabs):
    """Batches beyond 4 MiB merge the pieces of 49..128 bytes two to a warp
    and those of 17..48 bytes four to a warp: pieces of every length around
    those ranges (letters, CJK, punctuation, whole tokens and misses side by
    side, counts that leave a group part-filled) inside 4.3 MB of text."""
    reqs = []
    for n in range(15, 133):
        reqs += [" " + "a" * n, "日" * (n // 3 + 1), "(" * n, "ab" * (n // 2) + " x", "é" * (n // 2)]
    reqs.append("q" * 77)
    filler = synth.transcript(77, 3_500_000, synth.PROFILE_MIXED)
    check(cuda, vocabs["c1"], 1, reqs + [filler] + reqs[::-1])


@pytest.mark.parametrize("large", [False, True])
def test_out_of_order_merges_on_small_alphabets(cuda, large):
    """Letter pieces of 17..90 chars over two- and three-symbol alphabets
    (ASCII letters, a 2-byte and a 3-byte letter), runs of one letter among
    them, with a vocabulary of 3,000 merges trained on the same text: merges
    overlap and most pairs have a lower-ranked rival on one side, so merging
    a pair out of rank order when some lower-ranked merge could still take
    one of its tokens would change the IDs.  large: a batch beyond 4 MiB
    (pieces two and four to a warp)."""
    rng = random.Random(5)
    words = []
    for _ in range(3000):
        alpha = rng.choice(["ab", "abc", "ab日", "aé", "a"])
        words.append("".join(rng.choice(alpha) for _ in range(rng.randint(17, 90))))
    reqs = [" ".join(words[i:i + 30]) for i in range(0, len(words), 30)]
    merges = synth.train_merges(" ".join(reqs).encode(), 3000)
    vb, vo = synth.vocab_from_merges(merges)
    if large:
        reqs = reqs * 28
    check(cuda, (merges, vb, vo), 1, reqs)


@pytest.mark.parametrize("large", [False, True])
def test_renumbered_token_ids(cuda, vocabs, large):
    """The 100K-merge vocabulary with every token ID renumbered at random
    (byte tokens included): the byte-to-token map, the direct byte-pair and
    context tables and the hashed tables must all go through IDs, never
    assume that byte b is token b.  large: a batch beyond 4 MiB."""
    from conftest import permute_vocab
    m, vb, vo = vocabs["c1"]
    pm, pvb, pvo, _ = permute_vocab(m, vb, vo, 8)
    reqs = [synth.transcript(40 + i, 20000, synth.PROFILE_MIXED) for i in range(8)]
    if large:
        reqs.append(synth.transcript(49, 3_500_000, synth.PROFILE_MIXED))
    check(cuda, (pm, pvb, pvo), 1, reqs)


# ------------------------------------------------------------ edge cases
def test_empty_and_degenerate_batches(cuda, vocabs):
    merges, vb, vo = vocabs["small1"]
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    # n = 0
    o = torch.zeros(1, dtype=torch.int64, device="cuda")
    out = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    cuda.tt_encode_batch(tok.h, torch.zeros(1, dtype=torch.uint8, device="cuda"), o, 0,
                         torch.zeros(1, dtype=torch.int32, device="cuda"), out)
    torch.cuda.synchronize()
    assert out.item() == 0
    tok.close()
    check(cuda, vocabs["small1"], 1, [""])
    check(cuda, vocabs["small1"], 1, ["", "", ""])
    check(cuda, vocabs["small1"], 1, ["", "a", "", " ", "", "1", ""])


def test_invalid_utf8_requests_yield_no_ids(cuda, vocabs):
    bad = [b"\xff", b"a\xc3", b"\x80abc", b"\xed\xa0\x80", b"\xe0\x80\x80", b"\xf4\x90\x80\x80", b"\xc0\xaf",
           b"ok \xe2\x82", b"\xf0\x9f\x98"]
    good = [s.encode() for s in ["hello world", "don't 123456", "  \n\t x", "camelCase"]]
    reqs = []
    for i in range(len(bad)):
        reqs += [good[i % 4], bad[i]]
    reqs.append(good[0])
    got = check(cuda, vocabs["small1"], 1, reqs)
    io = got["id_offsets"]
    for r in range(1, len(reqs) - 1, 2):
        assert io[r + 1] == io[r]
    # a multi-byte char split across two requests is invalid on both sides
    check(cuda, vocabs["small1"], 1, ["ab\xc3".encode("latin-1"), b"\xa9cd", b"fine"])


@pytest.mark.parametrize("large", [False, True])
def test_utf8_sequences_straddling_tile_edges(cuda, vocabs, large):
    """Valid and invalid multi-byte sequences at every position across a
    4016-byte tile edge: each request is two tiles long and starts on a tile
    edge, so its sequence sits at the edge in its middle.  large: behind a
    filler that takes the batch past 4 MiB (the 16-bytes-a-thread kernels)."""
    tile = 4016
    seqs = ["é".encode(), "日".encode(), "\U0001F642".encode(), b"\xff", b"\xc3(", b"\x80", b"\xe4\xb8",
            b"\xe0\x80\x80", b"\xed\xa0\x80", b"\xf4\x90\x80\x80", b"\xf0\x9f\x98"]
    reqs = []
    if large:                                  # its length is a whole number of tiles too
        text, n = synth.transcript(78, 3_600_000, synth.PROFILE_MIXED), 1080 * tile
        cut = n
        while text[cut] & 0xC0 == 0x80:        # end on a char boundary
            cut -= 1
        reqs.append(text[:cut].ljust(n, b" "))
    for seq in seqs:
        for d in range(-5, 6):
            head = b"ab " * ((tile + d) // 3) + b"x" * ((tile + d) % 3)
            reqs.append((head + seq).ljust(2 * tile, b"z"))
    check(cuda, vocabs["c1"], 1, reqs)


@pytest.mark.parametrize("family", [1, 2, 3])
def test_carries_from_tiles_far_away(cuda, vocabs, family):
    """Runs of 35 tiles and more, so that a tile finds its carries several
    windows of 32 tile summaries away: a tab run before a letter and before
    CR/LF (the first later event of the reverse queries), an uppercase run
    before lowercase letters (o200k's rest-of-run-uppercase query), and
    combining marks far from the stretch start and trigger that decide
    whether they count as letters (o200k mark resolution).  The
    ASCII-trained vocabulary has no merges for these runs, which keeps the
    oracle fast."""
    n = 140_000
    reqs = ["\t" * n + "x", "\t" * n + "\r\n" + "y", "A" * n + "bc d", "x!!" + "\u0301" * (n // 2) + "a",
            "a" + "\u0301" * (n // 2) + " z", " " + "\u3042" * (n // 3) + "x", "tail"]
    check(cuda, vocabs["tiny"], family, reqs)


def test_offsets_with_nonzero_base(cuda, vocabs):
    merges, vb, vo = vocabs["small1"]
    reqs = [synth.transcript(3 + i, 5000, 1) for i in range(5)]
    data, offs = synth.batch(reqs)
    pad = 37
    data2 = np.concatenate([np.full(pad, 0x41, dtype=np.uint8), data])
    offs2 = offs + pad
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    d = torch.from_numpy(data2).cuda()
    o = torch.from_numpy(offs2).cuda()
    ids = torch.empty(len(data2), dtype=torch.int32, device="cuda")
    io = torch.empty(len(offs2), dtype=torch.int64, device="cuda")
    cuda.tt_encode_batch(tok.h, d, o, len(reqs), ids, io)
    io = io.cpu().numpy()
    ref = oracle.Oracle(merges, vb, vo, 1).run(data, offs)
    assert np.array_equal(io, ref["id_offsets"])
    assert np.array_equal(ids[:int(io[-1])].cpu().numpy(), ref["ids"])
    tok.close()


def test_graph_replay_eager_and_host_paths_agree(cuda, vocabs):
    merges, vb, vo = vocabs["c1"]
    reqs = synth.workload("burst_64_loguniform", scale=0.05)
    data, offs = synth.batch(reqs)
    ref = oracle.Oracle(merges, vb, vo, 1).run(data, offs, threads=NCPU)
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    outs = []
    for rep in range(3):                         # first call captures, later ones replay
        ids, io = tok.encode(d, o)
        torch.cuda.synchronize()
        outs.append((ids[:int(io[-1].item())].cpu().numpy(), io.cpu().numpy()))
    cuda.tt_profile(tok.h, 1)                    # eager launches with events
    ids, io = tok.encode(d, o)
    prof = cuda.tt_profile_read(tok.h)
    cuda.tt_profile(tok.h, 0)
    outs.append((ids[:int(io[-1].item())].cpu().numpy(), io.cpu().numpy()))
    hids, hio, st = tok.encode_host(data, offs)
    outs.append((hids, hio))
    for i, (a, b) in enumerate(outs):
        assert np.array_equal(b, ref["id_offsets"]), i
        assert np.array_equal(a, ref["ids"]), i
    assert st == 0
    assert set(prof) >= {"k_prepass", "k_pretok", "k_bpe_warp", "k_ids"} and all(v[1] == 1 for v in prof.values())
    tok.close()


def test_host_entry_point_pinned_direct_and_staged(cuda, vocabs):
    """tt_encode_host with page-locked input (read in place by the pre-pass)
    or pageable input (copied), and page-locked output buffers (written by the
    kernels directly) or pageable, mixed or too-small ones (staged and copied
    back): the same IDs and offsets, the same status for a rejected request,
    and repeated calls reusing the buffers."""
    merges, vb, vo = vocabs["c1"]
    reqs = synth.workload("burst_64_loguniform", scale=0.02) + [b"\xc3(", b"", "第3章 ok".encode()]
    data, offs = synth.batch(reqs)
    ref = oracle.Oracle(merges, vb, vo, 1).run(data, offs, threads=NCPU)
    ntok = int(ref["id_offsets"][-1])
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    pin_in = torch.from_numpy(data).pin_memory()
    pin_ids = torch.full((len(data) + 5,), -7, dtype=torch.int32).pin_memory()
    pin_io = torch.zeros(len(offs), dtype=torch.int64).pin_memory()
    cases = [("pinned", pin_ids.numpy(), pin_io.numpy()),
             ("pageable", np.full(len(data), -7, dtype=np.int32), np.zeros(len(offs), dtype=np.int64)),
             ("mixed", pin_ids.numpy(), np.zeros(len(offs), dtype=np.int64)),
             ("pinned, capacity below the bytes", pin_ids.numpy()[:ntok], pin_io.numpy())]
    for rep in range(2):
        for src_name, src in (("pinned input", pin_in.numpy()), ("pageable input", data)):
            for name, ids, io in cases:
                ids[:] = -7
                st = cuda.tt_encode_host(tok.h, src, offs, ids, io)
                assert st == cuda.TT_ERR_INVALID_UTF8, (src_name, name, st)
                assert np.array_equal(io, ref["id_offsets"]), (src_name, name)
                assert np.array_equal(ids[:ntok], ref["ids"]), (src_name, name)
    tok.close()


def test_two_streams_and_growing_batches(cuda, vocabs):
    merges, vb, vo = vocabs["c1"]
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    o1 = oracle.Oracle(merges, vb, vo, 1)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    # growing, then back to smaller buckets the streams already hold (each
    # (stream, bucket) keeps its workspace and replays its own graph)
    for size in (1000, 70000, 300000, 20000, 1000, 300000, 70000):
        jobs = []
        for si, s in enumerate(streams):
            reqs = [synth.transcript(100 * size + si * 7 + i, size // 4 + 1, 1) for i in range(4)]
            data, offs = synth.batch(reqs)
            with torch.cuda.stream(s):
                d = torch.from_numpy(data).cuda()
                o = torch.from_numpy(offs).cuda()
                ids, io = tok.encode(d, o, stream=s)
            jobs.append((data, offs, ids, io, s))
        for data, offs, ids, io, s in jobs:
            s.synchronize()
            io = io.cpu().numpy()
            ref = o1.run(data, offs)
            assert np.array_equal(io, ref["id_offsets"])
            assert np.array_equal(ids[:int(io[-1])].cpu().numpy(), ref["ids"])
    tok.close()


def test_capacity_bound_is_reported(cuda, vocabs):
    merges, vb, vo = vocabs["small1"]
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    data, offs = synth.batch([synth.transcript(9, 300000, 1)])
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    ids = torch.empty(len(data), dtype=torch.int32, device="cuda")
    io = torch.full((2,), 5, dtype=torch.int64, device="cuda")
    cuda.tt_encode_batch_bounded(tok.h, d, o, 1, 1000, ids, io)   # bound far below the batch
    status, _ = tok.status()
    assert status == cuda.TT_ERR_CAPACITY
    assert io.cpu().tolist() == [0, 0]
    ids, io = tok.encode(d, o)                                   # the handle keeps working
    torch.cuda.synchronize()
    assert tok.status()[0] == 0
    ref = oracle.Oracle(merges, vb, vo, 1).run(data, offs)
    assert np.array_equal(io.cpu().numpy(), ref["id_offsets"])
    tok.close()


@pytest.mark.parametrize("bound", [16, 4000, 9000])
def test_bound_below_the_batch_inside_its_bucket(cuda, vocabs, bound):
    """A stated bound below the true batch size, with the batch still inside
    the workspace's smallest size bucket (64 KiB): the kernels refuse it
    (TT_ERR_CAPACITY), zero the ID offsets and write no ID at all, so an IDs
    buffer sized to the bound is never overrun.  The spans entry point
    behaves the same, and the handle keeps working."""
    merges, vb, vo = vocabs["small1"]
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    data, offs = synth.batch([synth.transcript(5, 6000, 1), synth.transcript(6, 3000, 1)])
    assert bound < len(data) < 1 << 16
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    ids = torch.full((len(data) + 64,), -7, dtype=torch.int32, device="cuda")
    io = torch.full((3,), 5, dtype=torch.int64, device="cuda")
    cuda.tt_encode_batch_bounded(tok.h, d, o, 2, bound, ids, io)
    assert tok.status() == (cuda.TT_ERR_CAPACITY, -1)
    assert io.cpu().tolist() == [0, 0, 0]
    assert bool((ids == -7).all())
    spans = torch.full((len(data) + 64, 2), -7, dtype=torch.int32, device="cuda")
    cuda.tt_encode_batch_spans(tok.h, d, o, 2, bound, ids, io, spans)
    assert tok.status() == (cuda.TT_ERR_CAPACITY, -1)
    assert io.cpu().tolist() == [0, 0, 0]
    assert bool((ids == -7).all()) and bool((spans == -7).all())
    cuda.tt_encode_batch_bounded(tok.h, d, o, 2, len(data), ids, io)   # the true size: exact again
    torch.cuda.synchronize()
    assert tok.status() == (0, -1)
    ref = oracle.Oracle(merges, vb, vo, 1).run(data, offs)
    io = io.cpu().numpy()
    assert np.array_equal(io, ref["id_offsets"])
    assert np.array_equal(ids[:int(io[-1])].cpu().numpy(), ref["ids"])
    tok.close()


def test_lookback_wait_that_runs_out_yields_no_ids(cuda, vocabs):
    """A bounded device wait made to run out (one pre-tokenizer tile publishes
    nothing and the poll limit is small, a test setting): the batch reports
    TT_ERR_TIMEOUT, every request gets zero IDs and no ID is written -- never
    approximate IDs -- and the same handle is exact again once the setting is
    cleared.  Nothing faults or hangs: every wait gives up after its polls."""
    merges, vb, vo = vocabs["small1"]
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    reqs = [synth.transcript(40 + i, 20000, 1) for i in range(5)] + [b""]
    data, offs = synth.batch(reqs)
    assert len(data) > 20 * 4016                              # tiles after the withheld one
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    n = len(reqs)
    for withhold in (3, 0):
        cuda.tt_debug_lookback(tok.h, 2000, withhold)
        ids = torch.full((len(data),), -7, dtype=torch.int32, device="cuda")
        io = torch.full((n + 1,), 5, dtype=torch.int64, device="cuda")
        for _ in range(2):                                    # capture, then replay
            cuda.tt_encode_batch_bounded(tok.h, d, o, n, len(data), ids, io)
            assert tok.status() == (cuda.TT_ERR_TIMEOUT, -1)
            assert io.cpu().tolist() == [0] * (n + 1)
            assert bool((ids == -7).all())
        starts, po = tok.pretokenize(d, o)
        assert tok.status() == (cuda.TT_ERR_TIMEOUT, -1)
        assert po.cpu().tolist() == [0] * (n + 1)
    cuda.tt_debug_lookback(tok.h, 0, -1)
    got = run_gpu(cuda, tok, data, offs)
    ref = oracle.Oracle(merges, vb, vo, 1).run(data, offs)
    assert got["status"] == 0
    errs = compare_segmented(ref["piece_starts"], ref["piece_offsets"], got["piece_starts"], got["piece_offsets"],
                             "pieces")
    errs += compare_segmented(ref["ids"], ref["id_offsets"], got["ids"], got["id_offsets"], "ids")
    assert not errs, "\n".join(errs)
    with pytest.raises(cuda.TokTierError):
        cuda.tt_debug_lookback(tok.h, -1, -1)
    tok.close()


def test_decreasing_offsets_are_rejected_by_status(cuda, vocabs):
    merges, vb, vo = vocabs["small1"]
    tok = cuda.Tokenizer(merges, vb, vo, 1)
    data = np.frombuffer(b"hello world, this is fine", dtype=np.uint8).copy()
    offs = np.array([0, 12, 5, 25], dtype=np.int64)
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    tok.encode(d, o)
    status, _ = tok.status()
    assert status == cuda.TT_ERR_INVALID_ARG
    tok.close()
