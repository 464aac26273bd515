"""tt_encode_batch_noalloc: the entry point for callers that must not
allocate device memory once they are running (a fixed memory budget, an
allocator that forbids cudaMalloc/cudaFree after start-up, or a path where
an allocation would stall the device).  It runs the same kernels as the
regular entry point with a scratch array compiled into the library, so its
output must equal tt_encode_batch's exactly, call after call, even though
every call reuses the same scratch.

This file is collected last on purpose, and it must pass alone in a fresh
process as well as after the other tests."""
import numpy as np
import pytest

from exact_bpe_tokenization_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from exact_bpe_tokenization_gb300 import binding
    return binding


def regular(binding, tok, d, o, n):
    ids = torch.empty(max(d.numel(), 1), dtype=torch.int32, device="cuda")
    io = torch.empty(n + 1, dtype=torch.int64, device="cuda")
    binding.tt_encode_batch(tok.h, d, o, n, ids, io)
    torch.cuda.synchronize()
    io = io.cpu().numpy()
    return ids[:int(io[-1])].cpu().numpy(), io


def no_alloc(binding, tok, d, o, n):
    ids = torch.full((max(d.numel(), 1),), -7, dtype=torch.int32, device="cuda")
    io = torch.full((n + 1,), -7, dtype=torch.int64, device="cuda")
    binding.tt_encode_batch_noalloc(tok.h, d, o, n, d.numel(), ids, io)
    torch.cuda.synchronize()
    io = io.cpu().numpy()
    return ids[:int(io[-1])].cpu().numpy(), io


@pytest.mark.parametrize("family,profile", [(1, synth.PROFILE_MIXED), (2, synth.PROFILE_CAMEL_MARKS)])
def test_no_alloc_matches_regular_entry_point_on_consecutive_calls(env, family, profile):
    binding = env
    merges, vb, vo = synth.make_vocab(profile, 1 << 20, 8000)
    tok = binding.Tokenizer(merges, vb, vo, family)
    batches = [
        # a larger batch first, then a smaller one: the second call must not
        # see anything the first left in the shared scratch
        [synth.transcript(70 + i, 6000 + 1500 * i, profile) for i in range(12)] + [b"", b" " * 700 + b"x"],
        [synth.transcript(90 + i, 900 + 37 * i, profile) for i in range(40)] + ["don't 123456".encode()],
    ]
    for reqs in batches:
        data, offs = synth.batch(reqs)
        assert len(data) <= binding.TT_NOALLOC_MAX_BYTES and len(reqs) <= binding.TT_NOALLOC_MAX_REQUESTS
        d = torch.from_numpy(data).cuda()
        o = torch.from_numpy(offs).cuda()
        want_ids, want_io = regular(binding, tok, d, o, len(reqs))
        got_ids, got_io = no_alloc(binding, tok, d, o, len(reqs))
        assert np.array_equal(got_io, want_io)
        assert np.array_equal(got_ids, want_ids)
        assert tok.status() == (0, -1)
    tok.close()


def test_no_alloc_rejects_batches_beyond_its_limits(env):
    binding = env
    merges, vb, vo = synth.make_vocab(synth.PROFILE_MIXED, 1 << 20, 8000)
    tok = binding.Tokenizer(merges, vb, vo, 1)
    d = torch.zeros(16, dtype=torch.uint8, device="cuda")
    o = torch.tensor([0, 16], dtype=torch.int64, device="cuda")
    ids = torch.empty(16, dtype=torch.int32, device="cuda")
    io = torch.empty(2, dtype=torch.int64, device="cuda")
    with pytest.raises(binding.TokTierError) as e:
        binding.tt_encode_batch_noalloc(tok.h, d, o, 1, binding.TT_NOALLOC_MAX_BYTES + 1, ids, io)
    assert e.value.status == binding.TT_ERR_CAPACITY
    with pytest.raises(binding.TokTierError) as e:
        binding.tt_encode_batch_noalloc(tok.h, d, o, binding.TT_NOALLOC_MAX_REQUESTS + 1, 16, ids, io)
    assert e.value.status == binding.TT_ERR_CAPACITY
    tok.close()


def test_no_alloc_with_added_tokens(env):
    """Literal extraction runs on the fixed scratch too, equal to the
    regular entry point's output."""
    merges, vb, vo = synth.make_vocab(synth.PROFILE_MIXED, 8 << 20, 100000)
    n = len(vo) - 1
    lits = {b"<|endoftext|>": n + 1, b"<|im_start|>": n + 2, b"<|im": n + 3}
    text = synth.workload("single_1m_mixed", seed=11, scale=0.05)[0]
    keys = list(lits)
    reqs, at = [], 0
    for i in range(40):                        # 40 requests with literals at varied places
        c = text[at:at + 700]
        k = keys[i % 3]
        reqs.append(c[:i * 13 % 300] + k + c[i * 13 % 300:] if i % 4 else k + c)
        at += 700
    data, offs = synth.batch(reqs)
    assert len(data) <= env.TT_NOALLOC_MAX_BYTES
    tok = env.Tokenizer(merges, vb, vo, 1)
    tok.set_added_tokens(lits)
    d, o = torch.from_numpy(data).cuda(), torch.from_numpy(offs).cuda()
    want = regular(env, tok, d, o, len(reqs))
    for _ in range(2):
        got = no_alloc(env, tok, d, o, len(reqs))
        assert np.array_equal(got[1], want[1]) and np.array_equal(got[0], want[0])
    assert np.any(np.isin(want[0], [n + 1, n + 2, n + 3]))
    tok.close()
