"""tt_encode_batch_noalloc: the entry point for callers that must not
allocate device memory once they are running (a fixed memory budget, an
allocator that forbids cudaMalloc/cudaFree after start-up, or a path where
an allocation would stall the device).  It runs the same kernels as the
regular entry point with a scratch array compiled into the library, so its
output must equal the CPU oracle's exactly -- and tt_encode_batch's --
call after call, even though every call reuses the same scratch.

This file is collected last on purpose, and it must pass alone in a fresh
process as well as after the other tests."""
import numpy as np
import pytest

import oracle
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
def test_no_alloc_matches_oracle_on_consecutive_calls(env, family, profile):
    binding = env
    merges, vb, vo = synth.make_vocab(profile, 1 << 20, 8000)
    tok = binding.Tokenizer(merges, vb, vo, family)
    ref = oracle.Oracle(merges, vb, vo, family)
    batches = [
        # a larger batch first, then a smaller one: the second call must not
        # see anything the first left in the shared scratch
        [synth.transcript(70 + i, 6000 + 1500 * i, profile) for i in range(12)] + [b"", b" " * 700 + b"x"],
        [synth.transcript(90 + i, 900 + 37 * i, profile) for i in range(40)] + ["don't 123456".encode()],
        # a rejected request (invalid UTF-8) between valid ones
        [synth.transcript(120 + i, 3000, profile) for i in range(6)] + [b"ok \xc3\x28 bad", b"fine 1234"],
        # empty requests only, then empty requests around valid ones
        [b""] * 9,
        [b"", b"", synth.transcript(130, 5000, profile), b"", synth.transcript(131, 700, profile), b""],
    ]
    for reqs in batches:
        data, offs = synth.batch(reqs)
        assert len(data) <= binding.TT_NOALLOC_MAX_BYTES and len(reqs) <= binding.TT_NOALLOC_MAX_REQUESTS
        want = ref.run(data, offs)
        d = torch.from_numpy(data).cuda()
        o = torch.from_numpy(offs).cuda()
        got_ids, got_io = no_alloc(binding, tok, d, o, len(reqs))
        assert np.array_equal(got_io, want["id_offsets"])
        assert np.array_equal(got_ids, want["ids"])
        bad = np.nonzero(want["status"])[0]
        assert tok.status() == ((binding.TT_ERR_INVALID_UTF8, int(bad[0])) if len(bad) else (0, -1))
        reg_ids, reg_io = regular(binding, tok, d, o, len(reqs))   # and the regular entry point agrees
        assert np.array_equal(reg_io, got_io) and np.array_equal(reg_ids, got_ids)
        tok.status()
    tok.close()


def test_no_alloc_true_size_beyond_the_stated_bound(env):
    """A caller that states a bound below the batch's true size gets
    TT_ERR_CAPACITY from the device, zeroed offsets and no IDs written: an
    IDs buffer sized to the bound is never overrun, even though the batch
    fits the fixed scratch."""
    binding = env
    merges, vb, vo = synth.make_vocab(synth.PROFILE_MIXED, 1 << 20, 8000)
    tok = binding.Tokenizer(merges, vb, vo, 1)
    data, offs = synth.batch([synth.transcript(140, 8000, 1)])
    assert 16 < len(data) <= binding.TT_NOALLOC_MAX_BYTES
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    ids = torch.full((len(data),), -7, dtype=torch.int32, device="cuda")
    io = torch.full((2,), 5, dtype=torch.int64, device="cuda")
    for _ in range(2):
        binding.tt_encode_batch_noalloc(tok.h, d, o, 1, 16, ids, io)
        assert tok.status() == (binding.TT_ERR_CAPACITY, -1)
        assert io.cpu().tolist() == [0, 0]
        assert bool((ids == -7).all())
    got_ids, got_io = no_alloc(binding, tok, d, o, 1)
    want = oracle.Oracle(merges, vb, vo, 1).run(data, offs)
    assert np.array_equal(got_io, want["id_offsets"]) and np.array_equal(got_ids, want["ids"])
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
    ref = oracle.Oracle(merges, vb, vo, 1)
    ref.set_added_tokens(lits)
    want = ref.run(data, offs)
    d, o = torch.from_numpy(data).cuda(), torch.from_numpy(offs).cuda()
    for _ in range(2):
        got = no_alloc(env, tok, d, o, len(reqs))
        assert np.array_equal(got[1], want["id_offsets"]) and np.array_equal(got[0], want["ids"])
    reg = regular(env, tok, d, o, len(reqs))
    assert np.array_equal(reg[1], want["id_offsets"]) and np.array_equal(reg[0], want["ids"])
    assert np.any(np.isin(want["ids"], [n + 1, n + 2, n + 3]))
    tok.close()
