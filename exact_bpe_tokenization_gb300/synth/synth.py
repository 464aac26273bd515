"""Python side of the seeded input generators (ctypes over synth.c).

Everything here produces inputs: UTF-8 request batches and merge lists.  The
workload table mirrors the configurations the benchmark and the parity tests
use (tiny ASCII request; 1M-char mixed request; 64-request rebuild burst;
4.4M-char adversarial request; 256-request o200k-style batch; 64-request
deepseek-style batch of kana/CJK-mixed text).
"""
import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
REPO = os.path.dirname(os.path.dirname(HERE))
LIB_PATH = os.path.join(HERE, "libttsynth.so")
CACHE_DIR = os.path.join(REPO, "_build", "cache")

PROFILE_ASCII, PROFILE_MIXED, PROFILE_CAMEL_MARKS, PROFILE_KANA_HAN = 0, 1, 2, 3
# bumped whenever synth.c changes what it writes (part of every cache key)
GENERATOR_VERSION = 1

# pattern-family ids, as data (the same numbers the C ABI uses)
FAMILY_CL100K_STYLE, FAMILY_O200K_STYLE, FAMILY_DEEPSEEK_STYLE = 1, 2, 3

_lib = None
_lock = threading.Lock()


def elf_matches_host(path):
    """True if `path` is an ELF object built for this machine's architecture."""
    import platform
    import struct
    want = {"x86_64": 0x3E, "amd64": 0x3E, "aarch64": 0xB7, "arm64": 0xB7}.get(platform.machine().lower())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    return want is None or struct.unpack("<H", head[18:20])[0] == want


def build_lib(force=False):
    """Compile synth.c into libttsynth.so next to it (gcc, portable flags)."""
    src = os.path.join(HERE, "synth.c")
    if (not force and os.path.exists(LIB_PATH) and elf_matches_host(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(src)):
        return LIB_PATH
    tmp = LIB_PATH + ".%d.tmp" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=gnu11",
                           "-shared", "-fPIC", "-o", tmp, src, "-lm"])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _get():
    global _lib
    with _lock:
        if _lib is None:
            build_lib()
            lib = ctypes.CDLL(LIB_PATH)
            i64, u64, p = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
            lib.synth_transcript.argtypes = [u64, i64, ctypes.c_int, p, i64]
            lib.synth_transcript.restype = i64
            lib.synth_adversarial.argtypes = [u64, i64, p, i64]
            lib.synth_adversarial.restype = i64
            lib.synth_lengths_loguniform.argtypes = [u64, i64, i64, i64, p]
            lib.synth_lengths_lognormal.argtypes = [u64, i64, ctypes.c_double, ctypes.c_double, i64, p]
            lib.synth_train_bpe.argtypes = [p, i64, i64, ctypes.c_int, p]
            lib.synth_train_bpe.restype = i64
            _lib = lib
    return _lib


def _sized(call):
    n = call(None, 0)
    buf = np.empty(max(n, 1), dtype=np.uint8)
    m = call(buf.ctypes.data, n)
    assert m == n
    return buf[:n].tobytes()


def transcript(seed, n_chars, profile):
    """UTF-8 transcript text of exactly n_chars code points."""
    lib = _get()
    return _sized(lambda p, cap: lib.synth_transcript(seed, n_chars, profile, p, cap))


def adversarial(seed, n_chars):
    """Profile-1 text interleaved with pathological long-run blocks."""
    lib = _get()
    return _sized(lambda p, cap: lib.synth_adversarial(seed, n_chars, p, cap))


def lengths_loguniform(seed, n, lo, hi):
    out = np.empty(n, dtype=np.int64)
    _get().synth_lengths_loguniform(seed, n, lo, hi, out.ctypes.data)
    return out


def lengths_lognormal(seed, n, median, sigma, cap):
    out = np.empty(n, dtype=np.int64)
    _get().synth_lengths_lognormal(seed, n, float(median), float(sigma), cap, out.ctypes.data)
    return out


def train_merges(text, n_merges, case_split=False, han_split=False):
    """Greedy BPE merges (rank = row) trained on `text`; int32 [k, 2].
    case_split cuts training chunks at lower-to-upper changes; han_split
    makes kana / CJK ideograph runs chunks of their own."""
    buf = np.frombuffer(text, dtype=np.uint8)
    out = np.empty((n_merges, 2), dtype=np.int32)
    flags = int(bool(case_split)) | (int(bool(han_split)) << 1)
    k = _get().synth_train_bpe(buf.ctypes.data, len(buf), n_merges, flags, out.ctypes.data)
    return out[:k].copy()


def vocab_from_merges(merges):
    """Byte strings of ids 0..255 (single bytes) and 256+k (merge k's result)."""
    toks = [bytes([i]) for i in range(256)]
    for l, r in merges.tolist():
        toks.append(toks[l] + toks[r])
    offs = np.zeros(len(toks) + 1, dtype=np.int64)
    np.cumsum([len(t) for t in toks], out=offs[1:])
    return np.frombuffer(b"".join(toks), dtype=np.uint8).copy(), offs


def _cut_bytes(text, max_bytes):
    """Longest prefix of `text` of at most max_bytes that ends on a char boundary."""
    if len(text) <= max_bytes:
        return text
    i = max_bytes
    while i > 0 and (text[i] & 0xC0) == 0x80:
        i -= 1
    return text[:i]


def make_vocab(profile, corpus_bytes, n_merges, seed=0):
    """Train (or load from the build cache) a merge list on corpus_bytes of
    profile text from `seed`.  Returns (merges, vocab_bytes, vocab_offsets)."""
    key = "g%d_p%d_b%d_m%d_s%d" % (GENERATOR_VERSION, profile, corpus_bytes, n_merges, seed)
    path = os.path.join(CACHE_DIR, "merges_%s.npy" % key)
    merges = None
    if os.path.exists(path):
        try:
            merges = np.load(path)
        except Exception:
            merges = None
    if merges is None:
        # ~1.0-1.3 bytes per char for these profiles: ask for enough chars, then cut
        text = _cut_bytes(transcript(seed, corpus_bytes, profile), corpus_bytes)
        merges = train_merges(text, n_merges, case_split=(profile == PROFILE_CAMEL_MARKS),
                              han_split=(profile == PROFILE_KANA_HAN))
        os.makedirs(CACHE_DIR, exist_ok=True)
        tmp = path + ".%d.tmp.npy" % os.getpid()
        np.save(tmp, merges)
        os.replace(tmp, path)
    vb, vo = vocab_from_merges(merges)
    return merges, vb, vo


def batch(texts):
    """Concatenate request texts: (uint8 bytes, int64 byte_offsets[n+1])."""
    offs = np.zeros(len(texts) + 1, dtype=np.int64)
    np.cumsum([len(t) for t in texts], out=offs[1:])
    return np.frombuffer(b"".join(texts), dtype=np.uint8).copy(), offs


# The five workloads: (description, vocab spec, family, request builder)
MIB = 1 << 20
WORKLOADS = {
    "tiny_ascii_64k": dict(
        desc="1 request, 65,536 B ASCII transcript (seed 1); 4,096 merges on 1 MiB; cl100k-style",
        vocab=(PROFILE_ASCII, 1 * MIB, 4096), family=FAMILY_CL100K_STYLE),
    "single_1m_mixed": dict(
        desc="1 request of 1,000,000 chars mixed UTF-8 (seeds 1..32); 100,000 merges on 8 MiB; cl100k-style",
        vocab=(PROFILE_MIXED, 8 * MIB, 100000), family=FAMILY_CL100K_STYLE),
    "burst_64_loguniform": dict(
        desc="64 requests, log-uniform 10K..1M chars (seeds 1000+i); 100,000-merge vocab; cl100k-style",
        vocab=(PROFILE_MIXED, 8 * MIB, 100000), family=FAMILY_CL100K_STYLE),
    "adversarial_4_4m": dict(
        desc="1 request of 4.4M chars with 10K-digit, 50K-blank, CRLF, punctuation and a-a-a blocks (seed 7); "
             "100,000-merge vocab; cl100k-style",
        vocab=(PROFILE_MIXED, 8 * MIB, 100000), family=FAMILY_CL100K_STYLE),
    "o200k_256_lognormal": dict(
        desc="256 requests, lognormal chars (median 120K, sigma 1.0, cap 1M; seeds 1000+i); camelCase + marks; "
             "200,000 merges on 16 MiB; o200k-style",
        vocab=(PROFILE_CAMEL_MARKS, 16 * MIB, 200000), family=FAMILY_O200K_STYLE),
    "deepseek_64_loguniform": dict(
        desc="64 requests, log-uniform 10K..1M chars of kana/CJK-mixed text (seeds 2000+i); 100,000 merges on "
             "8 MiB; deepseek-style",
        vocab=(PROFILE_KANA_HAN, 8 * MIB, 100000), family=FAMILY_DEEPSEEK_STYLE),
}


def workload(name, seed=None, scale=1.0):
    """Request texts of a named workload.  `seed` picks the sample for the
    single-request workloads; `scale` < 1 shrinks every request length (used
    for oracle-sized parity cases; 1.0 is the full size)."""
    def n(x):
        return max(1, int(round(x * scale)))
    if name == "tiny_ascii_64k":
        return [transcript(1 if seed is None else seed, n(65536), PROFILE_ASCII)]
    if name == "single_1m_mixed":
        return [transcript(1 if seed is None else seed, n(1_000_000), PROFILE_MIXED)]
    if name == "burst_64_loguniform":
        lens = lengths_loguniform(2, 64, 10_000, 1_000_000)
        return [transcript(1000 + i, n(int(l)), PROFILE_MIXED) for i, l in enumerate(lens)]
    if name == "adversarial_4_4m":
        return [adversarial(7 if seed is None else seed, n(4_400_000))]
    if name == "o200k_256_lognormal":
        lens = lengths_lognormal(4, 256, 120_000, 1.0, 1_000_000)
        return [transcript(1000 + i, n(int(l)), PROFILE_CAMEL_MARKS) for i, l in enumerate(lens)]
    if name == "deepseek_64_loguniform":
        lens = lengths_loguniform(5, 64, 10_000, 1_000_000)
        return [transcript(2000 + i, n(int(l)), PROFILE_KANA_HAN) for i, l in enumerate(lens)]
    raise KeyError(name)


def digest(*arrays):
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()
