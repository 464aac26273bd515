"""Python wrapper of the CPU oracle (oracle.c).  TEST INFRASTRUCTURE: only
the tests, the smoke check and the benchmark's CPU-baseline / reference leg
use it.  It shares no code with the CUDA path; the frozen character-class
table is read here by this module's own parser.

See oracle.c for what is computed and which passages of "TokTier: Exact
Stateful CPU+GPU Tokenization for Agentic LLM Serving" each step follows.
"""
import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
REPO = os.path.dirname(HERE)
LIB_PATH = os.path.join(HERE, "liboracle.so")
CLASS_TABLE = os.path.join(REPO, "exact_bpe_tokenization_gb300", "data", "char_classes.txt")

FAMILY_CL100K_STYLE, FAMILY_O200K_STYLE, FAMILY_DEEPSEEK_STYLE = 1, 2, 3
ERR_UTF8 = 4

_lib = None
_cls = None
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
    src = os.path.join(HERE, "oracle.c")
    if (not force and os.path.exists(LIB_PATH) and elf_matches_host(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(src)):
        return LIB_PATH
    tmp = LIB_PATH + ".%d.tmp" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-shared", "-fPIC", "-pthread", "-o", tmp, src])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def load_lib(path):
    """Load an oracle shared library and declare its entry points."""
    lib = ctypes.CDLL(path)
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.oracle_create.argtypes = [p, ctypes.c_int, p, i64, p, p, i64, ctypes.POINTER(p)]
    lib.oracle_create.restype = ctypes.c_int
    lib.oracle_destroy.argtypes = [p]
    lib.oracle_run_batch.argtypes = [p, p, p, i64, ctypes.c_int, p, i64, p, p, i64, p, p]
    lib.oracle_run_batch.restype = ctypes.c_int
    lib.oracle_run_batch_spans.argtypes = [p, p, p, i64, ctypes.c_int, p, i64, p, p, p]
    lib.oracle_run_batch_spans.restype = ctypes.c_int
    lib.oracle_set_added_tokens.argtypes = [p, p, p, p, i64]
    lib.oracle_set_added_tokens.restype = ctypes.c_int
    lib.oracle_encode_bytes.argtypes = [p, p, i64, p]
    lib.oracle_encode_bytes.restype = i64
    lib.oracle_encode_bytes_plain.argtypes = [p, p, i64, p]
    lib.oracle_encode_bytes_plain.restype = i64
    return lib


def _get():
    global _lib
    with _lock:
        if _lib is None:
            build_lib()
            _lib = load_lib(LIB_PATH)
    return _lib


def load_class_table(path=CLASS_TABLE):
    """uint16 mask per code point (0x110000 entries) from the range file.
    Also checks the file's recorded body SHA-256."""
    masks = np.zeros(0x110000, dtype=np.uint16)
    body = []
    recorded = None
    with open(path, "r", encoding="ascii") as f:
        for line in f:
            if line.startswith("#"):
                if line.startswith("# body-sha256 "):
                    recorded = line.split()[2]
                continue
            body.append(line)
            a, b, m = line.split()
            masks[int(a, 16):int(b, 16) + 1] = int(m, 16)
    digest = hashlib.sha256("".join(body).encode("ascii")).hexdigest()
    if digest != recorded:
        raise ValueError("class table body does not match its recorded SHA-256")
    return masks


def class_table():
    global _cls
    with _lock:
        if _cls is None:
            _cls = load_class_table()
    return _cls


class Oracle:
    """The CPU oracle for one (merges, vocab, family)."""

    def __init__(self, merges, vocab_bytes, vocab_offsets, family, lib=None):
        lib = lib or _get()
        self._lib = lib
        self._cls = class_table()
        merges = np.ascontiguousarray(merges, dtype=np.int32).reshape(-1, 2)
        vb = np.ascontiguousarray(vocab_bytes, dtype=np.uint8)
        vo = np.ascontiguousarray(vocab_offsets, dtype=np.int64)
        h = ctypes.c_void_p()
        rc = lib.oracle_create(self._cls.ctypes.data, int(family), merges.ctypes.data, len(merges),
                               vb.ctypes.data if len(vb) else None, vo.ctypes.data, len(vo) - 1, ctypes.byref(h))
        if rc != 0:
            lib.oracle_destroy(h)
            raise ValueError("oracle_create failed: status %d" % rc)
        self._h = h
        self.family = family

    def set_added_tokens(self, literals):
        """literals: {bytes: id}; extracted leftmost-longest before the
        family tokenizes the rest (an empty dict clears them)."""
        items = list(literals.items())
        data = np.frombuffer(b"".join(k for k, _ in items), dtype=np.uint8).copy()
        offs = np.zeros(len(items) + 1, dtype=np.int64)
        np.cumsum([len(k) for k, _ in items], out=offs[1:])
        ids = np.array([v for _, v in items], dtype=np.int32)
        rc = self._lib.oracle_set_added_tokens(self._h, data.ctypes.data if len(data) else None, offs.ctypes.data,
                                               ids.ctypes.data if len(ids) else None, len(items))
        if rc != 0:
            raise ValueError("oracle_set_added_tokens failed: status %d" % rc)

    def close(self):
        if self._h:
            self._lib.oracle_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def run(self, data, offsets, threads=1, ids=True, pieces=True):
        """Tokenize a batch.  Returns a dict with ids/id_offsets (int32/int64),
        piece_starts (absolute byte offsets)/piece_offsets and status."""
        data = np.ascontiguousarray(np.frombuffer(data, dtype=np.uint8) if isinstance(data, (bytes, bytearray)) else data,
                                    dtype=np.uint8)
        offs = np.ascontiguousarray(offsets, dtype=np.int64)
        n = len(offs) - 1
        total = int(offs[-1] - offs[0]) if n > 0 else 0
        cap = max(total, 1)
        out = {"status": np.zeros(max(n, 1), dtype=np.int32)}
        oid = np.zeros(cap, dtype=np.int32) if ids else None
        oio = np.zeros(n + 1, dtype=np.int64) if ids else None
        ops = np.zeros(cap, dtype=np.int64) if pieces else None
        opo = np.zeros(n + 1, dtype=np.int64) if pieces else None
        dp = data.ctypes.data if len(data) else None
        rc = self._lib.oracle_run_batch(self._h, dp, offs.ctypes.data, n, int(threads),
                                     oid.ctypes.data if ids else None, cap, oio.ctypes.data if ids else None,
                                     ops.ctypes.data if pieces else None, cap,
                                     opo.ctypes.data if pieces else None, out["status"].ctypes.data)
        if rc != 0:
            raise RuntimeError("oracle_run_batch failed: status %d" % rc)
        out["status"] = out["status"][:n]
        if ids:
            out["ids"] = oid[:int(oio[-1])]
            out["id_offsets"] = oio
        if pieces:
            out["piece_starts"] = ops[:int(opo[-1])]
            out["piece_offsets"] = opo
        return out

    def run_spans(self, data, offsets, threads=1):
        """IDs with the source byte span of each: a dict with ids (int32),
        id_offsets (int64), spans (int64 [tokens, 2]: start, end as byte
        offsets from offsets[0]) and status."""
        data = np.ascontiguousarray(np.frombuffer(data, dtype=np.uint8) if isinstance(data, (bytes, bytearray)) else data,
                                    dtype=np.uint8)
        offs = np.ascontiguousarray(offsets, dtype=np.int64)
        n = len(offs) - 1
        total = int(offs[-1] - offs[0]) if n > 0 else 0
        cap = max(total, 1)
        status = np.zeros(max(n, 1), dtype=np.int32)
        ids = np.zeros(cap, dtype=np.int32)
        io = np.zeros(n + 1, dtype=np.int64)
        spans = np.zeros((cap, 2), dtype=np.int64)
        rc = self._lib.oracle_run_batch_spans(self._h, data.ctypes.data if len(data) else None, offs.ctypes.data, n,
                                              int(threads), ids.ctypes.data, cap, io.ctypes.data, spans.ctypes.data,
                                              status.ctypes.data)
        if rc != 0:
            raise RuntimeError("oracle_run_batch_spans failed: status %d" % rc)
        t = int(io[-1])
        return {"ids": ids[:t], "id_offsets": io, "spans": spans[:t], "status": status[:n]}

    def encode_bytes(self, b, plain=False):
        """E on one byte string (whole-piece shortcut unless plain=True)."""
        if len(b) == 0:
            return []
        buf = np.frombuffer(bytes(b), dtype=np.uint8)
        ids = np.zeros(len(buf), dtype=np.int32)
        f = self._lib.oracle_encode_bytes_plain if plain else self._lib.oracle_encode_bytes
        n = f(self._h, buf.ctypes.data, len(buf), ids.ctypes.data)
        return ids[:n].tolist()

    def pieces(self, text):
        """Pre-tokenizer pieces of one str (convenience for tests)."""
        b = text.encode("utf-8")
        r = self.run(b, np.array([0, len(b)], dtype=np.int64), ids=False)
        st = r["piece_starts"].tolist() + [len(b)]
        return [b[st[i]:st[i + 1]].decode("utf-8") for i in range(len(st) - 1)]

    def encode(self, text):
        b = text.encode("utf-8") if isinstance(text, str) else bytes(text)
        r = self.run(b, np.array([0, len(b)], dtype=np.int64), pieces=False)
        if r["status"][0] != 0:
            raise ValueError("invalid UTF-8")
        return r["ids"].tolist()


def byte_vocab():
    """The zero-merge vocabulary: ids 0..255 are the single bytes."""
    vb = np.arange(256, dtype=np.uint8)
    vo = np.arange(257, dtype=np.int64)
    return np.zeros((0, 2), dtype=np.int32), vb, vo


def pretokenizer(family, lib=None):
    """An oracle with the byte vocabulary, for pre-tokenizer-only checks."""
    m, vb, vo = byte_vocab()
    return Oracle(m, vb, vo, family, lib=lib)
