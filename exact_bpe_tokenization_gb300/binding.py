"""Thin ctypes binding of libtoktier.so (include/toktier.h).

Functions carry the C names and only marshal arguments: torch CUDA tensors
and numpy arrays are passed as raw pointers, streams as cudaStream_t.  Every
step of the tokenization runs in the library's CUDA kernels; there is no
Python or CPU fallback, and loading fails loudly if the library is missing.
"""
import ctypes
import os
import re
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtoktier.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "toktier.h")

TT_OK, TT_ERR_INVALID_ARG, TT_ERR_BAD_VOCAB, TT_ERR_BAD_FAMILY, TT_ERR_INVALID_UTF8, \
    TT_ERR_CAPACITY, TT_ERR_OOM, TT_ERR_CUDA, TT_ERR_TIMEOUT = range(9)
TT_FAMILY_CL100K_STYLE, TT_FAMILY_O200K_STYLE, TT_FAMILY_DEEPSEEK_STYLE = 1, 2, 3
TT_NOALLOC_MAX_BYTES, TT_NOALLOC_MAX_REQUESTS = 256 * 1024, 1024

_lib = None
_lock = threading.Lock()


class TokTierError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, status_string(status) if _lib else "", status))


def lib():
    """The loaded library with declared signatures (raises if not built)."""
    global _lib
    if _lib is not None:          # loaded once; no lock on the hot path
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libtoktier.so is not built (run __graft_entry__.build() or "
                                   "python -m exact_bpe_tokenization_gb300.build)")
            L = ctypes.CDLL(LIB_PATH)
            p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
            L.tt_create.argtypes = [p, i64, p, p, i64, i32, ctypes.POINTER(p)]
            L.tt_destroy.argtypes = [p]
            L.tt_encode_batch.argtypes = [p, p, p, i64, p, p, p]
            L.tt_encode_batch_bounded.argtypes = [p, p, p, i64, i64, p, p, p]
            L.tt_encode_batch_spans.argtypes = [p, p, p, i64, i64, p, p, p, p]
            L.tt_set_added_tokens.argtypes = [p, p, p, p, i64]
            L.tt_encode_batch_noalloc.argtypes = [p, p, p, i64, i64, p, p, p]
            L.tt_encode_host.argtypes = [p, p, p, i64, p, i64, p, p]
            L.tt_get_status.argtypes = [p, p, ctypes.POINTER(i64)]
            L.tt_pretokenize_batch.argtypes = [p, p, p, i64, p, p, p]
            L.tt_status_string.argtypes = [ctypes.c_int]
            L.tt_status_string.restype = ctypes.c_char_p
            L.tt_profile.argtypes = [p, ctypes.c_int]
            L.tt_profile_read.argtypes = [p, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(i64), ctypes.c_int]
            L.tt_launch_count.argtypes = [p]
            L.tt_launch_count.restype = i64
            L.tt_table_digest.restype = ctypes.c_char_p
            L.tt_debug_lookback.argtypes = [p, i32, i32]
            for name in ("tt_create", "tt_encode_batch", "tt_encode_batch_bounded", "tt_encode_batch_spans",
                         "tt_set_added_tokens",
                         "tt_encode_batch_noalloc",
                         "tt_encode_host",
                         "tt_get_status", "tt_pretokenize_batch", "tt_profile_read", "tt_debug_lookback"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def declared_symbols():
    """Names of the functions include/toktier.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(tt_\w+)\s*\(", text, flags=re.M)))


def _ptr(x):
    """Raw address of a torch tensor, numpy array or None."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return _np_addr(x)
    return int(x)


def _np_addr(a):
    """Address of a numpy array's data (a writable buffer through ctypes,
    a third of the cost of ndarray.ctypes; read-only or empty ones the slow way)."""
    try:
        return ctypes.addressof(ctypes.c_char.from_buffer(a))
    except (TypeError, ValueError):
        return a.ctypes.data


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _check(rc, what):
    if rc != TT_OK:
        raise TokTierError(rc, what)


def status_string(s):
    return lib().tt_status_string(int(s)).decode()


def tt_table_digest():
    return lib().tt_table_digest().decode()


def tt_create(merges, vocab_bytes, vocab_offsets, family):
    """Handle for (merges [k,2] int32, vocab bytes, vocab offsets [n+1] int64, family)."""
    m = np.ascontiguousarray(merges, dtype=np.int32).reshape(-1, 2)
    vb = np.ascontiguousarray(vocab_bytes, dtype=np.uint8)
    vo = np.ascontiguousarray(vocab_offsets, dtype=np.int64)
    h = ctypes.c_void_p()
    rc = lib().tt_create(m.ctypes.data if len(m) else None, len(m), vb.ctypes.data if len(vb) else None,
                         vo.ctypes.data, len(vo) - 1, int(family), ctypes.byref(h))
    _check(rc, "tt_create")
    return h


def tt_destroy(h):
    lib().tt_destroy(h)


def tt_encode_batch(h, d_utf8, d_byte_offsets, n_requests, d_out_ids, d_out_id_offsets, stream=None):
    _check(lib().tt_encode_batch(h, _ptr(d_utf8), _ptr(d_byte_offsets), int(n_requests), _ptr(d_out_ids),
                                 _ptr(d_out_id_offsets), _stream(stream)), "tt_encode_batch")


def tt_encode_batch_bounded(h, d_utf8, d_byte_offsets, n_requests, max_total_bytes, d_out_ids, d_out_id_offsets,
                            stream=None):
    _check(lib().tt_encode_batch_bounded(h, _ptr(d_utf8), _ptr(d_byte_offsets), int(n_requests),
                                         int(max_total_bytes), _ptr(d_out_ids), _ptr(d_out_id_offsets),
                                         _stream(stream)), "tt_encode_batch_bounded")


def tt_set_added_tokens(h, literals):
    """literals: {bytes: id} (host); an empty dict removes the set."""
    items = list(literals.items())
    data = np.frombuffer(b"".join(k for k, _ in items), dtype=np.uint8).copy()
    offs = np.zeros(len(items) + 1, dtype=np.int64)
    np.cumsum([len(k) for k, _ in items], out=offs[1:])
    ids = np.array([v for _, v in items], dtype=np.int32)
    _check(lib().tt_set_added_tokens(h, _ptr(data) if len(data) else None, _ptr(offs),
                                     _ptr(ids) if len(ids) else None, len(items)), "tt_set_added_tokens")


def tt_encode_batch_spans(h, d_utf8, d_byte_offsets, n_requests, max_total_bytes, d_out_ids, d_out_id_offsets,
                          d_out_spans, stream=None):
    _check(lib().tt_encode_batch_spans(h, _ptr(d_utf8), _ptr(d_byte_offsets), int(n_requests), int(max_total_bytes),
                                       _ptr(d_out_ids), _ptr(d_out_id_offsets), _ptr(d_out_spans),
                                       _stream(stream)), "tt_encode_batch_spans")


def tt_encode_batch_noalloc(h, d_utf8, d_byte_offsets, n_requests, max_total_bytes, d_out_ids, d_out_id_offsets,
                            stream=None):
    """As tt_encode_batch_bounded, with the library's fixed scratch: no device
    allocation, batches up to TT_NOALLOC_MAX_BYTES / TT_NOALLOC_MAX_REQUESTS."""
    _check(lib().tt_encode_batch_noalloc(h, _ptr(d_utf8), _ptr(d_byte_offsets), int(n_requests),
                                         int(max_total_bytes), _ptr(d_out_ids), _ptr(d_out_id_offsets),
                                         _stream(stream)), "tt_encode_batch_noalloc")


def tt_encode_host(h, utf8, byte_offsets, out_ids, out_id_offsets, stream=None):
    """Host buffers in and out (numpy).  Returns the batch's status code."""
    u = np.ascontiguousarray(utf8, dtype=np.uint8)
    o = np.ascontiguousarray(byte_offsets, dtype=np.int64)
    return lib().tt_encode_host(h, _np_addr(u) if len(u) else None, _np_addr(o), len(o) - 1,
                                _np_addr(out_ids), len(out_ids), _np_addr(out_id_offsets), _stream(stream))


def tt_get_status(h, stream=None):
    """(status code, lowest rejected request or -1); waits for the stream."""
    bad = ctypes.c_int64(-1)
    rc = lib().tt_get_status(h, _stream(stream), ctypes.byref(bad))
    return rc, bad.value


def tt_pretokenize_batch(h, d_utf8, d_byte_offsets, n_requests, d_piece_starts, d_piece_offsets, stream=None):
    _check(lib().tt_pretokenize_batch(h, _ptr(d_utf8), _ptr(d_byte_offsets), int(n_requests), _ptr(d_piece_starts),
                                      _ptr(d_piece_offsets), _stream(stream)), "tt_pretokenize_batch")


def tt_profile(h, enable):
    lib().tt_profile(h, int(bool(enable)))


def tt_profile_read(h, cap=16):
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_double * cap)()
    n = (ctypes.c_int64 * cap)()
    k = lib().tt_profile_read(h, names, ms, n, cap)
    return {names[i].decode(): (ms[i], n[i]) for i in range(k)}


def tt_launch_count(h):
    return lib().tt_launch_count(h)


def tt_debug_lookback(h, spin_limit, withhold_tile=-1):
    """Test setting: poll limit of the pre-tokenizer's look-back waits (0: the
    default) and a tile that publishes nothing (-1: none)."""
    _check(lib().tt_debug_lookback(h, int(spin_limit), int(withhold_tile)), "tt_debug_lookback")


class Tokenizer:
    """Convenience owner of a handle; device arrays are torch CUDA tensors."""

    def __init__(self, merges, vocab_bytes, vocab_offsets, family):
        self.h = tt_create(merges, vocab_bytes, vocab_offsets, family)
        self.family = family

    def close(self):
        if self.h is not None:
            tt_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def encode(self, d_utf8, d_offsets, max_total_bytes=None, stream=None, out_ids=None, out_offsets=None):
        """Encode a device batch; returns (ids, id_offsets) device tensors."""
        import torch
        n = d_offsets.numel() - 1
        if max_total_bytes is None:
            max_total_bytes = d_utf8.numel()
        if out_ids is None:
            out_ids = torch.empty(max(int(max_total_bytes), 1), dtype=torch.int32, device=d_utf8.device)
        if out_offsets is None:
            out_offsets = torch.empty(n + 1, dtype=torch.int64, device=d_utf8.device)
        tt_encode_batch_bounded(self.h, d_utf8, d_offsets, n, max_total_bytes, out_ids, out_offsets, stream)
        return out_ids, out_offsets

    def set_added_tokens(self, literals):
        """Reserve literal byte strings as single IDs ({bytes: id})."""
        tt_set_added_tokens(self.h, literals)

    def encode_spans(self, d_utf8, d_offsets, max_total_bytes=None, stream=None):
        """Encode a device batch with byte spans; returns (ids, id_offsets,
        spans) device tensors, spans int32 [capacity, 2] (start, end) from the
        batch start."""
        import torch
        n = d_offsets.numel() - 1
        if max_total_bytes is None:
            max_total_bytes = d_utf8.numel()
        cap = max(int(max_total_bytes), 1)
        out_ids = torch.empty(cap, dtype=torch.int32, device=d_utf8.device)
        out_offsets = torch.empty(n + 1, dtype=torch.int64, device=d_utf8.device)
        spans = torch.empty((cap, 2), dtype=torch.int32, device=d_utf8.device)
        tt_encode_batch_spans(self.h, d_utf8, d_offsets, n, max_total_bytes, out_ids, out_offsets, spans, stream)
        return out_ids, out_offsets, spans

    def pretokenize(self, d_utf8, d_offsets, stream=None):
        import torch
        n = d_offsets.numel() - 1
        starts = torch.empty(max(d_utf8.numel(), 1), dtype=torch.int64, device=d_utf8.device)
        offs = torch.empty(n + 1, dtype=torch.int64, device=d_utf8.device)
        tt_pretokenize_batch(self.h, d_utf8, d_offsets, n, starts, offs, stream)
        return starts, offs

    def encode_host(self, utf8, offsets, stream=None):
        """Host in, host out: (ids, id_offsets, status)."""
        offsets = np.asarray(offsets, dtype=np.int64)
        total = int(offsets[-1] - offsets[0]) if len(offsets) > 1 else 0
        ids = np.empty(max(total, 1), dtype=np.int32)
        io = np.empty(len(offsets), dtype=np.int64)
        st = tt_encode_host(self.h, np.frombuffer(utf8, dtype=np.uint8) if isinstance(utf8, (bytes, bytearray))
                            else utf8, offsets, ids, io, stream)
        return ids[:int(io[-1])], io, st

    def status(self, stream=None):
        return tt_get_status(self.h, stream)
