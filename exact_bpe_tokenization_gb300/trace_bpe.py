"""Ticket trace of the warp BPE kernel: which work finishes when.

Builds the tracing variant of the library (libtoktier_trace.so, compiled with
-DTT_TRACE: every ticket of k_bpe_warp records the globaltimer at its start
and end, its kind, its pieces, the longest of them and the most merge rounds
the warp ran for one of them), encodes one batch of a named workload (after a
warm-up call, with L2 flushed before the traced call), and prints, per kind of
ticket, the tickets, pieces, rounds, durations and when the last of them
finished, against the kernel's span (first ticket start to last ticket end).

    python -m exact_bpe_tokenization_gb300.trace_bpe single_1m_mixed

Needs a CUDA device.  The product library is not touched.
"""
import ctypes
import json
import os
import sys

import numpy as np

KINDS = ["piece of 129..256 B", "49..128 B pieces", "short-piece chunk", "17..48 B pieces", "last queued misses"]


class TraceRec(ctypes.Structure):
    _fields_ = [("t0", ctypes.c_uint64), ("t1", ctypes.c_uint64), ("kind", ctypes.c_int32),
                ("pieces", ctypes.c_int32), ("max_len", ctypes.c_int32), ("rounds", ctypes.c_int32)]


def trace(name):
    import torch
    from . import binding, build, synth
    path = build.build(trace=True)
    binding.LIB_PATH = path                     # this process loads the tracing variant only
    L = binding.lib()
    L.tt_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int]
    L.tt_trace_read.restype = ctypes.c_int
    W = synth.WORKLOADS[name]
    merges, vb, vo = synth.make_vocab(*W["vocab"])
    data, offs = synth.batch(synth.workload(name))
    tok = binding.Tokenizer(merges, vb, vo, W["family"])
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    cap = 1 << 20
    buf = (TraceRec * cap)()
    tok.encode(d, o)                            # warm-up (captures the graph)
    L.tt_trace_read(buf, cap)
    torch.empty(64 << 20, dtype=torch.int32, device="cuda").fill_(1)   # L2 flushed before the traced call
    tok.encode(d, o)
    n = L.tt_trace_read(buf, cap)
    status = tok.status()[0]
    tok.close()
    recs = np.ctypeslib.as_array(buf)[:min(n, cap)]
    t_first = int(recs["t0"].min())
    span = (int(recs["t1"].max()) - t_first) / 1e3
    out = {"workload": name, "bytes": int(len(data)), "status": status, "tickets": int(len(recs)),
           "kernel_span_us": span, "kinds": []}
    for k, label in enumerate(KINDS):
        r = recs[recs["kind"] == k]
        if not len(r):
            continue
        dur = (r["t1"] - r["t0"]) / 1e3
        out["kinds"].append({
            "kind": label, "tickets": int(len(r)), "pieces": int(r["pieces"].sum()),
            "longest_piece": int(r["max_len"].max()), "rounds_mean": float(r["rounds"].mean()),
            "rounds_max": int(r["rounds"].max()), "ticket_us_mean": float(dur.mean()),
            "ticket_us_max": float(dur.max()), "last_end_us": (int(r["t1"].max()) - t_first) / 1e3})
    late = recs[np.argsort(recs["t1"])[-5:]]
    out["last_tickets"] = [{"kind": KINDS[int(x["kind"])], "max_len": int(x["max_len"]), "rounds": int(x["rounds"]),
                            "start_us": (int(x["t0"]) - t_first) / 1e3, "end_us": (int(x["t1"]) - t_first) / 1e3}
                           for x in late]
    return out


def main():
    name = sys.argv[1] if len(sys.argv) > 1 else "single_1m_mixed"
    print(json.dumps(trace(name), indent=1))


if __name__ == "__main__":
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    main()
