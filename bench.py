"""Benchmark: exact full tokenization of 1M-char requests on one GB300.

Metric: full-tokenization input GB/s and p50 ms per 1M-char request
(fresh-sample protocol: every timed step encodes a different seeded
1,000,000-char mixed-UTF-8 transcript once, after warm-up on other seeds;
inputs are resident in HBM and L2 is flushed between steps).

One JSON line on stdout (rank 0).  Keys beyond the base contract:
  p50_ms / p99_ms   per-request device time over the timed steps
  e2e               the same requests through tt_encode_host (host buffers,
                    copies and the wait inside the timed region)
  roofline          the dominant kernel: algorithmic bytes / measured time
                    against the measured HBM copy bandwidth
  cpu_baseline      the CPU oracle on the host cores (a bounded sample)
  batched_gbs       the 64-request rebuild burst (~20 MB) as one call
  deepseek_batched_gbs  the same batch shape of kana/CJK-mixed text in the
                    deepseek-style family, as one call

--impl reference times the CPU oracle on the same workload and metric.
Under torchrun (N > 1) every rank encodes its own requests (replicas; the
requests are independent, so there is no collective on the data path).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "single_1m_mixed"
METRIC = "full-tokenization input GB/s (batched) and p50 ms per 1M-char request"
UNIT = "GB/s"
L2_FLUSH_BYTES = 256 << 20          # > 129 MB of L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-families", action="store_true", help="skip the deepseek-style batch line")
    ap.add_argument("--ncu-case", metavar="WORKLOAD", default=None,
                    help="encode one batch of WORKLOAD once and exit (a small case for an ncu capture)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seeds(rank, steps, warmup):
    """The request seeds a rank times and warms up on: every rank its own,
    none shared between ranks or between warm-up and timed steps."""
    return ([1 + rank * 10_000 + i for i in range(steps)],
            [100_001 + rank * 10_000 + i for i in range(warmup)])


def combine_ranks(device_s, nbytes, world, device):
    """Whole-job figures: the slowest rank's device time and all ranks' bytes."""
    if world <= 1:
        return device_s, float(nbytes)
    import torch
    import torch.distributed as dist
    t = torch.tensor([device_s, float(nbytes)], dtype=torch.float64, device=device)
    mx = t[:1].clone()
    sm = t[1:].clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[0])


def requests_for(seeds):
    from exact_bpe_tokenization_gb300 import synth
    return [synth.workload(WORKLOAD, seed=s)[0] for s in seeds]


def vocab():
    from exact_bpe_tokenization_gb300 import synth
    W = synth.WORKLOADS[WORKLOAD]
    return synth.make_vocab(*W["vocab"]), W["family"]


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = str(gpu_index)
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9 or p[0] != self.gpu:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (the driver's
    libnvidia-ml, ctypes, read-only queries) every millisecond from a thread:
    the timed loop is far shorter than nvidia-smi's sampling period.  The NVML
    device is the one whose UUID matches the CUDA device's."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, torch_device):
        self.dev = torch_device
        self.sm, self.reasons, self.max_mhz = [], set(), None
        self.ok = False
        self.stop = threading.Event()

    def _open(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        count = ctypes.c_uint()
        lib.nvmlDeviceGetCount_v2(ctypes.byref(count))
        want = str(getattr(torch.cuda.get_device_properties(self.dev), "uuid", "")).lower()
        chosen = None
        for i in range(count.value):
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(h)) != 0:
                continue
            buf = ctypes.create_string_buffer(96)
            lib.nvmlDeviceGetUUID(h, buf, 96)
            if want and buf.value.decode().lower().replace("gpu-", "") == want:
                chosen = h
        if chosen is None and count.value == 1:
            chosen = ctypes.c_void_p()
            lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(chosen))
        return (lib, chosen) if chosen is not None else None

    def _run(self, lib, h):
        import ctypes
        mhz, reasons = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:   # 1: SM clock
                self.sm.append(float(mhz.value))
            if lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(reasons)) == 0:
                for bit, name in self.REASONS.items():
                    if reasons.value & bit:
                        self.reasons.add(name)
            time.sleep(0.001)

    def __enter__(self):
        try:
            opened = self._open()
        except (OSError, AttributeError):
            opened = None
        if opened:
            import ctypes
            lib, h = opened
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.ok = True
            self.t = threading.Thread(target=self._run, args=(lib, h), daemon=True)
            self.t.start()
            while not self.sm and self.t.is_alive():        # first sample before the timed region
                time.sleep(0.0005)
        return self

    def __exit__(self, *exc):
        self.stop.set()
        if self.ok:
            self.t.join(timeout=2)

    def summary(self):
        return {"sm_mhz": statistics.median(self.sm) if self.sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.sm), "source": "nvml, 1 ms"}


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def piece_classes(binding, tok, d_in, d_off, ids, vocab_offsets, cap, dev):
    """Pieces of one request (from the pre-tokenizer test hook) split by the
    execution unit that encodes them, with their bytes and token counts (IDs
    are mapped back to pieces through the byte lengths of their tokens)."""
    import torch
    starts, po = tok.pretokenize(d_in, d_off)
    torch.cuda.synchronize(dev)
    n = int(po[-1].item())
    st = starts[:n].cpu().numpy() - int(d_off[0].item())
    total = int(d_off[-1].item() - d_off[0].item())
    lens = np.diff(np.append(st, total))
    tok_len = np.diff(np.asarray(vocab_offsets))[ids]
    ends = np.cumsum(tok_len)                     # byte end of every token
    piece_of_token = np.searchsorted(np.cumsum(lens), ends, side="left")
    tokens = np.bincount(piece_of_token, minlength=n)
    out = {}
    for name, lo, hi in (("small", 1, 16), ("mid", 17, 256), ("long", 257, 1 << 40)):
        sel = (lens >= lo) & (lens <= hi)
        out[name] = {"pieces": int(sel.sum()), "bytes": int(lens[sel].sum()), "tokens": int(tokens[sel].sum())}
    out["all"] = {"pieces": n, "bytes": total, "tokens": int(len(ids))}
    return out


def alg_bytes(kernel, c):
    """Algorithmic bytes of one launch: what a kernel must read and write at
    minimum for the pieces and tokens it handles (intermediate traffic such
    as hash-table gathers is not credited)."""
    a = c["all"]
    if kernel == "k_prepass":
        return a["bytes"]                                     # the batch bytes, read once
    if kernel == "k_pretok":
        return a["bytes"] + 4 * a["pieces"]                   # bytes in, int32 piece starts out
    cls = {"k_bpe_warp": ["small", "mid"], "k_bpe_long": ["long"]}.get(kernel)
    if cls:
        p = sum(c[k]["pieces"] for k in cls)
        return sum(c[k]["bytes"] + 4 * c[k]["tokens"] for k in cls) + 12 * p   # bytes + starts in, IDs + count out
    if kernel == "k_idscan":
        return 8 * ((a["pieces"] + 511) // 512) + 4          # chunk totals in, chunk offsets and the ID count out
    if kernel == "k_ids":
        return 8 * a["pieces"] + 8 * a["tokens"] + 16        # counts + starts in, IDs in and out, 2 offsets out
    return a["bytes"] + 4 * a["tokens"]


def recorded_traffic(kernel, workload, key="dram_bytes_per_launch"):
    """A per-launch counter (DRAM bytes; warp instructions) from the committed
    ncu summary, if it was taken on the current source of the kernel's file
    (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "roofline_traffic.txt")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    for r in rec.get("kernels", []):
        if r.get("kernel") != kernel or r.get("workload") != workload:
            continue
        src = os.path.join(ROOT, "exact_bpe_tokenization_gb300", "csrc", r.get("source", ""))
        try:
            sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        except OSError:
            return None
        return r.get(key) if sha == r.get("source_sha256") else None
    return None


SMS, SCHEDULERS_PER_SM = 152, 4


def issue_roofline(kernel, workload, launch_ms, sm_mhz):
    """The kernel's instruction issue against the GPU's issue peak: one warp
    instruction per cycle per scheduler, 4 schedulers per SM, at the SM clock
    sampled during the run."""
    inst = recorded_traffic(kernel, workload, "warp_inst_per_launch")
    if inst is None or not sm_mhz or not launch_ms:
        return None
    achieved = inst / (launch_ms / 1e3)
    peak = SMS * SCHEDULERS_PER_SM * sm_mhz * 1e6
    return {"achieved": achieved, "peak": peak, "unit": "warp-inst/s", "frac": achieved / peak,
            "warp_inst_per_launch": inst, "peak_from": "152 SMs x 4 schedulers x 1 warp-inst/cycle x SM clock"}


def cpu_baseline(merges_vocab, family, seeds):
    """The oracle as it stands on the host cores: one request per core."""
    import oracle
    merges, vb, vo = merges_vocab
    o = oracle.Oracle(merges, vb, vo, family)
    reqs = requests_for(seeds)
    from exact_bpe_tokenization_gb300 import synth
    data, offs = synth.batch(reqs)
    cores = os.cpu_count() or 1
    t = time.perf_counter()
    o.run(data, offs, threads=cores, pieces=False)
    dt = time.perf_counter() - t
    # single-thread latency of one request
    d1, o1 = synth.batch(reqs[:1])
    t = time.perf_counter()
    o.run(d1, o1, threads=1, pieces=False)
    one = time.perf_counter() - t
    return {"value": len(data) / dt / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d requests of 1,000,000 chars (seeds %d..%d), one request per core" % (
                len(reqs), seeds[0], seeds[-1]),
            "ms_per_request_1thread": one * 1e3}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    (merges, vb, vo), family = vocab()
    o = oracle.Oracle(merges, vb, vo, family)
    from exact_bpe_tokenization_gb300 import synth
    warm = requests_for(range(1001, 1001 + args.warmup))
    for r in warm:
        d, off = synth.batch([r])
        o.run(d, off, threads=1, pieces=False)
    reqs = requests_for(range(1, 1 + args.steps))
    times, nbytes = [], 0
    for r in reqs:
        d, off = synth.batch([r])
        t = time.perf_counter()
        o.run(d, off, threads=1, pieces=False)
        times.append(time.perf_counter() - t)
        nbytes += len(d)
    total = sum(times)
    value = nbytes / total / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "impl": "reference",
            "p50_ms": float(np.percentile(np.array(times) * 1e3, 50)),
            "p99_ms": float(np.percentile(np.array(times) * 1e3, 99)),
            "config": {"workload": WORKLOAD, "requests_per_step": 1, "chars_per_request": 1_000_000,
                       "protocol": "fresh sample: each step a different seeded request, CPU oracle, 1 thread"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "%d requests of 1,000,000 chars, one per step" % args.steps},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local if world > 1 else 0)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    from exact_bpe_tokenization_gb300 import binding, synth

    (merges, vb, vo), family = vocab()
    tok = binding.Tokenizer(merges, vb, vo, family)
    # each rank gets its own seeds (replicas of the same protocol)
    seeds, warm_seeds = rank_seeds(rank, args.steps, args.warmup)
    host = [np.frombuffer(r, dtype=np.uint8) for r in requests_for(seeds)]
    warm = [np.frombuffer(r, dtype=np.uint8) for r in requests_for(warm_seeds)]
    cap = max(len(h) for h in host + warm)
    dev_in = [torch.from_numpy(h.copy()).to(dev) for h in host]
    dev_warm = [torch.from_numpy(h.copy()).to(dev) for h in warm]
    offs = [torch.tensor([0, len(h)], dtype=torch.int64, device=dev) for h in host]
    offs_warm = [torch.tensor([0, len(h)], dtype=torch.int64, device=dev) for h in warm]
    out_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    out_off = torch.empty(2, dtype=torch.int64, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def encode(d, o):
        binding.tt_encode_batch_bounded(tok.h, d, o, 1, cap, out_ids, out_off, stream)

    for d, o in zip(dev_warm, offs_warm):
        encode(d, o)
        flush.fill_(1)
    torch.cuda.synchronize(dev)
    status, _ = tok.status()
    assert status == 0, binding.status_string(status)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = binding.tt_launch_count(tok.h)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk, NvmlClockSampler(dev) as nclk:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i)                       # evict the previous step's data from L2
            starts[i].record(stream)
            encode(dev_in[i], offs[i])
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    launches = binding.tt_launch_count(tok.h) - launches0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    nbytes = sum(len(h) for h in host)
    device_s = sum(step_ms) / 1e3
    device_s, nbytes_all = combine_ranks(device_s, nbytes, world, dev)
    status, _ = tok.status()
    assert status == 0, binding.status_string(status)
    # tokens of the last step (for the e2e byte counts)
    tokens = int(out_off[1].item())

    # per-kernel times: a second pass over the same steps with an event
    # around every kernel (direct launches), L2 flushed between steps
    binding.tt_profile(tok.h, 1)
    for i in range(args.steps):
        flush.fill_(i)
        encode(dev_in[i], offs[i])
    prof = binding.tt_profile_read(tok.h)
    binding.tt_profile(tok.h, 0)

    # steady state: one request encoded 200 times back to back, tables and
    # input hot in L2 (no flush), each replay timed on its own
    ss = []
    for i in range(203):
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        encode(dev_in[0], offs[0])
        s1.record(stream)
        s1.synchronize()
        if i >= 3:
            ss.append(s0.elapsed_time(s1))

    # small requests (the paper's Figure 10 quotes 1K chars): device time of a
    # 1,000-char request and of the 64 KB tiny configuration, 50 calls each
    # after one untimed call, L2 flushed before each
    small = {}
    for label, text in (("1k_chars", synth.transcript(5, 1000, synth.PROFILE_MIXED)),
                        ("tiny_ascii_64k", synth.workload("tiny_ascii_64k")[0])):
        dsm = torch.from_numpy(np.frombuffer(text, dtype=np.uint8).copy()).to(dev)
        osm = torch.tensor([0, len(text)], dtype=torch.int64, device=dev)
        tsm = []
        for k in range(51):
            flush.fill_(k)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            binding.tt_encode_batch_bounded(tok.h, dsm, osm, 1, len(text), out_ids, out_off, stream)
            s1.record(stream)
            s1.synchronize()
            if k:
                tsm.append(s0.elapsed_time(s1))
        small[label] = {"bytes": len(text), "p50_ms": float(np.percentile(tsm, 50)),
                        "p99_ms": float(np.percentile(tsm, 99)), "vocab": "the main line's 100,000 merges"}

    # end to end through host buffers (copies and the wait inside): each
    # step's request sits in pinned host memory before the timed call, and
    # its IDs come back into pinned host memory
    pin_in = []
    for h in host:
        t_in = torch.empty(len(h), dtype=torch.uint8, pin_memory=True)
        t_in.numpy()[:] = np.frombuffer(h, dtype=np.uint8)
        pin_in.append(t_in)
    pin_ids = torch.empty(max(len(h) for h in host) + 1, dtype=torch.int32, pin_memory=True)
    pin_io = torch.empty(2, dtype=torch.int64, pin_memory=True)
    ids_np, io_np = pin_ids.numpy(), pin_io.numpy()
    e2e_t, h2d, d2h, e2e_tokens = [], 0, 0, []
    for i, h in enumerate(host):
        o_np = np.array([0, len(h)], dtype=np.int64)
        t = time.perf_counter()
        st = binding.tt_encode_host(tok.h, pin_in[i].numpy(), o_np, ids_np, io_np, stream)
        e2e_t.append(time.perf_counter() - t)
        assert st == 0
        ids = ids_np[:int(io_np[-1])].copy()
        e2e_tokens.append(int(io_np[-1]))
        h2d += len(h) + o_np.nbytes
        d2h += ids.nbytes + io_np.nbytes

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak_gbs()
    per_kernel = {k: {"ms_per_launch": v[0] / max(v[1], 1), "launches": v[1]} for k, v in prof.items() if v[1]}
    dominant = max(per_kernel, key=lambda k: per_kernel[k]["ms_per_launch"])
    # algorithmic bytes of the dominant kernel for the last step's request
    last_ids = ids                                 # host IDs of the last e2e request (same input as step K)
    classes = piece_classes(binding, tok, dev_in[-1], offs[-1], last_ids, vo, cap, dev)
    flush.fill_(0)
    binding.tt_profile(tok.h, 1)
    encode(dev_in[-1], offs[-1])
    last_prof = binding.tt_profile_read(tok.h)
    binding.tt_profile(tok.h, 0)
    dom_ms = last_prof[dominant][0] / max(last_prof[dominant][1], 1)
    alg = alg_bytes(dominant, classes)
    achieved = alg / (dom_ms / 1e3) / 1e9
    mean_req_bytes = nbytes / args.steps
    p_ms = np.array(step_ms)
    p50_s = float(np.percentile(p_ms, 50)) / 1e3
    path_alg = mean_req_bytes + 4 * (sum(e2e_tokens) / len(e2e_tokens)) + 16
    line = {
        "metric": METRIC, "value": nbytes_all / device_s / 1e9, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": device_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "p50_ms": float(np.percentile(p_ms, 50)), "p99_ms": float(np.percentile(p_ms, 99)),
        "config": {"workload": WORKLOAD, "requests_per_step": 1, "chars_per_request": 1_000_000,
                   "bytes_per_request": mean_req_bytes, "pattern_family": "cl100k-style", "merges": len(merges),
                   "protocol": "fresh sample: each step a different seeded request, graph replay, "
                               "inputs resident in HBM",
                   "l2": "flushed between steps by a 256 MiB write", "parallelism": "replicas" if world > 1 else "1 GPU"},
        "gpu_launches": launches,
        "wall_s_timed_loop": wall,
        "clocks": nclk.summary() if nclk.sm else clk.summary(),
        "e2e": {"value": nbytes / sum(e2e_t) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d / args.steps,
                "d2h_bytes_per_step": d2h / args.steps, "p50_ms": float(np.percentile(np.array(e2e_t) * 1e3, 50)),
                "api": "tt_encode_host (pinned host buffers)"},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic(dominant, WORKLOAD),
                     "issue": issue_roofline(dominant, WORKLOAD, dom_ms,
                                             (nclk.summary() if nclk.sm else clk.summary()).get("sm_mhz")),
                     "alg_bytes_per_launch": alg, "launch_ms": dom_ms,
                     "path": {"alg_bytes_per_request": path_alg, "frac": path_alg / (peak * 1e9 * p50_s),
                              "definition": "UTF-8 in + 4 bytes per ID out + 16 bytes of offsets, over the p50 "
                                            "request time, against the same peak"},
                     "timing": "CUDA events around the kernel on its stream, L2 flushed before the launch",
                     "pieces": classes},
        "kernels_ms_per_launch": {k: round(v["ms_per_launch"], 5) for k, v in per_kernel.items()},
        "small_requests": small,
        "steady_state": {"p50_ms": float(np.percentile(ss, 50)), "p99_ms": float(np.percentile(ss, 99)),
                         "protocol": "one 1M-char request, 200 graph replays back to back, no L2 flush"},
    }
    def batched(name, h):
        """One named multi-request workload as one call: median of 50 calls,
        L2 flushed before each; and every request encoded alone (after one
        untimed call), for per-request p50 / p99."""
        reqs = synth.workload(name)
        data, bo = synth.batch(reqs)
        d = torch.from_numpy(data).to(dev)
        o = torch.from_numpy(bo).to(dev)
        bi = torch.empty(len(data), dtype=torch.int32, device=dev)
        bio = torch.empty(len(bo), dtype=torch.int64, device=dev)
        for _ in range(3):
            binding.tt_encode_batch_bounded(h, d, o, len(reqs), len(data), bi, bio, stream)
        alone = []                                 # (each size bucket has its own workspace and graph)
        for r in range(len(reqs)):
            dr = d[int(bo[r]):int(bo[r + 1])]
            orr = torch.tensor([0, int(bo[r + 1] - bo[r])], dtype=torch.int64, device=dev)
            for k in range(2):
                flush.fill_(k)
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record(stream)
                binding.tt_encode_batch_bounded(h, dr, orr, 1, len(dr), bi, bio, stream)
                e.record(stream)
                e.synchronize()
            alone.append(s.elapsed_time(e))
        ts = []
        for i in range(50):
            flush.fill_(i)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            binding.tt_encode_batch_bounded(h, d, o, len(reqs), len(data), bi, bio, stream)
            e.record(stream)
            e.synchronize()
            ts.append(s.elapsed_time(e))
        st, _ = binding.tt_get_status(h, stream)
        return {"workload": name, "bytes": len(data), "value": len(data) / (statistics.median(ts) / 1e3) / 1e9,
                "unit": UNIT, "ms_median": statistics.median(ts), "calls": len(ts), "status": st,
                "per_request_alone": {"p50_ms": float(np.percentile(alone, 50)),
                                      "p99_ms": float(np.percentile(alone, 99)), "requests": len(alone)}}

    # the batched burst (~20 MB, 64 requests) as one call, for the batched part of the metric
    try:
        line["batched_gbs"] = batched("burst_64_loguniform", tok.h)
    except Exception as exc:  # reported, never fatal to the main line
        line["batched_gbs"] = {"error": str(exc)}
    # the same shape of batch in the deepseek-style family (kana/CJK-mixed text)
    if not args.no_families:
        try:
            Wd = synth.WORKLOADS["deepseek_64_loguniform"]
            dtok = binding.Tokenizer(*synth.make_vocab(*Wd["vocab"]), Wd["family"])
            line["deepseek_batched_gbs"] = batched("deepseek_64_loguniform", dtok.h)
            dtok.close()
        except Exception as exc:  # reported, never fatal to the main line
            line["deepseek_batched_gbs"] = {"error": str(exc)}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline((merges, vb, vo), family, list(range(1, 25)))
    print(json.dumps(line), flush=True)
    tok.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_ncu_case(name):
    """One encode of a named workload, for a bounded ncu capture."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from exact_bpe_tokenization_gb300 import binding, synth
    W = synth.WORKLOADS[name]
    merges, vb, vo = synth.make_vocab(*W["vocab"])
    data, offs = synth.batch(synth.workload(name))
    tok = binding.Tokenizer(merges, vb, vo, W["family"])
    d = torch.from_numpy(data).cuda()
    o = torch.from_numpy(offs).cuda()
    ids, io = tok.encode(d, o)
    torch.cuda.synchronize()
    status, _ = tok.status()
    print(json.dumps({"ncu_case": name, "bytes": len(data), "tokens": int(io[-1].item()), "status": status}))
    tok.close()


def main():
    args = parse()
    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
