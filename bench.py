"""Benchmark: exact full tokenization on one GB300.

Metric: full-tokenization input GB/s (batched) and p50 ms per 1M-char
request.  `value` is the batched half on the 64-request rebuild burst
(burst_64_loguniform, ~17.6 MB): every step is one call that encodes the
whole batch, inputs resident in HBM, L2 flushed between steps.  The latency
half is measured on 1,000,000-char mixed-UTF-8 requests under the
fresh-sample protocol (every timed request a different seeded sample, each
encoded once after warm-up on other seeds).

One JSON line on stdout (rank 0).  Keys beyond the base contract:
  p50_ms_per_1m_char_request / p99_...   the latency half (single_1m_mixed)
  latency_1m          its protocol, steady state and small requests
  per_request_alone   each burst request encoded alone: p50 / p99 ms
  o200k_batched       the 256-request o200k-style batch (~58 MB) as one call
  adversarial_4_4m    the 4.4M-char adversarial request: p50 / p99 ms
  tiny_ascii_64k      the 64 KB request on its own 4,096-merge vocabulary
  e2e                 the burst through tt_encode_host (pinned host buffers,
                      copies and the wait inside the timed region)
  roofline            the dominant kernel: (B + 4T + 16 per request) of the
                      batch / its measured launch time, against the measured
                      HBM copy bandwidth; `path` the same bytes over whole
                      calls, per workload
  cpu_baseline        the CPU oracle on the host cores: a thread pool over
                      the burst and the o200k-style batch, pinned to one NUMA
                      node, and one thread on a 1M-char request
  deepseek_batched    the burst's shape of kana/CJK-mixed text in the
                      deepseek-style family, as one call

--impl reference times the CPU oracle (a thread pool over the host cores)
on the same workload and metric.  Under torchrun (N > 1) every rank encodes
its own copy of the batch (replicas: requests are independent, so there is
no collective on the data path).
"""
import argparse
import glob
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

WORKLOAD = "burst_64_loguniform"          # the batched half of the metric
LATENCY_WORKLOAD = "single_1m_mixed"      # the p50-per-1M-char half
METRIC = "full-tokenization input GB/s (batched) and p50 ms per 1M-char request"
UNIT = "GB/s"
L2_FLUSH_BYTES = 256 << 20          # > 129 MB of L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
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
    """The 1M-char request seeds a rank times and warms up on: every rank its
    own, none shared between ranks or between warm-up and timed steps."""
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
    return [synth.workload(LATENCY_WORKLOAD, seed=s)[0] for s in seeds]


def vocab(name=WORKLOAD):
    from exact_bpe_tokenization_gb300 import synth
    W = synth.WORKLOADS[name]
    return synth.make_vocab(*W["vocab"]), W["family"]


FAMILY_NAMES = {1: "cl100k-style", 2: "o200k-style", 3: "deepseek-style"}


def line_config(data_bytes, n_requests, family, n_merges):
    """The `config` of both arms' lines: the workload and nothing about the
    implementation, so that the two lines describe the same work."""
    return {"workload": WORKLOAD, "requests_per_step": n_requests, "bytes_per_step": int(data_bytes),
            "pattern_family": FAMILY_NAMES[family], "merges": int(n_merges)}


def parse_cpulist(text):
    out = []
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            out.extend(range(int(a), int(b) + 1))
        else:
            out.append(int(part))
    return out


def numa_placement():
    """The host cores to run the CPU oracle on: those this process may use,
    restricted to the NUMA node that holds most of them (the pages pin their
    CPU comparators to NUMA nodes).  Returns (cores, description)."""
    allowed = set(os.sched_getaffinity(0))
    nodes = {}
    for path in glob.glob("/sys/devices/system/node/node[0-9]*"):
        try:
            with open(os.path.join(path, "cpulist")) as f:
                cpus = [c for c in parse_cpulist(f.read()) if c in allowed]
        except (OSError, ValueError):
            continue
        if cpus:
            nodes[int(path.rsplit("node", 1)[1])] = cpus
    if not nodes:
        return sorted(allowed), {"numa_node": None, "nodes_with_allowed_cores": [],
                                 "placement": "no NUMA information: all %d allowed cores" % len(allowed)}
    node = max(sorted(nodes), key=lambda k: len(nodes[k]))
    return nodes[node], {"numa_node": node, "nodes_with_allowed_cores": sorted(nodes),
                         "placement": "threads pinned to the %d allowed cores of NUMA node %d "
                                      "(sched_setaffinity); inputs generated after pinning (first touch)"
                                      % (len(nodes[node]), node)}


class pinned_to:
    """Run a block with this process's CPU affinity set to `cores`."""

    def __init__(self, cores):
        self.cores = set(cores)

    def __enter__(self):
        self.old = os.sched_getaffinity(0)
        os.sched_setaffinity(0, self.cores)
        return self

    def __exit__(self, *exc):
        os.sched_setaffinity(0, self.old)


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


def alg_bytes(n_bytes, n_tokens, n_requests):
    """Algorithmic bytes of a batch (per request: UTF-8 bytes in, 4 bytes
    per int32 ID out, 16 bytes of offsets), summed over its requests.  Every
    kernel launch of an encode processes the whole batch, so this is also
    the per-launch figure.  Intermediate traffic (classes, piece tables, hash
    gathers) is not credited."""
    return int(n_bytes) + 4 * int(n_tokens) + 16 * int(n_requests)


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


def oracle_gbs(o, reqs, threads):
    """One oracle run over a batch: (GB/s of input, seconds, tokens)."""
    from exact_bpe_tokenization_gb300 import synth
    data, offs = synth.batch(reqs)
    t = time.perf_counter()
    r = o.run(data, offs, threads=threads, pieces=False)
    dt = time.perf_counter() - t
    return len(data) / dt / 1e9, dt, int(r["id_offsets"][-1])


def cpu_baseline(merges_vocab, family, seeds):
    """The oracle as it stands on the host cores, pinned to one NUMA node: a
    thread pool (one request per thread at a time) over the burst and over
    the o200k-style batch, and one thread on a 1M-char request."""
    import oracle
    from exact_bpe_tokenization_gb300 import synth
    cores, numa = numa_placement()
    merges, vb, vo = merges_vocab
    out = {"unit": UNIT, "cores": len(cores), "kind": "oracle", "numa": numa,
           "host_cores_online": os.cpu_count()}
    with pinned_to(cores):
        o = oracle.Oracle(merges, vb, vo, family)
        gbs, dt, _ = oracle_gbs(o, synth.workload(WORKLOAD), len(cores))
        out.update(value=gbs, sample="the whole %s batch once (%d requests), %d threads" % (
            WORKLOAD, 64, len(cores)), seconds=dt)
        one = requests_for(seeds[:1])
        _, dt1, _ = oracle_gbs(o, one, 1)
        out["ms_per_1m_char_request_1thread"] = dt1 * 1e3
        o.close()
        (m4, v4, o4), f4 = vocab("o200k_256_lognormal")
        o = oracle.Oracle(m4, v4, o4, f4)
        g4, d4, _ = oracle_gbs(o, synth.workload("o200k_256_lognormal"), len(cores))
        out["o200k_batched"] = {"value": g4, "unit": UNIT, "seconds": d4, "threads": len(cores),
                                "sample": "the whole o200k_256_lognormal batch once (256 requests)"}
        o.close()
    return out


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from exact_bpe_tokenization_gb300 import synth
    cores, numa = numa_placement()
    (merges, vb, vo), family = vocab()
    with pinned_to(cores):
        reqs = synth.workload(WORKLOAD)
        data, offs = synth.batch(reqs)
        o = oracle.Oracle(merges, vb, vo, family)
        for _ in range(args.warmup):
            o.run(data, offs, threads=len(cores), pieces=False)
        times = []
        for _ in range(args.steps):
            t = time.perf_counter()
            o.run(data, offs, threads=len(cores), pieces=False)
            times.append(time.perf_counter() - t)
        lat = []
        for r in requests_for(range(1, 4)):          # the latency half: one thread per request
            d1, o1 = synth.batch([r])
            t = time.perf_counter()
            o.run(d1, o1, threads=1, pieces=False)
            lat.append((time.perf_counter() - t) * 1e3)
    total = sum(times)
    value = len(data) * args.steps / total / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "impl": "reference",
            "config": line_config(len(data), len(reqs), family, len(merges)),
            "protocol": "each step the whole batch through the CPU oracle, a thread pool over the host cores of one "
                        "NUMA node (one request per thread at a time)",
            "p50_ms_per_1m_char_request": float(np.percentile(lat, 50)),
            "p99_ms_per_1m_char_request": float(np.percentile(lat, 99)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": len(cores), "kind": "oracle", "numa": numa,
                             "sample": "%d steps of the whole %s batch (%d requests, %d bytes)" % (
                                 args.steps, WORKLOAD, len(reqs), len(data))},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def device_times(stream, flush, call, n, warm=1):
    """Device time in ms of each of n calls (after `warm` untimed ones), one
    call at a time between CUDA events on `stream`, L2 flushed before each."""
    import torch
    out = []
    for k in range(warm + n):
        flush.fill_(k)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        call()
        e.record(stream)
        e.synchronize()
        if k >= warm:
            out.append(s.elapsed_time(e))
    return out


def pct(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


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
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    # ---------------- the batched half: the whole burst as one call per step
    reqs = synth.workload(WORKLOAD)
    data, bo = synth.batch(reqs)
    n = len(reqs)
    d = torch.from_numpy(data).to(dev)
    o = torch.from_numpy(bo).to(dev)
    ids = torch.empty(len(data), dtype=torch.int32, device=dev)
    io = torch.empty(n + 1, dtype=torch.int64, device=dev)

    def encode():
        binding.tt_encode_batch_bounded(tok.h, d, o, n, len(data), ids, io, stream)

    for k in range(args.warmup):
        flush.fill_(k)
        encode()
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
            encode()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    launches = binding.tt_launch_count(tok.h) - launches0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    device_s, nbytes_all = combine_ranks(sum(step_ms) / 1e3, len(data) * args.steps, world, dev)
    status, _ = tok.status()
    assert status == 0, binding.status_string(status)
    tokens = int(io[-1].item())
    clocks = nclk.summary() if nclk.sm else clk.summary()

    # per-kernel times over the same steps: events around every kernel
    # (direct launches, one kernel at a time), L2 flushed before each step
    binding.tt_profile(tok.h, 1)
    for i in range(args.steps):
        flush.fill_(i)
        encode()
    prof = binding.tt_profile_read(tok.h)
    binding.tt_profile(tok.h, 0)

    # end to end through host buffers: the batch in pinned host memory before
    # each timed call, its IDs and offsets written back into pinned host memory
    pin_in = torch.empty(len(data), dtype=torch.uint8, pin_memory=True)
    pin_in.numpy()[:] = data
    pin_ids = torch.empty(len(data), dtype=torch.int32, pin_memory=True)
    pin_io = torch.empty(n + 1, dtype=torch.int64, pin_memory=True)
    in_np, ids_np, io_np = pin_in.numpy(), pin_ids.numpy(), pin_io.numpy()
    e2e_t = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        st = binding.tt_encode_host(tok.h, in_np, bo, ids_np, io_np, stream)
        if i >= args.warmup:
            e2e_t.append(time.perf_counter() - t)
        assert st == 0, binding.status_string(st)
    assert int(io_np[-1]) == tokens

    def per_request_alone(h, rq, dd, bb):
        """Every request of a batch encoded alone (n = 1): device ms, L2
        flushed before each call, after one untimed call."""
        out_i = torch.empty(int(max(bb[1:] - bb[:-1])) + 1, dtype=torch.int32, device=dev)
        out_o = torch.empty(2, dtype=torch.int64, device=dev)
        times = []
        for r in range(len(rq)):
            dr = dd[int(bb[r]):int(bb[r + 1])]
            orr = torch.tensor([0, int(bb[r + 1] - bb[r])], dtype=torch.int64, device=dev)
            times += device_times(stream, flush, lambda: binding.tt_encode_batch_bounded(
                h, dr, orr, 1, len(dr), out_i, out_o, stream), 1)
        return {"p50_ms": pct(times, 50), "p99_ms": pct(times, 99), "requests": len(times)}

    burst_alone = per_request_alone(tok.h, reqs, d, bo)

    # ---------------- the latency half: 1M-char requests, fresh sample
    seeds, warm_seeds = rank_seeds(rank, args.steps, args.warmup)
    host = [np.frombuffer(r, dtype=np.uint8) for r in requests_for(seeds)]
    warm = [np.frombuffer(r, dtype=np.uint8) for r in requests_for(warm_seeds)]
    cap = max(len(h) for h in host + warm)
    dev_in = [torch.from_numpy(h.copy()).to(dev) for h in host]
    offs1 = [torch.tensor([0, len(h)], dtype=torch.int64, device=dev) for h in host + warm]
    out1 = torch.empty(cap, dtype=torch.int32, device=dev)
    io1 = torch.zeros((len(host), 2), dtype=torch.int64, device=dev)
    for k, h in enumerate(warm):
        dw = torch.from_numpy(h.copy()).to(dev)
        flush.fill_(k)
        binding.tt_encode_batch_bounded(tok.h, dw, offs1[len(host) + k], 1, cap, out1, io1[0], stream)
    lat = []
    for i in range(len(host)):
        lat += device_times(stream, flush, lambda: binding.tt_encode_batch_bounded(
            tok.h, dev_in[i], offs1[i], 1, cap, out1, io1[i], stream), 1, warm=0)
    status, _ = tok.status()
    assert status == 0, binding.status_string(status)
    lat_tokens = io1[:, 1].cpu().numpy()
    lat_bytes = np.array([len(h) for h in host])
    binding.tt_profile(tok.h, 1)
    for i in range(len(host)):
        flush.fill_(i)
        binding.tt_encode_batch_bounded(tok.h, dev_in[i], offs1[i], 1, cap, out1, io1[i], stream)
    prof1 = binding.tt_profile_read(tok.h)
    binding.tt_profile(tok.h, 0)
    # steady state: one request replayed back to back, tables and input hot in L2
    ss = []
    for i in range(203):
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        binding.tt_encode_batch_bounded(tok.h, dev_in[0], offs1[0], 1, cap, out1, io1[0], stream)
        s1.record(stream)
        s1.synchronize()
        if i >= 3:
            ss.append(s0.elapsed_time(s1))
    # a 1,000-char request (the paper's Figure 10 starts at 1K chars)
    t1k = synth.transcript(5, 1000, synth.PROFILE_MIXED)
    d1k = torch.from_numpy(np.frombuffer(t1k, dtype=np.uint8).copy()).to(dev)
    o1k = torch.tensor([0, len(t1k)], dtype=torch.int64, device=dev)
    small = device_times(stream, flush, lambda: binding.tt_encode_batch_bounded(
        tok.h, d1k, o1k, 1, len(t1k), out1, io1[0], stream), 50)

    # ---------------- the other configurations
    def single(name, h, calls=20):
        """p50 / p99 device ms of one named single-request workload."""
        text = synth.workload(name)[0]
        ds = torch.from_numpy(np.frombuffer(text, dtype=np.uint8).copy()).to(dev)
        os_ = torch.tensor([0, len(text)], dtype=torch.int64, device=dev)
        oi = torch.empty(len(text), dtype=torch.int32, device=dev)
        oo = torch.empty(2, dtype=torch.int64, device=dev)
        t = device_times(stream, flush, lambda: binding.tt_encode_batch_bounded(
            h, ds, os_, 1, len(text), oi, oo, stream), calls, warm=2)
        st, _ = binding.tt_get_status(h, stream)
        nt = int(oo[1].item())
        return {"workload": name, "bytes": len(text), "tokens": nt, "p50_ms": pct(t, 50), "p99_ms": pct(t, 99),
                "calls": calls, "status": st, "path_alg_bytes": alg_bytes(len(text), nt, 1)}

    def batched(name, h, calls=20):
        """One named multi-request workload as one call: median of `calls`,
        L2 flushed before each; and every request encoded alone."""
        rq = synth.workload(name)
        db, bb = synth.batch(rq)
        dd = torch.from_numpy(db).to(dev)
        oo = torch.from_numpy(bb).to(dev)
        bi = torch.empty(len(db), dtype=torch.int32, device=dev)
        bio = torch.empty(len(bb), dtype=torch.int64, device=dev)
        t = device_times(stream, flush, lambda: binding.tt_encode_batch_bounded(
            h, dd, oo, len(rq), len(db), bi, bio, stream), calls, warm=3)
        st, _ = binding.tt_get_status(h, stream)
        nt = int(bio[-1].item())
        med = statistics.median(t)
        return {"workload": name, "requests": len(rq), "bytes": len(db), "tokens": nt,
                "value": len(db) / (med / 1e3) / 1e9, "unit": UNIT, "ms_median": med, "ms_p99": pct(t, 99),
                "calls": calls, "status": st, "per_request_alone": per_request_alone(h, rq, dd, bb),
                "path_alg_bytes": alg_bytes(len(db), nt, len(rq))}

    others = {}
    try:
        others["adversarial_4_4m"] = single("adversarial_4_4m", tok.h)
    except Exception as exc:  # reported, never fatal to the main line
        others["adversarial_4_4m"] = {"error": str(exc)}
    try:
        (m0, v0, o0), f0 = vocab("tiny_ascii_64k")
        t0k = binding.Tokenizer(m0, v0, o0, f0)
        others["tiny_ascii_64k"] = dict(single("tiny_ascii_64k", t0k.h, 50), merges=len(m0))
        t0k.close()
    except Exception as exc:
        others["tiny_ascii_64k"] = {"error": str(exc)}
    try:
        (m4, v4, o4), f4 = vocab("o200k_256_lognormal")
        t4 = binding.Tokenizer(m4, v4, o4, f4)
        others["o200k_batched"] = dict(batched("o200k_256_lognormal", t4.h), merges=len(m4),
                                       pattern_family=FAMILY_NAMES[f4])
        t4.close()
    except Exception as exc:
        others["o200k_batched"] = {"error": str(exc)}
    if not args.no_families:
        try:
            (md, vd, od), fd = vocab("deepseek_64_loguniform")
            td = binding.Tokenizer(md, vd, od, fd)
            others["deepseek_batched"] = dict(batched("deepseek_64_loguniform", td.h), merges=len(md),
                                              pattern_family=FAMILY_NAMES[fd])
            td.close()
        except Exception as exc:
            others["deepseek_batched"] = {"error": str(exc)}

    if rank != 0:
        tok.close()
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak_gbs()
    per_kernel = {k: v[0] / max(v[1], 1) for k, v in prof.items() if v[1]}
    dominant = max(per_kernel, key=per_kernel.get)
    dom_ms = per_kernel[dominant]
    alg = alg_bytes(len(data), tokens, n)
    med_ms = statistics.median(step_ms)
    lat_alg = float(np.mean(lat_bytes + 4 * lat_tokens + 16))
    path = {WORKLOAD: {"alg_bytes": alg, "ms": med_ms, "frac": alg / (peak * 1e9 * med_ms / 1e3),
                       "over": "median step"},
            LATENCY_WORKLOAD: {"alg_bytes": lat_alg, "ms": pct(lat, 50),
                               "frac": lat_alg / (peak * 1e9 * pct(lat, 50) / 1e3), "over": "p50 request"}}
    for key in ("o200k_batched", "adversarial_4_4m"):
        r = others.get(key, {})
        ms = r.get("ms_median", r.get("p50_ms"))
        if ms:
            path[r["workload"]] = {"alg_bytes": r["path_alg_bytes"], "ms": ms,
                                   "frac": r["path_alg_bytes"] / (peak * 1e9 * ms / 1e3),
                                   "over": "median call" if "ms_median" in r else "p50 request"}
    line = {
        "metric": METRIC, "value": nbytes_all / device_s / 1e9, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": device_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "config": line_config(len(data), n, family, len(merges)),
        "protocol": "each step one tt_encode_batch_bounded call over the whole batch (graph replay), inputs "
                    "resident in HBM; L2 flushed between steps by a 256 MiB write; %s" % (
                        "replicas: every rank encodes its own copy" if world > 1 else "1 GPU"),
        "tokens_per_step": tokens,
        "p50_ms_per_1m_char_request": pct(lat, 50),
        "p99_ms_per_1m_char_request": pct(lat, 99),
        "gpu_launches": launches,
        "wall_s_timed_loop": wall,
        "clocks": clocks,
        "e2e": {"value": len(data) * len(e2e_t) / sum(e2e_t) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": int(data.nbytes + bo.nbytes), "d2h_bytes_per_step": int(4 * tokens + bo.nbytes),
                "p50_ms": pct(np.array(e2e_t) * 1e3, 50), "api": "tt_encode_host (pinned host buffers)"},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": alg / (dom_ms / 1e3) / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": alg / (dom_ms / 1e3) / 1e9 / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic(dominant, WORKLOAD),
                     "alg_bytes_per_launch": alg, "launch_ms": dom_ms,
                     "definition": "per request: UTF-8 bytes in + 4 bytes per ID out + 16 bytes of offsets, "
                                   "summed over the batch (every launch processes the whole batch), over the "
                                   "dominant kernel's mean launch time",
                     "issue": issue_roofline(dominant, WORKLOAD, dom_ms, clocks.get("sm_mhz")),
                     "timing": "CUDA events around each kernel on its stream over the same steps, L2 flushed "
                               "before each step",
                     "path": path},
        "kernels_ms_per_launch": {k: round(v, 5) for k, v in per_kernel.items()},
        "per_request_alone": burst_alone,
        "latency_1m": {"workload": LATENCY_WORKLOAD, "requests": len(lat), "p50_ms": pct(lat, 50),
                       "p99_ms": pct(lat, 99), "mean_bytes": float(lat_bytes.mean()),
                       "mean_tokens": float(lat_tokens.mean()),
                       "protocol": "fresh sample: each timed request a different seeded sample, encoded once "
                                   "after warm-up on other seeds; L2 flushed before each",
                       "kernels_ms_per_launch": {k: round(v[0] / max(v[1], 1), 5) for k, v in prof1.items()
                                                 if v[1]},
                       "steady_state": {"p50_ms": pct(ss, 50), "p99_ms": pct(ss, 99),
                                        "protocol": "one request, 200 graph replays back to back, no L2 flush"},
                       "request_1k_chars": {"bytes": len(t1k), "p50_ms": pct(small, 50), "p99_ms": pct(small, 99)}},
    }
    line.update(others)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline((merges, vb, vo), family, seeds)
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
