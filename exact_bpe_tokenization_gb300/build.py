"""Build libtoktier.so (the C ABI of include/toktier.h) in-tree.

Steps: turn the frozen character-class range file into a C include (checked
against its recorded SHA-256), compile every CUDA source for sm_103a in
parallel, link one shared library next to this file.  No cmake; nvcc only.
build(trace=True) builds the tracing variant instead (-DTT_TRACE, its own
objects and libtoktier_trace.so; see trace_bpe.py).
"""
import hashlib
import os
import platform
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
REPO = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(REPO, "_build", "toktier-" + platform.machine())
LIB = os.path.join(HERE, "libtoktier.so")
TRACE_LIB = os.path.join(HERE, "libtoktier_trace.so")
SOURCES = ["tt_api.cu", "tt_pretok.cu", "tt_bpe.cu", "tt_literals.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall"]


def nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def gen_class_include(out_dir):
    """C include with the class ranges: {first, last, mask} triples."""
    src = os.path.join(HERE, "data", "char_classes.txt")
    rows, body, recorded = [], [], None
    with open(src, encoding="ascii") as f:
        for line in f:
            if line.startswith("#"):
                if line.startswith("# body-sha256 "):
                    recorded = line.split()[2]
                continue
            body.append(line)
            a, b, m = line.split()
            rows.append((int(a, 16), int(b, 16), int(m, 16)))
    digest = hashlib.sha256("".join(body).encode("ascii")).hexdigest()
    if digest != recorded:
        raise RuntimeError("char_classes.txt does not match its recorded SHA-256")
    os.makedirs(out_dir, exist_ok=True)
    path = os.path.join(out_dir, "tt_char_classes.inc")
    text = ["// generated from data/char_classes.txt by build.py; do not edit",
            "static const uint32_t TT_CLASS_RANGES[][3] = {"]
    text += ["  {0x%X, 0x%X, 0x%X}," % r for r in rows]
    text += ["};", "static const int TT_CLASS_RANGE_COUNT = %d;" % len(rows),
             'static const char TT_CLASS_DIGEST[] = "%s";' % digest, ""]
    new = "\n".join(text)
    if not os.path.exists(path) or open(path).read() != new:
        with open(path, "w") as f:
            f.write(new)
    return path


def _stale(target, deps):
    if not os.path.exists(target) or not elf_matches_host(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def elf_matches_host(path):
    """True if `path` is an ELF object built for this machine's architecture."""
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


def build(force=False, verbose=False, trace=False):
    gen_dir = os.path.join(BUILD, "gen")
    inc = gen_class_include(gen_dir)
    obj_dir = BUILD + "-trace" if trace else BUILD
    lib_path = TRACE_LIB if trace else LIB
    extra = ["-DTT_TRACE"] if trace else []
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers += [inc, os.path.join(REPO, "include", "toktier.h")]
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(obj_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc()] + ARCH + NVCC_FLAGS + extra + ["-I", gen_dir, "-I", CSRC, "-c", s, "-o", o])
    os.makedirs(obj_dir, exist_ok=True)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s" % (" ".join(cmd), r.stdout + r.stderr))
        return r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        for out in ex.map(run, jobs):
            if verbose and out.strip():
                print(out)
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".%d.tmp" % os.getpid()
        run([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
