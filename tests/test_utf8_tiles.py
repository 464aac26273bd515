"""The pre-pass's UTF-8 check, as a design: tiles of 4,016 bytes in windows
of 4,096, each thread checking the sequences that start among its 8 or 16
bytes -- claimed continuation bytes at its start passed over, an open
sequence completed past its last byte -- must reject exactly the requests
Python's strict decoder rejects (RFC 3629), however sequences, request starts
and the batch end fall across tiles and threads.  This replays the
decomposition on the CPU (the kernel itself is pinned by the GPU fuzz and
tile-edge tests); a planted fault (a two-byte lead that keeps the previous
lead's second-byte range) must be caught."""
import bisect
import random

import pytest

from exact_bpe_tokenization_gb300 import synth

WIN, HALO_L, HALO_R = 4096, 48, 32
TILE = WIN - HALO_L - HALO_R


def lead_len(b):
    return 2 if 0xC2 <= b <= 0xDF else 3 if 0xE0 <= b <= 0xEF else 4 if 0xF0 <= b <= 0xF4 else 1


def rejected(data, offs, per_thread, keep_range_bug=False):
    total = len(data)
    starts = set(o for o in offs[:-1] if o < total)
    bad = set()

    def req(x):
        return bisect.bisect_right(offs, x) - 1

    for t in range((total + TILE - 1) // TILE):
        ts = t * TILE
        te = min(ts + TILE, total)
        ws = ts - HALO_L

        def byte(i):
            return data[ws + i] if 0 <= ws + i < total else 0

        def rs(i):
            return (ws + i) in starts

        for tid in range(WIN // per_thread):
            ks = [k for k in range(per_thread) if ts <= ws + per_thread * tid + k < te]
            if not ks or all(byte(per_thread * tid + k) < 0x80 for k in ks):
                continue
            f, e = per_thread * tid + ks[0], per_thread * tid + ks[-1] + 1
            p, reach = f, 0
            for d in (1, 2, 3):
                q = f - d
                if ws + q < 0:
                    break
                if (byte(q) & 0xC0) == 0x80:
                    if rs(q):
                        break
                    continue
                reach = lead_len(byte(q)) - d
                break
            while reach > 0 and p < e and (byte(p) & 0xC0) == 0x80 and not rs(p):
                p, reach = p + 1, reach - 1
            need, lead, lo, top = 0, -1, 0x80, 0xBF
            while p < e or need > 0:
                b = byte(p)
                if need > 0:
                    if not rs(p) and ws + p < total and lo <= b <= top:
                        need, lo, top, p = need - 1, 0x80, 0xBF, p + 1
                        continue
                    bad.add(req(ws + lead))
                    need = 0
                    if p >= e:
                        break
                if b >= 0x80:
                    lead = p
                    if 0xC2 <= b <= 0xDF:
                        need = 1
                        if not keep_range_bug:
                            lo, top = 0x80, 0xBF
                    elif 0xE0 <= b <= 0xEF:
                        need, lo, top = 2, 0xA0 if b == 0xE0 else 0x80, 0x9F if b == 0xED else 0xBF
                    elif 0xF0 <= b <= 0xF4:
                        need, lo, top = 3, 0x90 if b == 0xF0 else 0x80, 0x8F if b == 0xF4 else 0xBF
                    else:
                        bad.add(req(ws + p))
                p += 1
    return bad


def strict(data, offs):
    out = set()
    for r in range(len(offs) - 1):
        try:
            bytes(data[offs[r]:offs[r + 1]]).decode("utf-8", "strict")
        except UnicodeDecodeError:
            out.add(r)
    return out


def soup(seed, n):
    rng = random.Random(seed)
    alpha = [0x41, 0x80, 0xBF, 0xC2, 0xC0, 0xDF, 0xE0, 0xA0, 0xED, 0x9F, 0xF0, 0x90, 0xF4, 0x8F, 0xF5, 0xE4, 0xB8,
             0x20, 0xC3, 0xA9, 0xF0, 0x9F, 0x99, 0x82]
    reqs = [bytes(rng.choice(alpha) for _ in range(rng.randint(0, 9))) for _ in range(n)]
    # valid text around invalid requests, and long requests that span tiles
    reqs += ["日本語のテキスト é à ü 🙂 abc".encode() * rng.randint(1, 400) for _ in range(40)]
    rng.shuffle(reqs)
    return reqs


@pytest.mark.parametrize("per_thread", [8, 16])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_tiled_check_rejects_what_the_strict_decoder_rejects(per_thread, seed):
    data, offs = synth.batch(soup(seed, 4000))
    data, offs = bytes(data), [int(o) for o in offs]
    assert rejected(data, offs, per_thread) == strict(data, offs)


def test_a_planted_range_fault_is_caught():
    found = False
    for seed in range(1, 4):
        data, offs = synth.batch(soup(seed, 4000))
        data, offs = bytes(data), [int(o) for o in offs]
        found |= rejected(data, offs, 16, keep_range_bug=True) != strict(data, offs)
    assert found
