"""Comparators for parity tests: element-by-element, bit-exact.

Both levels are compared, as the paper insists (TokTier §4.1: the ID level
can hide a boundary failure, so piece boundaries are compared too)."""
import numpy as np


def first_diff(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    n = min(len(a), len(b))
    d = np.nonzero(a[:n] != b[:n])[0]
    if len(d):
        return int(d[0])
    return n if len(a) != len(b) else -1


def compare_segmented(exp_vals, exp_offs, got_vals, got_offs, what="ids"):
    """Compare two per-request segmented arrays.  Returns a list of
    human-readable mismatch descriptions (empty = identical)."""
    exp_offs = np.asarray(exp_offs, dtype=np.int64)
    got_offs = np.asarray(got_offs, dtype=np.int64)
    out = []
    if len(exp_offs) != len(got_offs):
        return ["%s: %d vs %d requests" % (what, len(exp_offs) - 1, len(got_offs) - 1)]
    for r in range(len(exp_offs) - 1):
        e = np.asarray(exp_vals[exp_offs[r]:exp_offs[r + 1]])
        g = np.asarray(got_vals[got_offs[r]:got_offs[r + 1]])
        k = first_diff(e, g)
        if k >= 0:
            out.append("%s: request %d differs at %d (lengths %d vs %d; expected %s, got %s)" % (
                what, r, k, len(e), len(g), e[k:k + 4].tolist(), g[k:k + 4].tolist()))
            if len(out) >= 8:
                break
    return out
