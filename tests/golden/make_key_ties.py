"""Writes key_ties.txt: rows whose sample needs the position tie-break.

The sample of a row is the f positions with the smallest (key, position),
key = Philox4x32-10 word (GARDEN page, Section IV-C: a uniform subset drawn
without altering the sampling distribution).  Two positions of a row with
equal keys occur about once per million rows, so no random test meets one.
This script searches node IDs v at hop 1 under a fixed seed for a row of a
given degree in which two positions share a key, and sets the fanout so that
exactly one of the two is taken (f = rank + 1, rank = the number of smaller
keys): the lower position must win.

The search uses its own vectorised Philox4x32-10, written from Salmon et al.,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11) and checked against the
published known-answer vectors in philox4x32_10_kat.txt before use.  The
tests check every line it writes with the oracle's own key function.

Run from the repository root:  python tests/golden/make_key_ties.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
MASK = np.uint64(0xFFFFFFFF)
SEED = 0x5EED0000CAFE1234
HOP = 1
# (degree, largest usable fanout, how many cases): an 8-lane group row
# (degree <= 256, f + 2 sqrt(f) + 4 <= 64), a warp row (degree <= 4096) and a
# block row (degree > 4096)
PLAN = [(256, 44, 1), (4000, 256, 2), (8000, 256, 2)]


def philox(c, k):
    """Philox4x32-10 on arrays: c = 4 counter words, k = 2 key words (uint64
    arrays holding 32-bit values)."""
    c0, c1, c2, c3 = c
    k0, k1 = k
    for _ in range(10):
        p0 = np.uint64(0xD2511F53) * c0
        p1 = np.uint64(0xCD9E8D57) * c2
        c0, c1, c2, c3 = (p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & MASK, (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & MASK
        k0 = (k0 + np.uint64(0x9E3779B9)) & MASK
        k1 = (k1 + np.uint64(0xBB67AE85)) & MASK
    return c0, c1, c2, c3


def check_kat():
    for line in open(os.path.join(HERE, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [np.uint64(int(x, 16)) for x in line.split()]
        out = philox([np.array([x]) for x in w[:4]], [np.array([x]) for x in w[4:6]])
        assert [int(o[0]) for o in out] == [int(x) for x in w[6:10]], "Philox does not match the known answers"


def row_keys(vs, deg):
    """keys[i, j] of node vs[i] at HOP, positions j < deg."""
    nq = (deg + 3) // 4
    q = np.tile(np.arange(nq, dtype=np.uint64), len(vs))
    v = np.repeat(np.asarray(vs, dtype=np.uint64), nq)
    z = np.zeros_like(q)
    k = (np.full_like(q, SEED & 0xFFFFFFFF), np.full_like(q, SEED >> 32))
    w = philox((q, v, z + np.uint64(HOP), z), k)
    keys = np.stack(w, axis=1).reshape(len(vs), nq * 4)
    return keys[:, :deg]


def search(deg, fmax, count, v0):
    found = []
    v = v0
    step = max(256, (1 << 22) // deg)
    while len(found) < count:
        vs = np.arange(v, v + step)
        keys = row_keys(vs, deg)
        srt = np.sort(keys, axis=1)
        dup = srt[:, 1:] == srt[:, :-1]
        for i in np.nonzero(dup.any(axis=1))[0]:
            r = int(np.nonzero(dup[i])[0][0])  # the smaller keys number r
            if r + 1 > fmax or r + 1 >= deg:
                continue
            x = srt[i, r]
            j1, j2 = [int(j) for j in np.nonzero(keys[i] == x)[0][:2]]
            found.append((int(vs[i]), deg, r + 1, j1, j2, int(x), r))
            if len(found) == count:
                break
        v += step
    return found, v


def main():
    check_kat()
    out = ["# Rows with two positions of equal key (written by make_key_ties.py; checked by",
           "# the oracle's key function in tests/test_oracle.py).  Seed %#x, hop %d." % (SEED, HOP),
           "# v degree fanout j_low j_high key rank (rank = keys below the tied key; the",
           "# fanout takes exactly one of the two, which must be j_low)"]
    v = 0
    for deg, fmax, count in PLAN:
        found, v = search(deg, fmax, count, v)
        for (vv, d, f, j1, j2, x, r) in found:
            out.append("%d %d %d %d %d %08x %d" % (vv, d, f, j1, j2, x, r))
            sys.stderr.write("v=%d deg=%d f=%d positions %d %d key %08x\n" % (vv, d, f, j1, j2, x))
    with open(os.path.join(HERE, "key_ties.txt"), "w") as fh:
        fh.write("\n".join(out) + "\n")


if __name__ == "__main__":
    main()
