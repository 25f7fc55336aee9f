"""Host model of the persistent decode kernel's work partition (the index
arithmetic of `Partition` in paged_kv_kernels.cuh, restated in Python).

The kernel cuts the flattened (sequence, KV head, block) space into one share
per warp: R = ceil(total / warps) blocks, of which the warp streams a static
head (all of it under 48 blocks; else 85 % with 2 tail chunks, 80 % with 3 or
4) and leaves the tail chunks (their number set by R) for any warp to claim.  A unit that one segment holds whole is written
directly; every other unit leaves one partial per segment that cuts it, in
slot 0 (the segment's first flush) or 1, and the merge finds them by testing
the segments of the shares the unit overlaps.  This checks, over random
shapes, that every block is streamed exactly once and that the merge's
enumeration finds exactly the partials the decode side writes, also when a
row's candidates are dealt to its warps in interleaved batches of 32 (one
warp per row, or four).  The GPU parity tests check the kernels themselves.
"""
import numpy as np


class Part:
    def __init__(self, total, nwarps):
        self.total, self.nwarps = total, nwarps
        self.R = -(-total // nwarps) if total > 0 else 1
        self.nchunks = 0 if self.R < 48 else 2 if self.R < 100 else 3 if self.R < 200 else 4

    def cum(self, k):
        if self.nchunks == 2:
            return [0, 8, 10][k]
        if self.nchunks == 3:
            return [0, 7, 9, 10][k]
        return [0, 4, 7, 9, 10][k]

    def head(self, w):
        s = min(self.total, w * self.R)
        n = min(self.total, (w + 1) * self.R) - s
        return s, s + (n if self.nchunks == 0 else n * 17 // 20 if self.nchunks == 2 else n * 4 // 5)

    def chunk(self, k, w):
        hs, he = self.head(w)
        tail = min(self.total, (w + 1) * self.R) - he
        return he + tail * self.cum(k) // 10, he + tail * self.cum(k + 1) // 10

    def segment_of(self, p):
        w = p // self.R
        s, e = self.head(w)
        if p < e:
            return w, s, e
        for k in range(self.nchunks):
            s, e = self.chunk(k, w)
            if p < e:
                return self.nwarps + k * self.nwarps + w, s, e
        raise AssertionError("block outside every segment")


def _check(lens, hkv, nwarps):
    nblk = (np.asarray(lens, np.int64) + 15) // 16
    B = len(nblk)
    P = np.concatenate([[0], np.cumsum(nblk)])
    total = hkv * int(P[B])
    part = Part(total, nwarps)

    def locate(f):
        b = int(np.searchsorted(hkv * P, f, side="right") - 1)
        while nblk[b] == 0:
            b -= 1
        rem = f - hkv * int(P[b])
        return b, rem // int(nblk[b]), rem % int(nblk[b])

    segs = []
    if total:
        segs += [(w, *part.head(w)) for w in range(nwarps)]
        for q in range(nwarps * part.nchunks):
            k, w = divmod(q, nwarps)
            segs.append((nwarps + q, *part.chunk(k, w)))
    seen = np.zeros(total, np.int64)
    written, complete = {}, set()
    for sid, s, e in segs:
        first, unit_first_j = True, 0
        for p in range(s, e):
            seen[p] += 1
            b, kvh, j = locate(p)
            if p == s or j == 0:
                unit_first_j = j
            if j == nblk[b] - 1 or p == e - 1:
                u = b * hkv + kvh
                if unit_first_j == 0 and j == nblk[b] - 1:
                    assert u not in complete
                    complete.add(u)
                else:
                    key = (sid, 0 if first else 1)
                    assert key not in written
                    written[key] = u
                first = False
    assert (seen == 1).all()
    sps = 1 + part.nchunks
    found = set()
    for b in range(B):
        nb = int(nblk[b])
        for kvh in range(hkv):
            if nb == 0:
                continue
            u = b * hkv + kvh
            U = hkv * int(P[b]) + kvh * nb
            Uend = U + nb
            _, _, e0 = part.segment_of(U)
            if e0 >= Uend:
                assert u in complete
                continue
            assert u not in complete
            w0 = U // part.R
            ncand = ((Uend - 1) // part.R - w0 + 1) * sps
            for wpr in (1, 4):  # warp `sub` of the row takes candidates sub + wpr * (32 k + lane)
                dealt = []
                for sub in range(wpr):
                    k = 0
                    while sub + wpr * 32 * k < ncand:
                        dealt += [c for c in (sub + wpr * (32 * k + lane) for lane in range(32)) if c < ncand]
                        k += 1
                assert sorted(dealt) == list(range(ncand))
            mine = set()
            for c in range(ncand):
                w, k = w0 + c // sps, c % sps
                if k == 0:
                    (s, e), sid = part.head(w), w
                else:
                    (s, e), sid = part.chunk(k - 1, w), nwarps + (k - 1) * nwarps + w
                if e > s and e > U and s < Uend:
                    mine.add((sid, 1 if U > s else 0))
            assert mine == {key for key, v in written.items() if v == u}
            found |= mine
    assert found == set(written)
    return part.nchunks


def test_partition_streams_every_block_once_and_merge_finds_every_piece():
    rng = np.random.default_rng(0)
    tiers = set()
    for trial in range(600):
        B = int(rng.integers(1, 24))
        hkv = int(rng.integers(1, 9))
        nwarps = int(rng.choice([8, 12])) * int(rng.integers(1, 12))
        mb = int(rng.integers(1, 300))
        lens = rng.integers(0, mb * 16 + 1, size=B)
        if trial % 11 == 0:
            lens[:] = 0
        if trial % 7 == 0:
            lens[:] = rng.integers(0, 3, size=B)
        tiers.add(_check(lens, hkv, nwarps))
    assert tiers == {0, 2, 3, 4}  # every tail-chunk tier was exercised


def test_partition_edge_shapes():
    _check([0], 1, 8)                      # nothing to do
    _check([1], 1, 8)                      # one block, one warp busy
    _check([16 * 300], 8, 8)               # one long sequence over few warps (4 tail chunks)
    _check([17, 0, 33, 4096], 2, 96)       # empty sequence in the middle
    _check([4096] * 64, 8, 1216)           # the headline batch shape, uniform lengths
