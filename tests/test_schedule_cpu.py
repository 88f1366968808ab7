"""CPU check of the varlen tile-slot arithmetic the kernel uses.

Sequence n owns the chunk slots [base(n), base(n+1)) with
base(n) = floor((cu[n] + 63 n) / 64); a slot maps back to its sequence by a
binary search for the largest n with base(n) <= slot.  This test restates that
arithmetic in Python and checks on many random cu_seqlens (empty sequences,
exact multiples of 64, single tokens) that every chunk of every sequence gets
exactly one slot, that no slot is claimed twice, that the slot count
floor((T + 63 B) / 64) is enough, and that at most one slot per sequence stays
empty."""
import numpy as np
import pytest


def base(cu, n):
    return (int(cu[n]) + 63 * n) // 64


def slot_to_chunk(cu, B, slot):
    lo, hi = 0, B
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if base(cu, mid) <= slot:
            lo = mid
        else:
            hi = mid - 1
    if lo >= B:
        return None
    s, e = int(cu[lo]), int(cu[lo + 1])
    c = slot - base(cu, lo)
    r0 = s + 64 * c
    if c < 0 or r0 >= e:
        return None
    return lo, c, r0, min(64, e - r0)


@pytest.mark.parametrize("seed", range(40))
def test_varlen_slots_cover_every_chunk_once(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    kinds = rng.integers(0, 5, size=B)
    lens = np.where(kinds == 0, 0, np.where(kinds == 1, 64 * rng.integers(1, 4, size=B),
                    np.where(kinds == 2, 1, rng.integers(1, 300, size=B))))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    n_slots = (T + 63 * B) // 64
    seen = {}
    empty_per_seq = np.zeros(B, dtype=int)
    for slot in range(n_slots):
        r = slot_to_chunk(cu, B, slot)
        if r is None:
            continue
        n, c, r0, L = r
        assert (n, c) not in seen
        seen[(n, c)] = slot
        assert 0 < L <= 64 and r0 + L <= cu[n + 1]
    for n in range(B):
        want = (int(lens[n]) + 63) // 64
        got = sum(1 for (m, _) in seen if m == n)
        assert got == want, (n, lens[n])
        empty_per_seq[n] = (base(cu, n + 1) if n + 1 <= B else n_slots) - base(cu, n) - want
    assert np.all(empty_per_seq >= 0) and np.all(empty_per_seq <= 1)


def _fastdiv(d):
    l = 0
    while (1 << l) < d:
        l += 1
    shift = 31 + l
    return ((1 << shift) + d - 1) // d, shift


@pytest.mark.parametrize("d", [1, 2, 3, 5, 7, 31, 32, 33, 64, 100, 255, 256, 257, 4095, 65537,
                               (1 << 20) + 1, (1 << 24), (1 << 30) + 3, (1 << 31) - 1])
def test_multiply_shift_division_by_invariant_divisor(d):
    # The tile schedule divides numerators n < 2^31 by a fixed d with
    # m = ceil(2^(31+l) / d), l = ceil(log2 d): floor(n/d) = (n*m) >> (31+l).
    m, shift = _fastdiv(d)
    assert m < (1 << 33)
    rng = np.random.default_rng(d)
    ns = np.concatenate([rng.integers(0, 1 << 31, size=2000), np.arange(0, 300),
                         [(1 << 31) - 1, (1 << 31) - 2, d - 1, d, d + 1, 2 * d - 1, 2 * d]])
    for n in ns:
        n = int(n)
        if n >= (1 << 31):
            continue
        assert (n * m) >> shift == n // d, (n, d)
        assert (n * m) < (1 << 64)


# ---------------------------------------------------------------------------
# The kernel does not search the schedule for every tile: each role walks an
# arithmetic sequence of tiles u, u + S, u + 2S, ... (S = 2 * grid for the
# producer's pairs, 2 * grid * 3 for one warpgroup's) and steps (slot, head) and
# the slot's (sequence, chunk) forward incrementally.  The walk below restates
# that arithmetic; the test checks it against the direct definition on random
# fixed-length and varlen layouts, for several grid sizes.

def _tile_direct(P, u):
    H = P["H"]
    slot, h = u // H, u % H
    if slot >= P["n_slots"]:
        return (0, 0, h)
    if P["cu"] is None:
        b, c = slot // P["NT"], slot % P["NT"]
        return (b * P["T"] + 64 * c, min(P["T"] - 64 * c, 64), h)
    cu, B = P["cu"], P["B"]
    r = slot_to_chunk(cu, B, slot)
    if r is None:
        return (0, 0, h)
    _, _, r0, L = r
    return (r0, L, h)


class _Walk:
    def __init__(self, P, u):
        self.P = P
        H = P["H"]
        self.slot, self.h = u // H, u % H
        self.b = self.c = 0
        self.n, self.s, self.e, self.bn1 = P["B"], 0, 0, 0
        if P["cu"] is None:
            self.b, self.c = self.slot // P["NT"], self.slot % P["NT"]
        elif self.slot < P["n_slots"]:
            cu, B = P["cu"], P["B"]
            lo, hi = 0, B
            while lo < hi:
                mid = (lo + hi + 1) >> 1
                if base(cu, mid) <= self.slot:
                    lo = mid
                else:
                    hi = mid - 1
            self.n = lo
            if lo < B:
                self.s, self.e = int(cu[lo]), int(cu[lo + 1])
                self.bn1 = base(cu, lo + 1)

    def advance(self, ds, dh):
        P = self.P
        inc = ds
        self.h += dh
        if self.h >= P["H"]:
            self.h -= P["H"]
            inc += 1
        self.slot += inc
        if P["cu"] is None:
            self.c += inc
            if self.c >= P["NT"]:
                q = self.c // P["NT"]
                self.b += q
                self.c -= q * P["NT"]
        else:
            while self.n < P["B"] and self.bn1 <= self.slot:
                self.n += 1
                self.s = self.e
                if self.n < P["B"]:
                    assert self.n + 1 <= P["B"]          # never reads past cu[B]
                    self.e = int(P["cu"][self.n + 1])
                    self.bn1 = base(P["cu"], self.n + 1)

    def tile(self):
        P = self.P
        if self.slot >= P["n_slots"]:
            return (0, 0, self.h)
        if P["cu"] is None:
            return (self.b * P["T"] + 64 * self.c, min(P["T"] - 64 * self.c, 64), self.h)
        if self.n >= P["B"]:
            return (0, 0, self.h)
        s, e = self.s, min(self.e, P["T"])
        c = self.slot - (s + 63 * self.n) // 64
        r0 = s + 64 * c
        if c < 0 or r0 >= e:
            return (0, 0, self.h)
        return (r0, min(e - r0, 64), self.h)


@pytest.mark.parametrize("seed", range(24))
def test_incremental_tile_walk_matches_direct_schedule(seed):
    rng = np.random.default_rng(1000 + seed)
    H = int(rng.choice([1, 2, 3, 5, 8, 32, 64]))
    if seed % 2 == 0:
        B, T, cu = int(rng.integers(1, 5)), int(rng.integers(1, 700)), None
        NT = (T + 63) // 64
        n_slots = B * NT
    else:
        B = int(rng.integers(1, 30))
        kinds = rng.integers(0, 5, size=B)
        lens = np.where(kinds == 0, 0, np.where(kinds == 1, 64 * rng.integers(1, 4, size=B),
                        np.where(kinds == 2, 1, rng.integers(1, 300, size=B))))
        lens[0] = max(int(lens[0]), 1)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        T = int(cu[-1])
        NT = (T + 63) // 64
        n_slots = (T + 63 * B) // 64
    P = dict(H=H, B=B, T=T, cu=cu, NT=NT, n_slots=n_slots)
    n_pairs = (n_slots * H + 1) // 2
    for G in sorted({1, 3, 7, min(152, n_pairs), n_pairs}):
        for blk in range(G):
            n_local = (n_pairs - 1 - blk) // G + 1
            for role_stride, starts in ((2 * G, [(0, 0), (0, 1)]), (6 * G, [(wg, tt) for wg in range(3) for tt in range(2)])):
                ds, dh = role_stride // H, role_stride % H
                step = role_stride // (2 * G)
                for q0, tt in starts:
                    if q0 >= n_local:
                        continue
                    w = _Walk(P, 2 * (blk + q0 * G) + tt)
                    q = q0
                    while True:
                        assert w.tile() == _tile_direct(P, 2 * (blk + q * G) + tt), (H, G, blk, q, tt)
                        q += step
                        if q >= n_local:
                            break
                        w.advance(ds, dh)
