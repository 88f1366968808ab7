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
