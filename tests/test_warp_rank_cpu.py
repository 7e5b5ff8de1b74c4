"""The one-warp segment build's ranking method, checked on CPU.

For batches of at most 32 tokens the build gives each lane (token) its slot in
the stable counting sort on key = adapter id (L for -1, bad or disabled ids, L + 1
for lanes past M): the key bits are taken from the top, one warp ballot per bit;
a lane adds the lanes that share its higher bits and have a 0 where it has a 1,
then keeps only the lanes with its own bit.  What is left are the lanes with its
key, and the slot is the smaller keys plus the equal keys on lower lanes.  The
first lane of each key writes the segment, indexed by the first lanes on lower
slots.  This test replays those steps with explicit 32-bit ballots and compares
the result with a stable sort (the oracle's definition of the segment table).
The kernels themselves are compared with the oracle bit for bit by the GPU tests.
"""
import random

FULL = 0xFFFFFFFF


def popc(x):
    return bin(x & FULL).count("1")


def ballot(pred):
    return sum(1 << lane for lane, p in enumerate(pred) if p)


def rank_build(ids, M, L):
    keys = [(ids[t] if 0 <= ids[t] < L else L) if t < M else L + 1 for t in range(32)]
    same, less = [FULL] * 32, [0] * 32
    for b in range((L + 1).bit_length() - 1, -1, -1):
        ones = ballot((k >> b) & 1 for k in keys)
        for t in range(32):
            if (keys[t] >> b) & 1:
                less[t] += popc(same[t] & ~ones)
                same[t] &= ones
            else:
                same[t] &= ~ones & FULL
    below = [(1 << t) - 1 for t in range(32)]
    rank = [less[t] + popc(same[t] & below[t]) for t in range(32)]
    first = [(same[t] & below[t]) == 0 for t in range(32)]
    first_slots = 0
    for t in range(32):
        if first[t]:
            first_slots |= 1 << rank[t]
    perm = [None] * M
    segments = {}
    for t in range(32):
        if t < M:
            perm[rank[t]] = t
        if first[t] and keys[t] < L:
            segments[popc(first_slots & ((1 << rank[t]) - 1))] = (keys[t], rank[t], popc(same[t]))
    return perm, [segments[i] for i in range(len(segments))]


def stable_sort_build(ids, M, L):
    keys = [ids[t] if 0 <= ids[t] < L else L for t in range(M)]
    perm = sorted(range(M), key=lambda t: (keys[t], t))
    segments, start = [], 0
    for a in range(L):
        n = keys.count(a)
        if n:
            segments.append((a, start, n))
            start += n
    return perm, segments


def test_matches_the_stable_counting_sort():
    rng = random.Random(5)
    for _ in range(4000):
        M = rng.randint(0, 32)
        L = rng.choice([1, 2, 3, 5, 16, 20, 31, 32, 33, 64, 100, 2047, 2048])
        pool = [-1, -2, L, L + 7] + list(range(min(L, 40))) * 3
        ids = [rng.choice(pool) for _ in range(M)]
        assert rank_build(ids, M, L) == stable_sort_build(ids, M, L), (M, L, ids)


def test_worked_cases():
    # equal ids keep token order; -1 and out-of-range ids are left out of the segments
    assert rank_build([2, 0, 2, -1, 0, 5], 6, 3) == ([1, 4, 0, 2, 3, 5], [(0, 0, 2), (2, 2, 2)])
    assert rank_build([], 0, 4) == ([], [])
    assert rank_build([-1] * 32, 32, 1) == (list(range(32)), [])
    assert rank_build([0] * 32, 32, 1) == (list(range(32)), [(0, 0, 32)])
