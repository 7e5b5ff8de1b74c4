"""The streaming path's plan, restated on the host, checked for coverage and bounds.

The plan kernel (csrc/stream.cu) cuts every group into row tiles, every tile's
shrink into K-chunks and its expand into units, and gives each block of the
shrink and expand launches a contiguous run of that work by bytes.  A mistake
there shows up on the GPU as work done twice or never, or as a copy past a
staging buffer.  This test restates the same arithmetic in Python (the sizes
are read from the kernel source, so the two cannot drift apart silently) and
checks, over the benchmark workloads and adversarial group orders (large and
small groups interleaved, single rows, the widest A block):

  * every (tile, chunk) and every (tile, unit) belongs to exactly one block,
    and the blocks' runs are contiguous and in order;
  * tiles of one group differ by at most one row and share the chunk cut, the
    stage K and the unit width (the summation order may not depend on which
    tile a row lands in);
  * every shrink stage, expand stage, S buffer and tensor-memory accumulator
    fits its buffer, and the partials stay within their per-row bound.
"""
import os
import re

import numpy as np
import pytest

from segmented_rank_gemm_lora_gb300 import synth

SRC = os.path.join(os.path.dirname(__file__), "..", "segmented_rank_gemm_lora_gb300", "csrc", "stream.cu")


def _constants():
    text = open(SRC).read()
    out = {}
    for name in ("kPlanItems", "kPartialPerRow", "kTileRows", "kShStageBytes", "kExBBytes", "kExYBytes",
                 "kExSBytes", "kExAccCols", "kCostUnit", "kExPoolDiv", "kExUposCap"):
        m = re.search(r"constexpr int %s = ([0-9* ]+);" % name, text)
        assert m, name
        out[name] = int(eval(m.group(1)))
    return out


C = _constants()


def rpad(r):
    return (r + 15) // 16 * 16


def f32(x):
    return np.float32(x)


def plan(groups, ranks, K, slice_n, n_a, grid, tile_max=128):
    """groups: list of (adapter, count).  Returns tiles (dicts), shrink and expand cost prefixes."""
    ntl = []
    est = 0
    for a, cnt in groups:
        R = n_a * rpad(ranks[a])
        tmax = min(tile_max, C["kTileRows"])
        n = -(-cnt // tmax)
        ntl.append(n)
        est += K * 2 * (R * n + cnt)
    target = max(f32(1), f32(est) / (f32(grid) * f32(C["kPlanItems"])))
    tiles = []
    for g, (a, cnt) in enumerate(groups):
        rp = rpad(ranks[a])
        R = n_a * rp
        n = ntl[g]
        base, rem = divmod(cnt, n)
        m_max = base + (1 if rem else 0)
        ks = min(512, C["kShStageBytes"] // 2 // (R + (m_max + 15) // 16 * 16)) // 16 * 16
        k_all = -(-K // ks) * ks
        kcap = k_all
        kc_min = min(-(-(-(-K * R // C["kPartialPerRow"])) // ks) * ks, kcap)
        want = min(f32(target / f32(2 * (R + m_max))), f32(k_all))
        kc = int(np.ceil(f32(want / f32(ks)))) * ks
        kc = min(max(kc, max(ks, kc_min)), kcap)
        n_kc = -(-K // kc)
        npad_max = -(-m_max // 16) * 16
        W = 1024
        while W > 128 and (W * rp * 2 > C["kExBBytes"] or W * m_max * 2 > C["kExYBytes"]
                           or (W // 128) * npad_max > C["kExAccCols"]):
            W //= 2
        n_units = sum(-(-s // W) for s in slice_n)
        row = 0
        for i in range(n):
            m = base + (1 if i < rem else 0)
            tiles.append(dict(g=g, a=a, m=m, row0=row, rp=rp, R=R, n_pad=-(-m // 16) * 16, kc=kc, n_kc=n_kc,
                              ks=ks, W=W, n_units=n_units, m_max=m_max,
                              cs=max(1, kc * (R + m) * 2 // C["kCostUnit"]),
                              cu=max(1, W * (rp + 2 * m) * 2 // C["kCostUnit"])))
            row += m
    sh = [t["n_kc"] * t["cs"] for t in tiles]
    ex = [t["n_units"] * t["cu"] for t in tiles]
    sh_pre = np.concatenate([[0], np.cumsum(sh)]).astype(np.int64)
    ex_pre = np.concatenate([[0], np.cumsum(ex)]).astype(np.int64)
    return tiles, sh_pre, ex_pre


def block_start(pre, tiles, T, G, c, key, T_split=None):
    """First (tile, item) of block c: shares of T_split (T unless given) that differ by at most one, block c
    starting at c q + min(c, r) with q = T_split // G, r = T_split % G (so block G starts at T_split); the
    first item at or past that position."""
    nt = len(tiles)
    T_split = T if T_split is None else T_split
    q, r = divmod(T_split, G)
    lo = c * q + min(c, r)
    if lo >= T:
        return (nt, 0)
    l = int(np.searchsorted(pre, lo, side="right")) - 1
    n = tiles[l][key]
    per = (pre[l + 1] - pre[l]) // n
    j = (lo - pre[l] + per - 1) // per
    return (l + 1, 0) if j >= n else (l, int(j))


def walk(start, end, tiles, key):
    t, j = start
    out = []
    while (t, j) < end:
        out.append((t, j))
        j += 1
        if j == tiles[t][key]:
            t, j = t + 1, 0
    return out


def check(groups, ranks, K, slice_n, n_a, grid, tile_max=128):
    tiles, sh_pre, ex_pre = plan(groups, ranks, K, slice_n, n_a, grid, tile_max)
    for key, pre in (("n_kc", sh_pre), ("n_units", ex_pre)):
        T = int(pre[-1])
        # the expand splits all but the last 1 / kExPoolDiv of its cost ahead of time; the units from block
        # `grid`'s start on are claimed one by one (launch-wide index u0[tile] + unit)
        T_split = T
        if key == "n_units" and len(tiles) <= C["kExUposCap"]:
            T_split = T - T // C["kExPoolDiv"]
        starts = [block_start(pre, tiles, T, grid, c, key, T_split) for c in range(grid + 1)]
        if T_split == T:
            assert starts[-1] == (len(tiles), 0)
        seen = []
        for c in range(grid):
            assert starts[c] <= starts[c + 1]
            seen += walk(starts[c], starts[c + 1], tiles, key)
        pool = walk(starts[grid], (len(tiles), 0), tiles, key)
        every = [(t, j) for t in range(len(tiles)) for j in range(tiles[t][key])]
        assert seen + pool == every, key
        if key == "n_units":
            u0 = np.concatenate([[0], np.cumsum([t[key] for t in tiles])]).astype(np.int64)
            g0 = int(u0[starts[grid][0]]) + starts[grid][1]
            for g in range(g0, int(u0[-1])):   # a claim's tile lookup
                l = int(np.searchsorted(u0, g, side="right")) - 1
                assert pool[g - g0] == (l, g - int(u0[l]))
    for t in tiles:
        assert 1 <= t["m"] <= C["kTileRows"] and t["m"] <= tile_max
        assert (t["R"] + t["n_pad"]) * t["ks"] * 2 <= C["kShStageBytes"]
        assert t["W"] * t["rp"] * 2 <= C["kExBBytes"] and t["W"] * t["m"] * 2 <= C["kExYBytes"]
        assert (t["W"] // 128) * t["n_pad"] <= C["kExAccCols"]
        assert t["rp"] * t["n_pad"] * 2 <= C["kExSBytes"]
        assert t["kc"] % t["ks"] == 0 and t["ks"] % 16 == 0 and 16 <= t["ks"] <= 512 and t["W"] % 128 == 0
        assert t["n_kc"] * t["R"] <= max(C["kPartialPerRow"] + t["R"], -(-K // t["kc"]) * t["R"])
        assert (t["n_kc"] - 1) * t["kc"] < K <= t["n_kc"] * t["kc"]
    by_group = {}
    for t in tiles:
        by_group.setdefault(t["g"], []).append(t)
    for g, ts in by_group.items():
        assert max(t["m"] for t in ts) - min(t["m"] for t in ts) <= 1
        assert sum(t["m"] for t in ts) == groups[g][1]
        for k in ("kc", "ks", "W", "n_kc", "n_units"):
            assert len({t[k] for t in ts}) == 1, k
    return tiles


def counts(ids, L):
    return [(a, int((ids == a).sum())) for a in range(L) if (ids == a).sum() > 0]


# (ids, ranks, K, slice widths, n_a) of the benchmark workloads, without drawing their weights
WORKLOADS = {
    "decode": lambda: (synth.ids_decode(1), synth.cycle_ranks(20), 4096, [4096], 1),
    "prefill": lambda: (synth.ids_prefill(2), synth.cycle_ranks(16), 4096, [4096], 1),
    "stacked_qkv": lambda: (synth.ids_stacked(3), [64] * 32, 4096, [4096, 1024, 1024], 3),
    "stacked_gate_up": lambda: (synth.ids_stacked(3), [64] * 32, 4096, [14336, 14336], 2),
    "stacked_down": lambda: (synth.ids_stacked(3), [64] * 32, 14336, [4096], 1),
}


@pytest.mark.parametrize("name", sorted(WORKLOADS))
@pytest.mark.parametrize("tile_max", [128, 16])
def test_plan_covers_the_workloads_exactly_once(name, tile_max):
    ids, ranks, K, slices, n_a = WORKLOADS[name]()
    check(counts(ids, len(ranks)), ranks, K, slices, n_a, 152, tile_max)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("n_a,slices", [(1, [4096]), (3, [4096, 1024, 1024]), (4, [256, 128, 384, 136]),
                                        (1, [72, 136])])
def test_plan_under_adversarial_group_orders(seed, n_a, slices):
    """Long, short and single-row groups interleaved in every order, ranks 1..64, grids of 1..1024 blocks."""
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 48))
    ranks = [int(r) for r in rng.integers(1, 65, L)]
    sizes = rng.choice([1, 2, 15, 16, 17, 31, 33, 64, 65, 127, 128, 129, 300, 512, 1000], L)
    groups = [(a, int(s)) for a, s in zip(rng.permutation(L), sizes)]
    K = int(rng.choice([8, 200, 264, 4096, 14336]))
    for grid in (1, 7, 152, 1024):
        check(groups, ranks, K, slices, n_a, grid, tile_max=16 if grid == 7 else 128)


def test_plan_with_one_tiny_group_and_a_huge_grid():
    check([(0, 1)], [8], 8, [8], 1, 1024)
    check([(0, 1)], [64], 1 << 20, [4096], 1, 152)
