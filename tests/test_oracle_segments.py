"""Pins for the segment-table and MoE-alignment oracles (CPU only).

The segment table is checked against a library sort on the key
(bucket, token index) -- the definition of a stable bucketing -- and against
the id examples worked out by hand from "vLLM-Ascend dynamic LoRA fused
operator" sections 2.3 and 3.4 (tests/golden/p1_segment_examples.txt).
The MoE alignment is checked against numpy lexsort plus a vectorised padding
layout, and against the invariants moe_lora_align_block_size must keep
("[SGLang] LoRA + MoE fusion", MoE LoRA Alignment).
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def sorted_reference(ids, L, enabled=None):
    ids = np.asarray(ids)
    M = len(ids)
    ok = (ids >= 0) & (ids < L)
    if enabled is not None:
        ok &= np.asarray(enabled, bool)[np.clip(ids, 0, L - 1)]
    bucket = np.where(ok, ids, L)
    perm = np.array(sorted(range(M), key=lambda t: (bucket[t], t)), np.int32)
    segs = []
    start = 0
    for a in range(L):
        n = int((bucket == a).sum())
        if n:
            segs.append((a, start, n))
        start += n
    return perm, segs, int(ok.sum())


def load_golden_segments():
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, "p1_segment_examples.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0]}
            cases.append(cur)
        elif key == "L":
            cur["L"] = int(vals[0])
        elif key in ("ids", "perm"):
            cur[key] = [int(v) for v in vals]
        elif key == "segments":
            cur["segments"] = [tuple(int(u) for u in v.split(":")) for v in vals]
    return cases


@pytest.mark.parametrize("case", load_golden_segments(), ids=lambda c: c["name"])
def test_golden_examples_from_the_pages(case):
    s = oracle.build_segments(np.array(case["ids"], np.int32), case["L"])
    assert s["perm"].tolist() == case["perm"]
    got = list(zip(s["seg_adapter"].tolist(), s["seg_start"].tolist(), s["seg_len"].tolist()))
    assert got == case["segments"]


def _maps():
    rng = np.random.default_rng(0)
    yield "random", rng.integers(-1, 20, 300).astype(np.int32), 20
    yield "all_none", np.full(50, -1, np.int32), 4
    yield "one_adapter", np.full(33, 2, np.int32), 4
    yield "single_token", np.array([3], np.int32), 4
    yield "empty", np.zeros(0, np.int32), 4
    yield "each_once", rng.permutation(64).astype(np.int32), 64
    yield "edges", np.array([0, 63, 0, 63, -1, 63], np.int32), 64
    yield "bad_ids", np.array([0, 7, -3, 1, 4, -1, 1], np.int32), 4
    yield "prefill_runs", np.repeat(rng.permutation(16), rng.integers(1, 40, 16)).astype(np.int32), 16


@pytest.mark.parametrize("name,ids,L", list(_maps()), ids=[m[0] for m in _maps()])
def test_segments_match_stable_sort(name, ids, L):
    s = oracle.build_segments(ids, L)
    perm, segs, nv = sorted_reference(ids, L)
    assert s["perm"].tolist() == perm.tolist()
    got = list(zip(s["seg_adapter"].tolist(), s["seg_start"].tolist(), s["seg_len"].tolist()))
    assert got == segs
    assert s["num_valid"] == nv
    assert s["bad"] == int(((ids < -1) | (ids >= L)).sum())
    # invariants: a permutation, runs of one id, ascending token order in a run
    assert sorted(s["perm"].tolist()) == list(range(len(ids)))
    for a, st, n in got:
        toks = s["perm"][st:st + n]
        assert (ids[toks] == a).all() and (np.diff(toks) > 0).all()


def test_segments_enabled_mask():
    ids = np.array([0, 1, 2, 1, 0, 2, -1], np.int32)
    en = np.array([1, 0, 1], np.uint8)
    s = oracle.build_segments(ids, 3, enabled=en)
    perm, segs, nv = sorted_reference(ids, 3, en)
    assert s["perm"].tolist() == perm.tolist() and s["num_valid"] == nv == 4
    assert s["seg_adapter"].tolist() == [0, 2]


# ----------------------------------------------------------------------------
# MoE alignment
# ----------------------------------------------------------------------------
def align_reference(ids, topk_ids, L, E, bm, enabled=None):
    """numpy lexsort on (adapter, expert, pair) plus a vectorised padded layout."""
    M, topk = topk_ids.shape
    P = M * topk
    P_max, B_max = oracle.moe_padded_sizes(M, topk, E, bm)
    pl = np.repeat(ids, topk)
    pe = topk_ids.reshape(-1)
    pp = np.arange(P)
    ok = (pl >= 0) & (pl < L) & (pe >= 0) & (pe < E)
    if enabled is not None:
        ok &= np.asarray(enabled, bool)[np.clip(pl, 0, L - 1)]
    sel = np.nonzero(ok)[0]
    order = sel[np.lexsort((pp[sel], pe[sel], pl[sel]))]
    srt = np.full((L, P_max), P, np.int32)
    eid = np.full((L, B_max), -1, np.int32)
    ntpp = np.zeros(L, np.int32)
    counts = np.zeros((L, E), np.int64)
    np.add.at(counts, (pl[order], pe[order]), 1)
    padded = -(-counts // bm) * bm
    starts = np.concatenate([np.zeros((L, 1), np.int64), np.cumsum(padded, axis=1)[:, :-1]], axis=1)
    first = np.concatenate([[0], np.cumsum(counts.reshape(-1))[:-1]]).reshape(L, E)
    for l in range(L):
        for e in range(E):
            c = counts[l, e]
            srt[l, starts[l, e]:starts[l, e] + c] = order[first[l, e]:first[l, e] + c]
            eid[l, starts[l, e] // bm:(starts[l, e] + padded[l, e]) // bm] = e
        ntpp[l] = padded[l].sum()
    return srt, eid, ntpp


def _moe_cases():
    rng = np.random.default_rng(1)
    M, topk, E, L = 40, 2, 4, 3
    ids = rng.integers(-1, L, M).astype(np.int32)
    tk = np.stack([rng.permutation(E)[:topk] for _ in range(M)]).astype(np.int32)
    yield "random", ids, tk, L, E, 8
    yield "block1", ids, tk, L, E, 1
    yield "all_none", np.full(M, -1, np.int32), tk, L, E, 8
    yield "one_expert", np.zeros(12, np.int32), np.zeros((12, 1), np.int32), 2, 4, 4
    M2 = 512
    ids2 = rng.integers(0, 8, M2).astype(np.int32)
    tk2 = np.stack([rng.permutation(8)[:2] for _ in range(M2)]).astype(np.int32)
    yield "moe_full_size", ids2, tk2, 8, 8, 64


@pytest.mark.parametrize("name,ids,tk,L,E,bm", list(_moe_cases()), ids=[c[0] for c in _moe_cases()])
def test_moe_alignment_matches_lexsort_layout(name, ids, tk, L, E, bm):
    r = oracle.moe_align(ids, tk, L, E, bm)
    srt, eid, ntpp = align_reference(ids, tk, L, E, bm)
    assert np.array_equal(r["sorted_ids"], srt)
    assert np.array_equal(r["expert_ids"], eid)
    assert np.array_equal(r["ntpp"], ntpp)
    # invariants: every real pair exactly once, groups padded to bm, blocks carry their expert
    M, topk = tk.shape
    P = M * topk
    real = r["sorted_ids"][r["sorted_ids"] != P]
    expect = [p for p in range(P) if 0 <= ids[p // topk] < L]
    assert sorted(real.tolist()) == expect
    assert (r["ntpp"] % bm == 0).all()
    for l in range(L):
        for b in range(r["ntpp"][l] // bm):
            e = r["expert_ids"][l, b]
            blk = r["sorted_ids"][l, b * bm:(b + 1) * bm]
            blk = blk[blk != P]
            assert ((tk.reshape(-1)[blk] == e) & (ids[blk // topk] == l)).all()


def test_moe_alignment_enabled_and_bad_experts():
    ids = np.array([0, 1, 1, 0, 2], np.int32)
    tk = np.array([[0, 1], [1, 5], [2, 0], [0, 3], [1, 1]], np.int32)   # expert 5 out of range for E=4
    en = np.array([1, 1, 0], np.uint8)
    r = oracle.moe_align(ids, tk, 3, 4, 2, enabled=en)
    assert r["bad"] == 1
    ok_tk = tk.copy()
    srt, eid, ntpp = align_reference(ids, ok_tk, 3, 4, 2, enabled=en)
    assert np.array_equal(r["sorted_ids"], srt) and np.array_equal(r["ntpp"], ntpp)
    assert r["ntpp"][2] == 0
