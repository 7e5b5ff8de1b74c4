"""Device segment table and MoE alignment vs the CPU oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from segmented_rank_gemm_lora_gb300 import lora, synth

pytestmark = pytest.mark.gpu


def id_maps():
    rng = np.random.default_rng(7)
    yield "tiny", synth.ids_tiny(0), 4
    yield "decode", synth.ids_decode(1), 20
    yield "prefill", synth.ids_prefill(2), 16
    yield "stacked", synth.ids_stacked(3), 32
    yield "all_none", np.full(100, -1, np.int32), 8
    yield "one_adapter", np.full(77, 5, np.int32), 8
    yield "single", np.array([2], np.int32), 4
    yield "each_once", rng.permutation(64).astype(np.int32), 64
    yield "edges", np.array([0, 63, 0, 63, -1, 63] * 9, np.int32), 64
    yield "large", rng.integers(-1, 100, 5000).astype(np.int32), 100
    yield "many_adapters", rng.integers(-1, 3000, 2500).astype(np.int32), 3000


@pytest.mark.parametrize("name,ids,L", list(id_maps()), ids=[m[0] for m in id_maps()])
def test_segments_bit_exact(name, ids, L):
    ws = lora.Workspace(len(ids), L)
    lora.lora_build_segments(ws, torch.from_numpy(ids).cuda())
    assert lora.lora_get_status(ws) == lora.LORA_OK
    got = ws.read_segments()
    ref = oracle.build_segments(ids, L)
    assert got["M"] == len(ids)
    assert np.array_equal(got["perm"], ref["perm"])
    assert got["num_segments"] == ref["num_segments"] and got["num_valid"] == ref["num_valid"]
    segs = got["segments"]
    assert np.array_equal(segs[:, 0], ref["seg_adapter"])
    assert (segs[:, 1] == 0).all()
    assert np.array_equal(segs[:, 2], ref["seg_start"])
    assert np.array_equal(segs[:, 3], ref["seg_len"])


def test_empty_map():
    ws = lora.Workspace(8, 4)
    lora.lora_build_segments(ws, torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert lora.lora_get_status(ws) == lora.LORA_OK
    got = ws.read_segments()
    assert got["M"] == 0 and got["num_segments"] == 0 and got["num_valid"] == 0


def test_bad_ids_are_dropped_and_reported():
    ids = np.array([0, 9, 1, -5, 2, -1, 3], np.int32)
    ws = lora.Workspace(len(ids), 4)
    lora.lora_build_segments(ws, torch.from_numpy(ids).cuda())
    assert lora.lora_get_status(ws) == lora.LORA_ERR_BAD_ADAPTER_ID
    assert lora.lora_get_status(ws) == lora.LORA_OK          # sticky word was cleared
    got = ws.read_segments()
    ref = oracle.build_segments(ids, 4)
    assert np.array_equal(got["perm"], ref["perm"]) and got["num_valid"] == ref["num_valid"] == 4


def test_enabled_mask():
    ids = synth.ids_decode(5)
    en = (np.arange(20) % 3 != 1).astype(np.uint8)
    ws = lora.Workspace(len(ids), 20)
    lora.lora_build_segments(ws, torch.from_numpy(ids).cuda(), enabled=torch.from_numpy(en).cuda())
    got = ws.read_segments()
    ref = oracle.build_segments(ids, 20, enabled=en)
    assert np.array_equal(got["perm"], ref["perm"])
    assert np.array_equal(got["segments"][:, 0], ref["seg_adapter"])


def moe_cases():
    ids, tk, _ = synth.moe_routing(4, 512, 8, 2, 8)
    yield "moe_config", ids, tk, 8, 8, 64
    rng = np.random.default_rng(3)
    ids = rng.integers(-1, 5, 300).astype(np.int32)
    tk = np.stack([rng.permutation(16)[:4] for _ in range(300)]).astype(np.int32)
    yield "topk4_e16", ids, tk, 5, 16, 16
    yield "bm1", ids, tk, 5, 16, 1
    yield "one_pair", np.array([0], np.int32), np.array([[3]], np.int32), 1, 4, 64


@pytest.mark.parametrize("name,ids,tk,L,E,bm", list(moe_cases()), ids=[c[0] for c in moe_cases()])
def test_moe_alignment_bit_exact(name, ids, tk, L, E, bm):
    M, topk = tk.shape
    ws = lora.Workspace(M, L, topk, E, bm)
    lora.lora_build_segments(ws, torch.from_numpy(ids).cuda(), torch.from_numpy(np.ascontiguousarray(tk)).cuda())
    assert lora.lora_get_status(ws) == lora.LORA_OK
    got = ws.read_segments()
    ref = oracle.moe_align(ids, tk, L, E, bm)
    assert got["P_max"] == ref["P_max"] and got["B_max"] == ref["B_max"]
    assert np.array_equal(got["sorted_ids"], ref["sorted_ids"])
    assert np.array_equal(got["expert_ids"], ref["expert_ids"])
    assert np.array_equal(got["ntpp"], ref["ntpp"])
    # group list: every non-empty (adapter, expert) with its start and count
    groups = got["moe_groups"]
    P = M * topk
    for l, e, start, cnt in groups:
        row = ref["sorted_ids"].reshape(-1)[start:start + cnt]
        assert (row != P).all() and (tk.reshape(-1)[row] == e).all() and (ids[row // topk] == l).all()
    assert groups[:, 3].sum() == int((ref["sorted_ids"] != P).sum())


def test_moe_bad_expert_reported():
    ids = np.array([0, 1, 0], np.int32)
    tk = np.array([[0, 1], [7, 2], [3, 0]], np.int32)
    ws = lora.Workspace(3, 2, 2, 4, 2)
    lora.lora_build_segments(ws, torch.from_numpy(ids).cuda(), torch.from_numpy(tk).cuda())
    assert lora.lora_get_status(ws) == lora.LORA_ERR_BAD_EXPERT_ID
    got = ws.read_segments()
    ref = oracle.moe_align(ids, tk, 2, 4, 2)
    assert np.array_equal(got["sorted_ids"], ref["sorted_ids"])
