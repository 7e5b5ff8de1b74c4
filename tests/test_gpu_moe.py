"""lora_moe_delta on the GPU vs the CPU oracle (gate/up before SiLU-mul, down
before the top-k reduce), at the full MoE workload size and on small shapes."""
import numpy as np
import pytest
import torch

import oracle
from segmented_rank_gemm_lora_gb300 import lora, synth
from gpu_util import PATHS, check_close, dev_bf16, forced_path, host_bits, host_f64

pytestmark = pytest.mark.gpu


def _tables(p):
    gu = lora.lora_pack_weights([dev_bf16(a) for a in p.A_gu], [dev_bf16(b) for b in p.B_gu], p.ranks, p.scales,
                                p.H, [2 * p.I], 1, E_A=p.A_gu[0].shape[0], E_B=p.B_gu[0].shape[0])
    dn = lora.lora_pack_weights([dev_bf16(a) for a in p.A_d], [dev_bf16(b) for b in p.B_d], p.ranks, p.scales,
                                p.I, [p.H], 1, E_A=p.A_d[0].shape[0], E_B=p.B_d[0].shape[0])
    return gu, dn


def run_moe(p, weights=False):
    gu, dn = _tables(p)
    ws = lora.Workspace(p.M, p.L, p.topk, p.E, p.block_m)
    lora.lora_build_segments(ws, torch.from_numpy(p.ids).cuda(), torch.from_numpy(p.topk_ids).cuda())
    x = dev_bf16(p.x)
    c1 = dev_bf16(p.cache1)
    c2 = dev_bf16(p.cache2)
    c3 = dev_bf16(p.cache3)
    w = torch.from_numpy(p.topk_weights.reshape(-1).copy()).cuda() if weights else None
    lora.lora_moe_delta(gu, lora.LORA_MOE_GATE_UP, ws, x, c1)
    lora.lora_moe_delta(dn, lora.LORA_MOE_DOWN, ws, c2, c3, w)
    assert lora.lora_get_status(ws) == lora.LORA_OK
    return c1, c3


def refs(p, weights=False):
    r1, _ = oracle.moe_delta(p.ids, p.topk_ids, p.x, p.cache1, p.A_gu, p.B_gu, p.ranks, p.scales, p.E, True)
    r3, _ = oracle.moe_delta(p.ids, p.topk_ids, p.cache2, p.cache3, p.A_d, p.B_d, p.ranks, p.scales, p.E, False,
                             topk_weights=p.topk_weights if weights else None)
    return r1, r3


@pytest.mark.parametrize("zero_base", [False, True])
def test_moe_workload_matches_oracle(zero_base):
    p = synth.moe(zero_base=zero_base)
    r1, r3 = refs(p)
    for path in PATHS:
        with forced_path(path):
            c1, c3 = run_moe(p)
        check_close(host_f64(c1), r1, "gate_up path %d" % path)
        check_close(host_f64(c3), r3, "down path %d" % path)


@pytest.mark.parametrize("shared", [True, False])
@pytest.mark.parametrize("weights", [False, True])
def test_moe_small_shapes(shared, weights):
    ids = np.random.default_rng(2).integers(-1, 3, 45).astype(np.int32)
    p = synth.make_moe(5, 45, 264, 200, 6, 3, [8, 24, 64], block_m=16, ids=ids, shared_outer=shared,
                       zero_base=True)
    r1, r3 = refs(p, weights)
    for path in PATHS:
        with forced_path(path):
            c1, c3 = run_moe(p, weights)
        check_close(host_f64(c1), r1, "gate_up path %d" % path)
        check_close(host_f64(c3), r3, "down path %d" % path)
        none = np.repeat(ids < 0, p.topk)
        assert np.array_equal(host_bits(c1)[none], p.cache1[none])
        assert np.array_equal(host_bits(c3)[none], p.cache3[none])
