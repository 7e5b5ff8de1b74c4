"""adapter_enabled under CUDA-graph capture, and group orders that interleave long and short runs.

"[SGLang] LoRA + MoE fusion" runs the LoRA layers inside a captured graph and switches adapters on and off
through a device mask (adapter_enabled) rather than by re-capturing.  Here the build and the apply (dense),
or the build and both MoE deltas, are captured once; the mask is rewritten in place between replays.  Each
replay must match the oracle run with the same mask: tokens of disabled adapters come out bit-identical to
y_base, the rest within the tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from segmented_rank_gemm_lora_gb300 import lora, synth
from gpu_util import PATHS, check_close, dev_bf16, forced_path, host_bits, host_f64, oracle_dense, pack_dense, run_dense

pytestmark = pytest.mark.gpu

MASKS = ("all", "even", "none_but_one", "odd")


def mask_of(kind, L):
    m = np.ones(L, np.uint8)
    if kind == "even":
        m[1::2] = 0
    elif kind == "odd":
        m[0::2] = 0
    elif kind == "none_but_one":
        m[:] = 0
        m[L // 2] = 1
    return m


@pytest.mark.parametrize("workload,path", [("decode", 0), ("decode", 1), ("stacked_qkv", 0), ("prefill", 3)])
@pytest.mark.parametrize("y_base", ["zero", "random"])
def test_dense_graph_replays_follow_the_mask(workload, path, y_base):
    if workload == "decode":
        p = synth.decode(3, y_base=y_base)
    elif workload == "prefill":
        p = synth.prefill(4, y_base=y_base)
    else:
        p = synth.stacked("qkv", seed=5, y_base=y_base)
    table = pack_dense(p)
    ws = lora.Workspace(p.M, p.L)
    ids = torch.from_numpy(p.ids).cuda()
    x = dev_bf16(p.x)
    y0 = dev_bf16(p.y_base)
    y = y0.clone()
    en = torch.ones(p.L, dtype=torch.uint8, device="cuda")
    with forced_path(path):
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            lora.lora_build_segments(ws, ids, enabled=en)
            lora.lora_apply(table, ws, x, y)
        for kind in MASKS:
            m = mask_of(kind, p.L)
            en.copy_(torch.from_numpy(m))
            y.copy_(y0)
            g.replay()
            torch.cuda.synchronize()
            assert lora.lora_get_status(ws) == lora.LORA_OK
            ref, bad = oracle.lora_apply(p.ids, p.x, p.y_base, p.A, p.B, p.ranks, p.scales, p.slice_n, p.n_a,
                                         enabled=m)
            assert bad == 0
            got_bits = host_bits(y)
            off = (p.ids < 0) | (m[np.clip(p.ids, 0, p.L - 1)] == 0)
            assert np.array_equal(got_bits[off], p.y_base[off]), "%s mask %s: disabled rows moved" % (workload, kind)
            if (~off).any():
                check_close(host_f64(y)[~off], ref[~off], "%s path %d mask %s" % (workload, path, kind))
    table.destroy()


@pytest.mark.parametrize("path", [0, 1])
def test_moe_graph_replays_follow_the_mask(path):
    p = synth.make_moe(6, 128, 2048, 1536, 8, 2, synth.cycle_ranks(6), block_m=64, zero_base=True)
    gu = lora.lora_pack_weights([dev_bf16(a) for a in p.A_gu], [dev_bf16(b) for b in p.B_gu], p.ranks, p.scales,
                                p.H, [2 * p.I], 1, E_A=p.A_gu[0].shape[0], E_B=p.B_gu[0].shape[0])
    dn = lora.lora_pack_weights([dev_bf16(a) for a in p.A_d], [dev_bf16(b) for b in p.B_d], p.ranks, p.scales,
                                p.I, [p.H], 1, E_A=p.A_d[0].shape[0], E_B=p.B_d[0].shape[0])
    ws = lora.Workspace(p.M, p.L, p.topk, p.E, p.block_m)
    ids = torch.from_numpy(p.ids).cuda()
    tk = torch.from_numpy(p.topk_ids).cuda()
    x = dev_bf16(p.x)
    c1_0, c3_0 = dev_bf16(p.cache1), dev_bf16(p.cache3)
    c2 = dev_bf16(p.cache2)
    c1, c3 = c1_0.clone(), c3_0.clone()
    en = torch.ones(p.L, dtype=torch.uint8, device="cuda")
    with forced_path(path):
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            lora.lora_build_segments(ws, ids, tk, enabled=en)
            lora.lora_moe_delta(gu, lora.LORA_MOE_GATE_UP, ws, x, c1)
            lora.lora_moe_delta(dn, lora.LORA_MOE_DOWN, ws, c2, c3)
        for kind in MASKS:
            m = mask_of(kind, p.L)
            en.copy_(torch.from_numpy(m))
            c1.copy_(c1_0)
            c3.copy_(c3_0)
            g.replay()
            torch.cuda.synchronize()
            assert lora.lora_get_status(ws) == lora.LORA_OK
            r1, _ = oracle.moe_delta(p.ids, p.topk_ids, p.x, p.cache1, p.A_gu, p.B_gu, p.ranks, p.scales, p.E, True,
                                     enabled=m)
            r3, _ = oracle.moe_delta(p.ids, p.topk_ids, p.cache2, p.cache3, p.A_d, p.B_d, p.ranks, p.scales, p.E,
                                     False, enabled=m)
            off = np.repeat((p.ids < 0) | (m[np.clip(p.ids, 0, p.L - 1)] == 0), p.topk)
            assert np.array_equal(host_bits(c1)[off], p.cache1[off]), "gate_up mask %s: disabled rows moved" % kind
            assert np.array_equal(host_bits(c3)[off], p.cache3[off]), "down mask %s: disabled rows moved" % kind
            if (~off).any():
                check_close(host_f64(c1)[~off], r1[~off], "gate_up path %d mask %s" % (path, kind))
                check_close(host_f64(c3)[~off], r3[~off], "down path %d mask %s" % (path, kind))
    gu.destroy()
    dn.destroy()


def test_long_short_long_runs_every_path():
    """A prefill-like map whose natural group order interleaves long runs (several 64- or 128-row tiles)
    with short ones (one small tile): long, short, long, short, long, with a decode tail."""
    rng = np.random.default_rng(23)
    runs = [(0, 300), (1, 5), (2, 260), (3, 2), (4, 411), (5, 17), (6, 129)]
    ids = np.concatenate([np.full(n, a, np.int32) for a, n in runs] + [rng.integers(-1, 7, 40).astype(np.int32)])
    p = synth.make_dense("long_short_long", 23, ids, 4096, [4096], [64, 16, 32, 64, 16, 32, 64], y_base="random")
    ref = oracle_dense(p)
    table = pack_dense(p)
    ws = lora.Workspace(p.M, p.L)
    for path in PATHS:
        with forced_path(path):
            y, _, _ = run_dense(p, table=table, ws=ws)
        assert lora.lora_get_status(ws) == lora.LORA_OK
        check_close(host_f64(y), ref, "long/short/long path=%d" % path)
    table.destroy()
