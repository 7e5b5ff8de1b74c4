"""Pins for the MoE LoRA delta oracle (CPU only).

"[SGLang] LoRA + MoE fusion" states why the deltas go where they go: added
before the activation (stage 1.5) and before the final reduce (stage 3.5),
the LoRA MoE block equals an MoE block whose expert weights are merged,
W13'[e] = W13[e] + scale * B_gu[e] A_gu and W2'[e] = W2[e] + scale * B_d A_d[e].
These tests build that merged block with numpy in float64 and compare; a
negative test shows that moving the gate/up delta after SiLU-mul breaks the
identity, and planted mistakes in a copy of the oracle are rejected.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from segmented_rank_gemm_lora_gb300 import synth

bf = synth.bf16_bits_to_f32


def silu_mul(c, I):
    g, u = c[:, :I], c[:, I:]
    return g / (1.0 + np.exp(-g)) * u


def _problem(seed=0, shared=True, L=2, M=7, H=24, I=16, E=4, topk=2, ranks=(8, 16)):
    p = synth.make_moe(seed, M, H, I, E, topk, list(ranks)[:L], block_m=4, shared_outer=shared, zero_base=True)
    p.scales = [1.5 + 0.5 * l for l in range(L)]
    rng = np.random.default_rng(seed + 99)
    W13 = synth.f32_to_bf16_bits(rng.standard_normal((E, 2 * I, H)).astype(np.float32) / np.sqrt(H))
    W2 = synth.f32_to_bf16_bits(rng.standard_normal((E, H, I)).astype(np.float32) / np.sqrt(I))
    return p, bf(W13).astype(np.float64), bf(W2).astype(np.float64)


def lora_block(p, W13, W2, delta_after_act=False):
    """MoE block with the oracle's deltas at the pages' insertion points; returns (cache1, act_bits, cache3, y)."""
    x = bf(p.x).astype(np.float64)
    P = p.M * p.topk
    e = p.topk_ids.reshape(-1)
    t = np.arange(P) // p.topk
    base1 = np.einsum("ph,pnh->pn", x[t], W13[e])
    d1, _ = oracle.moe_delta(p.ids, p.topk_ids, p.x, np.zeros((P, 2 * p.I), np.uint16), p.A_gu, p.B_gu,
                             p.ranks, p.scales, p.E, src_is_token=True)
    if delta_after_act:
        act = silu_mul(base1, p.I) + d1[:, :p.I]
    else:
        act = silu_mul(base1 + d1, p.I)
    act_bits = synth.f32_to_bf16_bits(act.astype(np.float32))
    a = bf(act_bits).astype(np.float64)
    base3 = np.einsum("pi,phi->ph", a, W2[e])
    d3, _ = oracle.moe_delta(p.ids, p.topk_ids, act_bits, np.zeros((P, p.H), np.uint16), p.A_d, p.B_d,
                             p.ranks, p.scales, p.E, src_is_token=False)
    c3 = base3 + d3
    y = (p.topk_weights.reshape(-1, 1).astype(np.float64) * c3).reshape(p.M, p.topk, p.H).sum(1)
    return base1 + d1, act_bits, c3, y


def merged_block(p, W13, W2, act_bits):
    x = bf(p.x).astype(np.float64)
    P = p.M * p.topk
    e_of = p.topk_ids.reshape(-1)
    c1 = np.zeros((P, 2 * p.I))
    c3 = np.zeros((P, p.H))
    a = bf(act_bits).astype(np.float64)
    for q in range(P):
        t, e = q // p.topk, e_of[q]
        l = p.ids[t]
        W13m, W2m = W13[e].copy(), W2[e].copy()
        if 0 <= l < p.L:
            Agu = bf(p.A_gu[l][0 if p.A_gu[l].shape[0] == 1 else e]).astype(np.float64)
            Bgu = bf(p.B_gu[l][0 if p.B_gu[l].shape[0] == 1 else e]).astype(np.float64)
            Ad = bf(p.A_d[l][0 if p.A_d[l].shape[0] == 1 else e]).astype(np.float64)
            Bd = bf(p.B_d[l][0 if p.B_d[l].shape[0] == 1 else e]).astype(np.float64)
            W13m += p.scales[l] * Bgu @ Agu
            W2m += p.scales[l] * Bd @ Ad
        c1[q] = W13m @ x[t]
        c3[q] = W2m @ a[q]
    return c1, c3


@pytest.mark.parametrize("shared", [True, False])
@pytest.mark.parametrize("seed", [0, 1])
def test_moe_block_equals_merged_weight_block(shared, seed):
    p, W13, W2 = _problem(seed, shared)
    p.ids[1] = -1
    c1, act_bits, c3, _ = lora_block(p, W13, W2)
    m1, m3 = merged_block(p, W13, W2, act_bits)
    assert np.abs(c1 - m1).max() <= 1e-12 * np.abs(m1).max()
    assert np.abs(c3 - m3).max() <= 1e-12 * np.abs(m3).max()
    # the merged activation rounds to the same bf16 input of the down projection
    m_act = synth.f32_to_bf16_bits(silu_mul(m1, p.I).astype(np.float32))
    assert (m_act != act_bits).mean() < 0.01


def test_delta_after_activation_breaks_the_identity():
    p, W13, W2 = _problem(3, True)
    c1, act_bits, _, _ = lora_block(p, W13, W2)
    _, act_wrong, _, _ = lora_block(p, W13, W2, delta_after_act=True)
    m1, _ = merged_block(p, W13, W2, act_bits)
    right = np.abs(bf(act_bits) - silu_mul(m1, p.I)).max()
    wrong = np.abs(bf(act_wrong) - silu_mul(m1, p.I)).max()
    assert wrong > 50 * right


def test_topk_weights_scale_the_down_delta():
    p, _, _ = _problem(4, True)
    P = p.M * p.topk
    plain, _ = oracle.moe_delta(p.ids, p.topk_ids, p.cache2, np.zeros((P, p.H), np.uint16), p.A_d, p.B_d,
                                p.ranks, p.scales, p.E, src_is_token=False)
    wtd, _ = oracle.moe_delta(p.ids, p.topk_ids, p.cache2, np.zeros((P, p.H), np.uint16), p.A_d, p.B_d,
                              p.ranks, p.scales, p.E, src_is_token=False, topk_weights=p.topk_weights)
    w = p.topk_weights.reshape(-1, 1).astype(np.float64)
    assert np.abs(wtd - w * plain).max() <= 1e-12 * np.abs(wtd).max()


def test_none_and_disabled_pairs_copy_the_cache():
    p, _, _ = _problem(5, True, L=2)
    p.ids[:] = [0, -1, 1, 0, 5, 1, -1]
    p.cache1 = synth.f32_to_bf16_bits(np.random.default_rng(0).standard_normal((p.M * p.topk, 2 * p.I))
                                      .astype(np.float32))
    out, bad = oracle.moe_delta(p.ids, p.topk_ids, p.x, p.cache1, p.A_gu, p.B_gu, p.ranks, p.scales, p.E,
                                src_is_token=True, enabled=np.array([1, 0], np.uint8))
    assert bad == 2   # both pairs of the out-of-range token
    c = bf(p.cache1).astype(np.float64)
    for t in range(p.M):
        rows = slice(t * p.topk, (t + 1) * p.topk)
        if p.ids[t] != 0:
            assert np.array_equal(out[rows], c[rows])
        else:
            assert not np.array_equal(out[rows], c[rows])


MUTANTS = {
    "expert_of_token": ("int32_t e = topk_ids[p];\n        if (l == -1) continue;",
                        "int32_t e = topk_ids[t * topk];\n        if (l == -1) continue;"),
    "src_per_pair": ("(src_is_token ? t : p)", "(src_is_token ? p % M : p)"),
    "expert_B_ignored": ("(E_B == 1 ? 0 : e) * N * r", "0 * N * r"),
    "drop_weight": ("double w = topk_weights ? (double)topk_weights[p] : 1.0;", "double w = 1.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "lora_oracle.c")).read()
    a, b = MUTANTS[name]
    assert a in src, name
    (tmp_path / "m.c").write_text(src.replace(a, b))
    so = tmp_path / "m.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-ffp-contract=off", "-shared", "-fPIC", "-o", str(so),
                    str(tmp_path / "m.c")], check=True)
    lib = ctypes.CDLL(str(so))
    lib.oracle_moe_delta.restype = ctypes.c_int
    lib.oracle_moe_delta.argtypes = oracle._load().oracle_moe_delta.argtypes
    saved = oracle._lib.oracle_moe_delta
    caught = False
    try:
        oracle._lib.oracle_moe_delta = lib.oracle_moe_delta
        for fn in (lambda: test_moe_block_equals_merged_weight_block(True, 0),
                   lambda: test_moe_block_equals_merged_weight_block(False, 1),
                   test_topk_weights_scale_the_down_delta):
            try:
                fn()
            except AssertionError:
                caught = True
    finally:
        oracle._lib.oracle_moe_delta = saved
    assert caught, "pins accepted the planted mistake " + name
