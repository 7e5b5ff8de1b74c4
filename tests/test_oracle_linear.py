"""Pins of the oracle's LoRA linear layer (base projection x W^T plus the delta; "vLLM-Ascend dynamic
LoRA fused operator", section 3.3), against values fixed independently of it:

  * a worked example small enough to check by hand;
  * W = I (N = K) and no adapter: y equals x exactly;
  * W a permutation of one-hot rows: column n of y is column pi(n) of x, exactly;
  * W = 0: y is the delta alone, as the (separately pinned) lora_apply gives it on y_base = 0;
  * the delta is added once: with scale 0 every token gets the base projection alone.
"""
import numpy as np

import oracle
from segmented_rank_gemm_lora_gb300 import synth


def bits(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_worked_example():
    x = bits([[1, 2], [3, 4]])
    W = bits([[1, 0], [1, 1], [0, 2]])
    A = [bits(np.zeros((16, 2)))]
    B = [bits(np.zeros((3, 16)))]
    y, bad = oracle.lora_linear(np.array([-1, -1], np.int32), x, W, A, B, [16], [1.0], [3])
    assert bad == 0
    assert np.array_equal(y, [[1, 3, 4], [3, 7, 8]])


def test_identity_weight_returns_x():
    rng = np.random.default_rng(0)
    p = synth.make_dense("pin", 1, np.full(7, -1, np.int32), 48, [48], [16, 32], y_base="zero")
    W = bits(np.eye(48))
    y, _ = oracle.lora_linear(p.ids, p.x, W, p.A, p.B, p.ranks, p.scales, p.slice_n, p.n_a)
    assert np.array_equal(y, synth.bf16_bits_to_f32(p.x).astype(np.float64))


def test_one_hot_rows_select_columns():
    rng = np.random.default_rng(1)
    K, N = 40, 24
    pi = rng.integers(0, K, N)
    Wf = np.zeros((N, K), np.float32)
    Wf[np.arange(N), pi] = 1.0
    p = synth.make_dense("pin", 2, np.full(5, -1, np.int32), K, [N], [16], y_base="zero")
    y, _ = oracle.lora_linear(p.ids, p.x, bits(Wf), p.A, p.B, p.ranks, p.scales, p.slice_n, p.n_a)
    assert np.array_equal(y, synth.bf16_bits_to_f32(p.x).astype(np.float64)[:, pi])


def test_zero_weight_is_the_delta_alone():
    ids = np.random.default_rng(2).integers(-1, 3, 21).astype(np.int32)
    p = synth.make_dense("pin", 3, ids, 72, [32, 40], [8, 16, 48], y_base="zero")
    W = np.zeros((72, 72), np.uint16)[:p.N]
    y, bad = oracle.lora_linear(p.ids, p.x, W, p.A, p.B, p.ranks, p.scales, p.slice_n, p.n_a)
    ref, bad2 = oracle.lora_apply(p.ids, p.x, np.zeros((p.M, p.N), np.uint16), p.A, p.B, p.ranks, p.scales,
                                  p.slice_n, p.n_a)
    assert bad == bad2 == 0
    assert np.array_equal(y, ref)


def test_zero_scale_gives_the_base_projection():
    ids = np.random.default_rng(3).integers(-1, 3, 9).astype(np.int32)
    p = synth.make_dense("pin", 4, ids, 32, [24], [16, 32, 8], y_base="zero")
    W = bits(np.random.default_rng(4).standard_normal((24, 32)))
    y, _ = oracle.lora_linear(p.ids, p.x, W, p.A, p.B, p.ranks, [0.0] * 3, p.slice_n, p.n_a)
    y_none, _ = oracle.lora_linear(np.full(p.M, -1, np.int32), p.x, W, p.A, p.B, p.ranks, p.scales, p.slice_n,
                                   p.n_a)
    assert np.array_equal(y, y_none)
