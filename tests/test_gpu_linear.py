"""lora_linear (the base projection and the LoRA delta in one kernel) on the GPU against the oracle.

Every case checks: y against the oracle's LoRA linear layer (x W^T plus the delta, fp64); the rows of
tokens without an adapter against a plain x W^T computed here; the delta alone (W = 0) against the
oracle's delta; integer inputs bit for bit.  Shapes cover token tiles of one and of several 128-row
tiles per segment, a tail of tokens without an adapter, K with a last 8-column step, output slices
whose last 128-column tile is partial, and the widest A block (four slices of rank 64).
"""
import numpy as np
import pytest
import torch

import oracle
from segmented_rank_gemm_lora_gb300 import lora, synth
from gpu_util import check_close, dev_bf16, host_bits, host_f64, pack_dense

pytestmark = pytest.mark.gpu


def weight(seed, N, K):
    rng = np.random.default_rng(seed)
    return synth.f32_to_bf16_bits((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32))


def run_linear(p, W, table=None):
    table = table or pack_dense(p)
    ws = lora.Workspace(max(p.M, 1), p.L)
    lora.lora_build_segments(ws, torch.from_numpy(p.ids).cuda())
    y = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lora.lora_linear(table, ws, dev_bf16(p.x), dev_bf16(W), y)
    assert lora.lora_get_status(ws) == lora.LORA_OK
    return y, table


CASES = {
    # name: (ids maker, K, slices, ranks, n_a)
    "prefill_like": (lambda r: np.concatenate([np.full(n, a, np.int32) for a, n in [(0, 150), (1, 40), (2, 300)]]
                                              + [r.integers(-1, 3, 60).astype(np.int32)]), 512, [256, 128],
                     [16, 32, 64], None),
    "decode_like": (lambda r: r.integers(-1, 16, 32).astype(np.int32), 1024, [1024], synth.cycle_ranks(16), None),
    "ragged_k": (lambda r: r.integers(-1, 4, 70).astype(np.int32), 200, [136, 72], [8, 24, 40, 64], None),
    "widest_a": (lambda r: r.integers(-1, 3, 140).astype(np.int32), 256, [128, 128, 128, 136], [64, 48, 16], None),
    "shared_a": (lambda r: r.integers(-1, 3, 90).astype(np.int32), 264, [128, 128], [16, 32, 64], 1),
    "no_adapter_only": (lambda r: np.full(200, -1, np.int32), 384, [256], [16, 32], None),
}


@pytest.mark.parametrize("name", list(CASES))
def test_linear_matches_the_oracle(name):
    make_ids, K, slices, ranks, n_a = CASES[name]
    rng = np.random.default_rng(sum(name.encode()))
    p = synth.make_dense(name, 31, make_ids(rng), K, slices, ranks, n_a=n_a, y_base="zero")
    W = weight(7, p.N, p.K)
    y, table = run_linear(p, W)
    got = host_f64(y)
    ref, bad = oracle.lora_linear(p.ids, p.x, W, p.A, p.B, p.ranks, p.scales, p.slice_n, p.n_a)
    assert bad == 0
    check_close(got, ref, name)
    # tokens without an adapter: the plain projection, computed here
    none = p.ids < 0
    if none.any():
        base = synth.bf16_bits_to_f32(p.x[none]).astype(np.float64) @ synth.bf16_bits_to_f32(W).astype(np.float64).T
        check_close(got[none], base, name + " rows without an adapter")
    # the delta alone (W = 0) against the oracle's delta
    if (~none).any():
        yd, _ = run_linear(p, np.zeros_like(W), table)
        delta, _ = oracle.lora_apply(p.ids, p.x, np.zeros((p.M, p.N), np.uint16), p.A, p.B, p.ranks, p.scales,
                                     p.slice_n, p.n_a)
        check_close(host_f64(yd), delta, name + " delta alone")
        assert np.array_equal(host_bits(yd)[none], np.zeros((int(none.sum()), p.N), np.uint16))
    table.destroy()


@pytest.mark.parametrize("K", [192, 200])
def test_linear_integer_inputs_are_bit_exact(K):
    ids = np.random.default_rng(K).integers(-1, 4, 150).astype(np.int32)
    ids[:40] = 1
    p = synth.make_dense_int(15, ids, K, [136, 128], [8, 16, 32, 64])
    rng = np.random.default_rng(K + 1)
    Wf = rng.integers(-1, 2, (p.N, K)).astype(np.float32) * (rng.random((p.N, K)) < 0.05)
    W = synth.f32_to_bf16_bits(Wf)
    ref, _ = oracle.lora_linear(p.ids, p.x, W, p.A, p.B, p.ranks, p.scales, p.slice_n, p.n_a)
    assert np.abs(ref).max() <= 256 and np.array_equal(ref, np.round(ref))
    y, table = run_linear(p, W)
    assert np.array_equal(host_f64(y), ref)
    table.destroy()


def test_linear_repeatable_and_token_order_invariant():
    ids = np.random.default_rng(3).integers(-1, 5, 260).astype(np.int32)
    p = synth.make_dense("order", 32, ids, 320, [384], [16, 32, 64, 48, 16], y_base="zero")
    W = weight(8, p.N, p.K)
    y1, table = run_linear(p, W)
    y2, _ = run_linear(p, W, table)
    assert np.array_equal(host_bits(y1), host_bits(y2))
    perm = np.random.default_rng(4).permutation(p.M)
    q = synth.DenseProblem(**{**p.__dict__})
    q.ids, q.x = p.ids[perm], p.x[perm]
    yq, _ = run_linear(q, W, table)
    assert np.array_equal(host_bits(yq), host_bits(y1)[perm])
    table.destroy()
