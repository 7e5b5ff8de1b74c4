"""Embedding LoRA (lora_embedding_apply) and the LM-head LoRA (lora_apply over a vocabulary-wide table) on
the GPU against the oracle ("[SGLang] LoRA Layers", VocabParallelEmbeddingWithLoRA and
ParallelLMHeadWithLoRA).  Gates as everywhere: max|y - y_ref| <= 1e-2 max|y_ref|, on the full rows and on
the delta alone (y_base = 0); rows of tokens without an adapter bit-identical; out-of-range vocabulary ids
reported and their rows left unchanged."""
import numpy as np
import pytest
import torch

import oracle
from segmented_rank_gemm_lora_gb300 import lora, synth
from gpu_util import check_close, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu


def bits(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def embedding_problem(seed, ids, V, N, ranks, base):
    rng = np.random.default_rng(seed)
    M = len(ids)
    vocab = rng.integers(0, V, M).astype(np.int32)
    A = [bits(rng.standard_normal((r, V))) for r in ranks]
    B = [bits(rng.standard_normal((N, r)) / np.sqrt(r)) for r in ranks]
    yb = bits(rng.standard_normal((M, N)) * 4.0) if base else np.zeros((M, N), np.uint16)
    return ids.astype(np.int32), vocab, A, B, yb


def run_embedding(ids, vocab, A, B, yb, ranks, scales, V, N):
    table = lora.lora_pack_weights([dev_bf16(a) for a in A], [dev_bf16(b) for b in B], ranks, scales, V, [N], 1)
    ws = lora.Workspace(len(ids), len(ranks))
    lora.lora_build_segments(ws, torch.from_numpy(ids).cuda())
    y = dev_bf16(yb)
    lora.lora_embedding_apply(table, ws, torch.from_numpy(vocab).cuda(), y)
    status = lora.lora_get_status(ws)
    table.destroy()
    return y, status


@pytest.mark.parametrize("case", ["decode", "prefill"])
@pytest.mark.parametrize("base", [True, False])
def test_embedding_matches_the_oracle(case, base):
    rng = np.random.default_rng(5)
    if case == "decode":
        ids, V, N, ranks = rng.integers(-1, 20, 32), 32768, 4096, synth.cycle_ranks(20)
    else:
        ids = np.concatenate([np.full(n, a) for a, n in [(0, 70), (1, 5), (2, 200), (3, 33)]] + [rng.integers(-1, 4, 40)])
        V, N, ranks = 1024, 520, [16, 48, 64, 8]
    scales = [2.0] * len(ranks)
    ids, vocab, A, B, yb = embedding_problem(11, ids, V, N, ranks, base)
    y, status = run_embedding(ids, vocab, A, B, yb, ranks, scales, V, N)
    assert status == lora.LORA_OK
    ref, bad = oracle.embedding_apply(ids, vocab, yb, A, B, ranks, scales)
    assert bad == 0
    check_close(host_f64(y), ref, "%s base=%s" % (case, base))
    none = ids < 0
    assert np.array_equal(host_bits(y)[none], yb[none])


def test_out_of_range_vocabulary_ids_are_reported_and_left_alone():
    rng = np.random.default_rng(6)
    ids = rng.integers(0, 3, 40)
    ids, vocab, A, B, yb = embedding_problem(12, ids, 256, 256, [16, 32, 64], True)
    vocab[[3, 17]] = [256, -5]
    y, status = run_embedding(ids, vocab, A, B, yb, [16, 32, 64], [1.0] * 3, 256, 256)
    assert status == lora.LORA_ERR_BAD_ADAPTER_ID
    got = host_bits(y)
    assert np.array_equal(got[[3, 17]], yb[[3, 17]])
    ok = np.ones(len(ids), bool)
    ok[[3, 17]] = False
    ref, bad = oracle.embedding_apply(ids, vocab, yb, A, B, [16, 32, 64], [1.0] * 3)
    assert bad == 2
    check_close(synth.bf16_bits_to_f32(got[ok]).astype(np.float64), ref[ok])


def test_lm_head_lora_is_lora_apply_over_the_vocabulary():
    """ParallelLMHeadWithLoRA: logits += (hidden A^T) B^T with N = the vocabulary; under tensor parallelism
    B is cut by vocabulary rows, which is the same call on the shard's rows of B (and of the logits)."""
    rng = np.random.default_rng(7)
    H, V, ranks = 512, 8192, [16, 32, 64, 16]
    ids = rng.integers(-1, 4, 48).astype(np.int32)
    p = synth.make_dense("lm_head", 41, ids, H, [V], ranks, y_base="random")
    for lo, hi in [(0, V), (2048, 6144)]:
        B = [b[lo:hi] for b in p.B]
        table = lora.lora_pack_weights([dev_bf16(a) for a in p.A], [dev_bf16(b) for b in B], p.ranks, p.scales, H,
                                       [hi - lo], 1)
        ws = lora.Workspace(p.M, p.L)
        lora.lora_build_segments(ws, torch.from_numpy(p.ids).cuda())
        y = dev_bf16(np.ascontiguousarray(p.y_base[:, lo:hi]))
        lora.lora_apply(table, ws, dev_bf16(p.x), y)
        assert lora.lora_get_status(ws) == lora.LORA_OK
        ref, _ = oracle.lora_apply(p.ids, p.x, p.y_base, p.A, p.B, p.ranks, p.scales, [V], 1)
        check_close(host_f64(y), ref[:, lo:hi], "vocabulary rows %d..%d" % (lo, hi))
        table.destroy()
