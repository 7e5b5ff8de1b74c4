"""Pins of the oracle's embedding LoRA ("[SGLang] LoRA Layers", VocabParallelEmbeddingWithLoRA: A used as an
embedding lookup over the vocabulary, B as a plain matmul), against values fixed independently of it:

  * the lookup is the dense shrink of a one-hot row: with x[t] the one-hot row of vocab[t] (K = V), the
    separately pinned dense delta (lora_apply) gives the same numbers;
  * a worked example small enough to check by hand;
  * out-of-range vocabulary or adapter ids leave the row at y_base and are counted.
"""
import numpy as np

import oracle
from segmented_rank_gemm_lora_gb300 import synth


def bits(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_lookup_equals_the_dense_delta_of_one_hot_rows():
    rng = np.random.default_rng(0)
    V, N, M = 96, 40, 23
    ranks = [16, 32, 8]
    ids = rng.integers(-1, 3, M).astype(np.int32)
    vocab = rng.integers(0, V, M).astype(np.int32)
    A = [bits(rng.standard_normal((r, V))) for r in ranks]
    B = [bits(rng.standard_normal((N, r))) for r in ranks]
    yb = bits(rng.standard_normal((M, N)))
    y, bad = oracle.embedding_apply(ids, vocab, yb, A, B, ranks, [2.0, 0.5, 1.0])
    x = np.zeros((M, V), np.float32)
    x[np.arange(M), vocab] = 1.0
    ref, bad2 = oracle.lora_apply(ids, bits(x), yb, A, B, ranks, [2.0, 0.5, 1.0], [N], 1)
    assert bad == bad2 == 0
    assert np.array_equal(y, ref)


def test_worked_example():
    # one adapter of rank 2 over a vocabulary of 3: A = [[1, 2, 3], [4, 5, 6]], B = [[1, 0], [0, 1], [1, 1]]
    A = [bits([[1, 2, 3], [4, 5, 6]])]
    B = [bits([[1, 0], [0, 1], [1, 1]])]
    yb = bits([[10, 20, 30], [0, 0, 0]])
    y, bad = oracle.embedding_apply(np.array([0, 0], np.int32), np.array([1, 2], np.int32), yb, A, B, [2], [1.0])
    # token 0: S = A[:, 1] = (2, 5) -> B S = (2, 5, 7); token 1: S = (3, 6) -> (3, 6, 9)
    assert bad == 0
    assert np.array_equal(y, [[12, 25, 37], [3, 6, 9]])


def test_out_of_range_ids_keep_the_base_row():
    A = [bits(np.ones((16, 5)))]
    B = [bits(np.ones((4, 16)))]
    yb = bits(np.arange(12).reshape(3, 4))
    y, bad = oracle.embedding_apply(np.array([0, 3, -1], np.int32), np.array([7, 0, 1], np.int32), yb, A, B, [16], [1.0])
    assert bad == 2
    assert np.array_equal(y, synth.bf16_bits_to_f32(yb).astype(np.float64))
