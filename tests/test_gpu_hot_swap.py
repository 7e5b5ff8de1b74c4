"""lora_table_set_adapter: hot-swapping adapters of a live table ("vLLM-Ascend dynamic LoRA fused operator",
section 3.1, a per-rank-group device pool; section 4.3, replacing an adapter while steps run).

  * launches enqueued before a swap read the old adapter and launches after it the new one, with no host
    synchronisation in between (stream order), each matching the oracle on its own weights;
  * a swap may change the adapter's rank (16 -> 64 -> 32), on the streaming path and on the engine;
  * repeated swaps reuse pool blocks: the table's device bytes stop growing;
  * bad arguments are refused.
"""
import numpy as np
import pytest
import torch

from segmented_rank_gemm_lora_gb300 import lora, synth
from gpu_util import check_close, dev_bf16, forced_path, host_f64, oracle_dense, pack_dense

pytestmark = pytest.mark.gpu


def new_weights(p, seed, rank):
    rng = np.random.default_rng(seed)
    A = synth.f32_to_bf16_bits((rng.standard_normal((p.n_a * rank, p.K)) / np.sqrt(p.K)).astype(np.float32))
    B = synth.f32_to_bf16_bits((rng.standard_normal((p.N, rank)) / np.sqrt(rank)).astype(np.float32))
    return A, B


@pytest.mark.parametrize("M,path", [(32, 0), (300, 0), (300, 1)])
def test_swaps_take_effect_in_stream_order(M, path):
    rng = np.random.default_rng(M)
    ids = rng.integers(-1, 6, M).astype(np.int32)
    p = synth.make_dense("swap", 13, ids, 1024, [512, 256], [16, 32, 64, 16, 32, 64], y_base="random")
    table = pack_dense(p)
    ws = lora.Workspace(p.M, p.L)
    idd = torch.from_numpy(p.ids).cuda()
    x = dev_bf16(p.x)
    q = synth.DenseProblem(**{**p.__dict__})
    q.A, q.B, q.ranks, q.scales = list(p.A), list(p.B), list(p.ranks), list(p.scales)
    swaps = [(2, 13, 16, 1.5), (4, 14, 64, 2.0), (1, 15, 48, 0.5)]
    dev_new = []
    for index, seed, rank, scale in swaps:
        A, B = new_weights(p, seed, rank)
        q.A[index], q.B[index], q.ranks[index], q.scales[index] = A, B, rank, scale
        dev_new.append((index, dev_bf16(A), dev_bf16(B), rank, scale))
    with forced_path(path):
        y1, y2 = dev_bf16(p.y_base), dev_bf16(p.y_base)
        torch.cuda.synchronize()
        lora.lora_build_segments(ws, idd)
        lora.lora_apply(table, ws, x, y1)                  # enqueued before the swaps
        for index, A, B, rank, scale in dev_new:
            lora.lora_table_set_adapter(table, index, A, B, rank, scale)
        lora.lora_apply(table, ws, x, y2)                  # after them
        torch.cuda.synchronize()
    assert lora.lora_get_status(ws) == lora.LORA_OK
    check_close(host_f64(y1), oracle_dense(p), "before the swaps")
    check_close(host_f64(y2), oracle_dense(q), "after the swaps")
    assert table.stored_rank(4) == 64 and table.stored_rank(1) == 48
    table.destroy()


def test_repeated_swaps_reuse_pool_blocks():
    ids = np.random.default_rng(3).integers(-1, 4, 64).astype(np.int32)
    p = synth.make_dense("swap", 16, ids, 512, [384], [16, 32, 64, 16], y_base="random")
    table = pack_dense(p)
    ws = lora.Workspace(p.M, p.L)
    lora.lora_build_segments(ws, torch.from_numpy(p.ids).cuda())
    x = dev_bf16(p.x)
    q = synth.DenseProblem(**{**p.__dict__})
    q.A, q.B, q.ranks, q.scales = list(p.A), list(p.B), list(p.ranks), list(p.scales)
    sizes = []
    for k in range(12):
        rank = (16, 64)[k % 2]
        A, B = new_weights(p, 100 + k, rank)
        q.A[1], q.B[1], q.ranks[1] = A, B, rank
        lora.lora_table_set_adapter(table, 1, dev_bf16(A), dev_bf16(B), rank, q.scales[1])
        y = dev_bf16(p.y_base)
        lora.lora_apply(table, ws, x, y)
        torch.cuda.synchronize()
        check_close(host_f64(y), oracle_dense(q), "swap %d" % k)
        sizes.append(table.info().device_bytes)
    # at most one new chunk per stored rank: later swaps take blocks back from the pool
    assert sizes[-1] == sizes[3], sizes
    table.destroy()


def test_bad_swaps_are_refused():
    p = synth.decode(1, y_base="random")
    table = pack_dense(p)
    A, B = new_weights(p, 1, 16)
    for index, rank in [(-1, 16), (p.L, 16), (0, 0), (0, 65)]:
        with pytest.raises(lora.LoraError) as e:
            lora.lora_table_set_adapter(table, index, dev_bf16(A), dev_bf16(B), rank, 1.0)
        assert e.value.code == lora.LORA_ERR_INVALID_ARG
    table.destroy()
