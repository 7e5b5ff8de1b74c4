"""lora_apply_static_scratch: one step with no device memory from the caller.

This entry point serves callers that cannot allocate device memory (they can
only hand over their inputs and outputs): it keeps the segment table and the
hand-off scratch in a fixed array inside the library.  Its output must match
the CPU oracle, and the workspace-based path (lora_build_segments +
lora_apply), within the tolerance every GPU test here uses, on consecutive
calls that reuse the array; several calls issued back to back on one stream
(programmatic dependent launch on, no host synchronisation between them) must
each come out right; calls past the documented limits must return their
status code before launching anything.  This file is collected last so a
failure here cannot hide any other test.
"""
import numpy as np
import pytest
import torch

from segmented_rank_gemm_lora_gb300 import lora, synth
from gpu_util import check_close, dev_bf16, host_f64, oracle_dense, pack_dense, run_dense

pytestmark = pytest.mark.gpu

STATIC_PARTIAL_FLOATS = 1 << 23   # the fixed array's hand-off partials (include/lora.h)
MIN_KC = 64                       # the shortest K-chunk the engine cuts


def static_apply(table, ids, x, y, M=None):
    lib = lora.load()
    M = int(ids.numel()) if M is None else M
    return lib.lora_apply_static_scratch(table.handle, ids.data_ptr(), M, x.data_ptr(), x.stride(0),
                                         y.data_ptr(), y.stride(0), torch.cuda.current_stream().cuda_stream)


def static_need(M, R, K, L):
    """Partial floats the documented limit charges a call of M tokens."""
    return M * R * (-(-K // MIN_KC) + 1) + 64 * R * min(M, L)


def problem(name):
    if name == "decode":
        return synth.decode(1, y_base="random")
    if name == "decode_delta_only":
        return synth.decode(7, y_base="zero")
    if name == "tiny":
        return synth.tiny(0, y_base="xw")
    if name == "prefill":
        return synth.prefill(2, y_base="random")
    # 128 tokens of the stacked batch keep the three-slice QKV within the fixed array
    q = synth.stacked("qkv", y_base="zero")
    p = synth.DenseProblem(**{**q.__dict__})
    p.ids, p.x, p.y_base, p.M = q.ids[384:512], q.x[384:512], q.y_base[384:512], 128
    return p


@pytest.mark.parametrize("name", ["decode", "decode_delta_only", "tiny", "prefill", "stacked_qkv_128"])
def test_static_scratch_matches_the_oracle_and_the_workspace_path_on_consecutive_calls(name):
    p = problem(name)
    table = pack_dense(p)
    y_ws, _, ws = run_dense(p, table=table)
    assert lora.lora_get_status(ws) == lora.LORA_OK
    ref = oracle_dense(p)
    ws_out = host_f64(y_ws)
    check_close(ws_out, ref, "%s workspace path" % name)
    ids = torch.from_numpy(p.ids).cuda()
    x = dev_bf16(p.x)
    for call in range(2):
        y = dev_bf16(p.y_base)
        assert static_apply(table, ids, x, y) == lora.LORA_OK
        torch.cuda.synchronize()
        got = host_f64(y)
        check_close(got, ref, "%s call %d against the oracle" % (name, call))
        check_close(got, ws_out, "%s call %d against the workspace path" % (name, call))
    table.destroy()


def test_static_scratch_calls_back_to_back_with_pdl():
    """Four calls with different id maps (and sizes) on one stream, no host sync between them, PDL on."""
    old = lora.lora_get_option(lora.LORA_OPT_PDL)
    lora.lora_set_option(lora.LORA_OPT_PDL, 1)
    try:
        base = synth.decode(1, y_base="random")
        table = pack_dense(base)
        rng = np.random.default_rng(11)
        cases = []
        for M in (32, 9, 200, 32):   # decode-sized and larger calls alternate between the engine's set-ups
            rows = rng.integers(0, base.M, M)
            p = synth.DenseProblem(**{**base.__dict__})
            p.ids = rng.integers(-1, base.L, M).astype(np.int32)
            p.x = np.ascontiguousarray(base.x[rows])
            p.y_base = np.ascontiguousarray(base.y_base[rows])
            p.M = M
            cases.append(p)
        dev = [(torch.from_numpy(p.ids).cuda(), dev_bf16(p.x), dev_bf16(p.y_base)) for p in cases]
        torch.cuda.synchronize()
        for ids, x, y in dev:
            assert static_apply(table, ids, x, y) == lora.LORA_OK
        torch.cuda.synchronize()
        for k, (p, (_, _, y)) in enumerate(zip(cases, dev)):
            check_close(host_f64(y), oracle_dense(p), "back-to-back call %d (M=%d)" % (k, p.M))
        table.destroy()
    finally:
        lora.lora_set_option(lora.LORA_OPT_PDL, old)


def test_static_scratch_at_its_partial_limit():
    """The largest call the documented limit admits runs and matches the oracle; one token more is refused."""
    p = synth.decode(1, y_base="random")   # K = 4096, ranks up to 64: the bound binds near 2000 tokens
    R = max(p.n_a * ((r + 15) // 16 * 16) for r in p.ranks)
    M = 1
    while static_need(M + 1, R, p.K, p.L) <= STATIC_PARTIAL_FLOATS:
        M += 1
    assert M < 4096, "the limit under test is the partial bound, not the token cap"
    rng = np.random.default_rng(5)
    q = synth.DenseProblem(**{**p.__dict__})
    q.ids = rng.integers(-1, p.L, M).astype(np.int32)
    rows = rng.integers(0, p.M, M)
    q.x = np.ascontiguousarray(p.x[rows])
    q.y_base = np.ascontiguousarray(p.y_base[rows])
    q.M = M
    table = pack_dense(q)
    ids = torch.from_numpy(q.ids).cuda()
    x = dev_bf16(q.x)
    y = dev_bf16(q.y_base)
    assert static_apply(table, ids, x, y) == lora.LORA_OK
    torch.cuda.synchronize()
    check_close(host_f64(y), oracle_dense(q), "M=%d at the limit" % M)
    ids1 = torch.zeros(M + 1, dtype=torch.int32, device="cuda")
    x1 = torch.zeros(M + 1, q.K, dtype=torch.bfloat16, device="cuda")
    y1 = torch.zeros(M + 1, q.N, dtype=torch.bfloat16, device="cuda")
    assert static_apply(table, ids1, x1, y1) == lora.LORA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y1 == 0).all())
    table.destroy()


def test_static_scratch_rejects_oversized_calls():
    p = synth.decode(1, y_base="random")
    table = pack_dense(p)
    ids = torch.zeros(4097, dtype=torch.int32, device="cuda")
    x = torch.zeros(4097, p.K, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(4097, p.N, dtype=torch.bfloat16, device="cuda")
    assert static_apply(table, ids, x, y) == lora.LORA_ERR_WORKSPACE
    assert bool((y == 0).all())
    table.destroy()


def test_static_scratch_rejects_tables_past_the_build_key_limit():
    """16000 adapters (16001 keys with "none") is past the segment build's limit: refused, nothing launched."""
    L, K, N, r = 16000, 8, 8, 16
    A = [torch.zeros(r, K, dtype=torch.bfloat16, device="cuda")] * L
    B = [torch.zeros(N, r, dtype=torch.bfloat16, device="cuda")] * L
    table = lora.lora_pack_weights(A, B, [r] * L, [1.0] * L, K, [N], 1)
    torch.cuda.synchronize()
    ids = torch.zeros(40, dtype=torch.int32, device="cuda")
    x = torch.zeros(40, K, dtype=torch.bfloat16, device="cuda")
    y = torch.ones(40, N, dtype=torch.bfloat16, device="cuda")
    assert static_apply(table, ids, x, y) == lora.LORA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((y == 1).all())
    table.destroy()
