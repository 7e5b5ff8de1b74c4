"""lora_apply on the GPU vs the CPU oracle.

Gates: max|y - y_ref| <= 1e-2 max|y_ref| on every config, plus the same gate
on the delta alone (y_base = 0), because y_base dominates |y|; rows of tokens
without an adapter bit-identical; integer inputs bit-exact; results invariant
(bitwise) to token order and repeatable.
"""
import numpy as np
import pytest
import torch

from segmented_rank_gemm_lora_gb300 import lora, synth
from gpu_util import PATHS, check_close, dev_bf16, forced_path, host_bits, host_f64, oracle_dense, pack_dense, padded, run_dense

pytestmark = pytest.mark.gpu


def problems():
    yield "tiny", lambda base: synth.tiny(0, y_base="xw" if base else "zero")
    yield "decode", lambda base: synth.decode(1, y_base="random" if base else "zero")
    yield "prefill", lambda base: synth.prefill(2, y_base="random" if base else "zero")
    yield "stacked_qkv", lambda base: synth.stacked("qkv", y_base="random" if base else "zero")
    yield "stacked_gate_up", lambda base: synth.stacked("gate_up", y_base="random" if base else "zero")
    yield "stacked_down", lambda base: synth.stacked("down", y_base="random" if base else "zero")
    yield "ragged", lambda base: synth.make_dense("ragged", 9, np.random.default_rng(9).integers(-1, 3, 37)
                                                  .astype(np.int32), 200, [72, 136], [8, 24, 40],
                                                  y_base="random" if base else "zero")
    yield "shared_a", lambda base: synth.make_dense("shared", 10, np.random.default_rng(10).integers(-1, 4, 50)
                                                    .astype(np.int32), 264, [128, 128], [16, 32, 8, 64], n_a=1,
                                                    y_base="random" if base else "zero")


@pytest.mark.parametrize("name,make", list(problems()), ids=[n for n, _ in problems()])
def test_apply_matches_oracle(name, make):
    """Every path (auto, small tiles forced, 128-row tensor-core tiles forced) against the oracle, full
    output and delta only."""
    for base in (True, False):
        p = make(base)
        ref = oracle_dense(p)
        table = pack_dense(p)
        ws = lora.Workspace(max(p.M, 1), p.L)
        for path in PATHS:
            with forced_path(path):
                y, _, _ = run_dense(p, table=table, ws=ws)
            assert lora.lora_get_status(ws) == lora.LORA_OK
            check_close(host_f64(y), ref, "%s base=%s path=%d" % (name, base, path))
            none = p.ids < 0
            assert np.array_equal(host_bits(y)[none], p.y_base[none])
        table.destroy()


def test_canary_columns_and_rows_untouched():
    p = synth.decode(3, y_base="random")
    y, table, ws = run_dense(p, x_extra=8, y_extra=24)
    yb = host_bits(y)
    assert (yb[:, p.N:] == 0x7FC1).all()
    check_close(synth.bf16_bits_to_f32(yb[:, :p.N]).astype(np.float64), oracle_dense(p))


@pytest.mark.parametrize("slices,n_a", [([96], None), ([64, 32, 32], None), ([48, 48], 1)])
def test_integer_inputs_are_bit_exact(slices, n_a):
    ids = np.random.default_rng(4).integers(-1, 5, 90).astype(np.int32)
    ids[:20] = 2   # one segment large enough to span several row tiles
    p = synth.make_dense_int(12, ids, 384, slices, [8, 16, 32, 64, 40], n_a=n_a)
    ref = oracle_dense(p)
    assert np.abs(ref).max() <= 256 and np.array_equal(ref, np.round(ref))
    for path in PATHS:
        with forced_path(path):
            y, _, ws = run_dense(p)
        assert lora.lora_get_status(ws) == lora.LORA_OK
        assert np.array_equal(host_f64(y), ref), "path %d" % path


def test_integer_inputs_bit_exact_with_ragged_k_on_tensor_cores():
    # K = 200 ends on an odd 8-wide K-group: the zero-filled half step must add nothing
    ids = np.repeat(np.arange(3, dtype=np.int32), [70, 130, 5])
    p = synth.make_dense_int(13, ids, 200, [136, 72], [16, 48, 8])
    ref = oracle_dense(p)
    assert np.abs(ref).max() <= 256
    for path in PATHS:
        with forced_path(path):
            y, _, ws = run_dense(p)
        assert lora.lora_get_status(ws) == lora.LORA_OK
        assert np.array_equal(host_f64(y), ref), "path %d" % path


@pytest.mark.parametrize("path", PATHS)
def test_token_order_invariance_is_bitwise(path):
    p = synth.prefill(2, y_base="random")
    with forced_path(path):
        y, table, ws = run_dense(p)
        perm = np.random.default_rng(1).permutation(p.M)
        q = synth.DenseProblem(**{**p.__dict__})
        q.ids, q.x, q.y_base = p.ids[perm], p.x[perm], p.y_base[perm]
        yq, _, _ = run_dense(q, table=table, ws=ws)
    assert np.array_equal(host_bits(yq), host_bits(y)[perm])


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_repeatable(name):
    p = synth.decode(1, y_base="random") if name == "decode" else synth.prefill(2, y_base="random")
    y1, table, ws = run_dense(p)
    y2, _, _ = run_dense(p, table=table, ws=ws)
    y3, _, _ = run_dense(p, table=table, ws=ws, build=False)   # second apply on the same segment table
    assert np.array_equal(host_bits(y1), host_bits(y2))
    assert np.array_equal(host_bits(y1), host_bits(y3))


def test_all_none_and_empty_batches_are_no_ops():
    p = synth.decode(1, y_base="random")
    p.ids[:] = -1
    y, table, ws = run_dense(p)
    assert lora.lora_get_status(ws) == lora.LORA_OK
    assert np.array_equal(host_bits(y), p.y_base)
    ws0 = lora.Workspace(4, p.L)
    lora.lora_build_segments(ws0, torch.zeros(0, dtype=torch.int32, device="cuda"))
    x = torch.ones(1, p.K, dtype=torch.bfloat16, device="cuda")
    yy = torch.ones(1, p.N, dtype=torch.bfloat16, device="cuda")
    lora.lora_apply(table, ws0, x, yy)       # no segments: the launch does nothing
    assert lora.lora_get_status(ws0) == lora.LORA_OK
    assert bool((yy == 1).all())


def test_bad_ids_leave_rows_and_report():
    p = synth.decode(6, y_base="random")
    p.ids[[0, 5]] = [25, -4]
    y, table, ws = run_dense(p)
    assert lora.lora_get_status(ws) == lora.LORA_ERR_BAD_ADAPTER_ID
    yb = host_bits(y)
    assert np.array_equal(yb[[0, 5]], p.y_base[[0, 5]])
    q = synth.DenseProblem(**{**p.__dict__})
    ref = oracle_dense(q)
    check_close(synth.bf16_bits_to_f32(yb).astype(np.float64), ref)


def test_one_workspace_serves_every_projection():
    ids = synth.ids_stacked(3)
    ws = lora.Workspace(len(ids), 32)
    lora.lora_build_segments(ws, torch.from_numpy(ids).cuda())
    for proj in ("qkv", "gate_up", "down"):
        p = synth.stacked(proj, y_base="zero")
        y, table, _ = run_dense(p, ws=ws, build=False)
        assert lora.lora_get_status(ws) == lora.LORA_OK
        check_close(host_f64(y), oracle_dense(p), proj)
        table.destroy()


def test_stored_ranks_follow_the_padding_rule():
    p = synth.make_dense("r", 1, np.zeros(4, np.int32), 64, [64], [16, 20, 8, 33, 64])
    table = pack_dense(p)
    assert [table.stored_rank(i) for i in range(5)] == [16, 32, 16, 48, 64]
    info = table.info()
    assert info.num_rank_groups == 4 and info.L == 5 and info.N == 64


@pytest.mark.parametrize("path", PATHS)
def test_handoff_wait_times_out_cleanly_and_recovers(path):
    p = synth.decode(1, y_base="random")
    table = pack_dense(p)
    ws = lora.Workspace(p.M, p.L)
    old = lora.lora_get_option(lora.LORA_OPT_WAIT_TIMEOUT_NS)
    try:
        lora.lora_set_option(lora.LORA_OPT_WAIT_TIMEOUT_NS, 2_000_000)
        lora.lora_set_option(lora.LORA_OPT_TEST_WITHHOLD_HANDOFF, 1)
        with forced_path(path):
            y, _, _ = run_dense(p, table=table, ws=ws)
        assert lora.lora_get_status(ws) == lora.LORA_ERR_TIMEOUT
        assert np.array_equal(host_bits(y), p.y_base)      # nothing was added
    finally:
        lora.lora_set_option(lora.LORA_OPT_TEST_WITHHOLD_HANDOFF, 0)
        lora.lora_set_option(lora.LORA_OPT_WAIT_TIMEOUT_NS, old)
    with forced_path(path):
        y, _, _ = run_dense(p, table=table, ws=ws)               # rebuild resets the scratch
    assert lora.lora_get_status(ws) == lora.LORA_OK
    check_close(host_f64(y), oracle_dense(p))


def test_graph_capture_replays():
    p = synth.decode(2, y_base="random")
    table = pack_dense(p)
    ws = lora.Workspace(p.M, p.L)
    ids = torch.from_numpy(p.ids).cuda()
    x = dev_bf16(p.x)
    y = dev_bf16(p.y_base)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        lora.lora_build_segments(ws, ids)
        lora.lora_apply(table, ws, x, y)
    y.copy_(dev_bf16(p.y_base))
    g.replay()
    torch.cuda.synchronize()
    assert lora.lora_get_status(ws) == lora.LORA_OK
    check_close(host_f64(y), oracle_dense(p))


def test_widest_a_block_every_path():
    """Four stacked slices of rank up to 64 (an A block of 256 rows, the widest the table stores): groups
    small and large, on every path, against the oracle."""
    rng = np.random.default_rng(21)
    ids = np.concatenate([np.full(n, a, np.int32) for a, n in [(0, 3), (1, 40), (2, 150), (3, 17), (4, 9)]])
    ids = np.concatenate([ids, rng.integers(-1, 5, 30).astype(np.int32)])
    p = synth.make_dense("widest", 21, ids, 1024, [256, 128, 384, 136], [64, 48, 16, 64, 32], y_base="random")
    ref = oracle_dense(p)
    table = pack_dense(p)
    ws = lora.Workspace(p.M, p.L)
    for path in PATHS:
        with forced_path(path):
            y, _, _ = run_dense(p, table=table, ws=ws)
        assert lora.lora_get_status(ws) == lora.LORA_OK
        check_close(host_f64(y), ref, "widest path=%d" % path)
    table.destroy()


def test_large_batch_sampled_rows():
    """A 4096-token batch (prefill-like runs over 24 adapters, K = N = 4096) checked on 96 sampled rows:
    a token's delta depends on its own row only, so the oracle runs on the sample."""
    rng = np.random.default_rng(22)
    lens = synth.power_law_lengths(rng, 64, 16, 512)
    ids = np.concatenate([np.full(int(n), j % 24, np.int32) for j, n in enumerate(lens)])[:4096]
    ids = np.concatenate([ids, rng.integers(-1, 24, 4096 - len(ids)).astype(np.int32)])
    assert len(ids) == 4096
    p = synth.make_dense("large", 22, ids, 4096, [4096], synth.cycle_ranks(24), y_base="random")
    y, table, ws = run_dense(p)
    assert lora.lora_get_status(ws) == lora.LORA_OK
    rows = np.sort(rng.choice(4096, 96, replace=False))
    sub = synth.DenseProblem(**{**p.__dict__})
    sub.ids, sub.x, sub.y_base, sub.M = p.ids[rows], p.x[rows], p.y_base[rows], len(rows)
    check_close(host_f64(y)[rows], oracle_dense(sub), "large batch, sampled rows")
    table.destroy()


def test_back_to_back_steps_on_one_workspace_with_and_without_pdl():
    """Steps with different ids enqueued back to back on one workspace (no host sync between them): with
    programmatic dependent launches the next build may be scheduled while the previous apply still runs,
    so every kernel must wait before it touches the workspace.  The outputs equal those of plain stream
    order, bit for bit, eager and replayed from a CUDA graph."""
    base = synth.decode(11, y_base="random")
    probs = [base]
    for q in [synth.decode(12, y_base="random"), synth.decode(13, y_base="random"),
              synth.prefill(14, y_base="random")]:   # same weights, other batches
        r = synth.DenseProblem(**{**base.__dict__})
        r.ids, r.x, r.y_base, r.M = q.ids, q.x, q.y_base, q.M
        probs.append(r)
    L = base.L
    M = max(p.M for p in probs)
    table = pack_dense(base)
    ws = lora.Workspace(M, L)
    ids = [torch.from_numpy(p.ids).cuda() for p in probs]
    xs = [dev_bf16(p.x) for p in probs]

    def steps(ys):
        for k in range(3):
            for i, p in enumerate(probs):
                lora.lora_build_segments(ws, ids[i])
                lora.lora_apply(table, ws, xs[i], ys[3 * i + k])

    outs = {}
    old = lora.lora_get_option(lora.LORA_OPT_PDL)
    try:
        for pdl in (0, 1):
            lora.lora_set_option(lora.LORA_OPT_PDL, pdl)
            ys = [dev_bf16(p.y_base) for p in probs for _ in range(3)]
            steps(ys)
            torch.cuda.synchronize()
            assert lora.lora_get_status(ws) == lora.LORA_OK
            outs[pdl] = [host_bits(y) for y in ys]
        # graph capture with PDL on
        lora.lora_set_option(lora.LORA_OPT_PDL, 1)
        ys = [dev_bf16(p.y_base) for p in probs for _ in range(3)]
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            steps(ys)
        for i, p in enumerate(probs):
            for k in range(3):
                ys[3 * i + k].copy_(dev_bf16(p.y_base))
        g.replay()
        torch.cuda.synchronize()
        assert lora.lora_get_status(ws) == lora.LORA_OK
        outs["graph"] = [host_bits(y) for y in ys]
    finally:
        lora.lora_set_option(lora.LORA_OPT_PDL, old)
    for a, b, c in zip(outs[0], outs[1], outs["graph"]):
        assert np.array_equal(a, b) and np.array_equal(a, c)
    for i, p in enumerate(probs):
        check_close(synth.bf16_bits_to_f32(outs[1][3 * i]).astype(np.float64), oracle_dense(p), "step %d" % i)
    table.destroy()


def _fused_vs_separate(p, table, ws_a, ws_b):
    ids = torch.from_numpy(p.ids).cuda()
    x = dev_bf16(p.x)
    ya, yb = dev_bf16(p.y_base), dev_bf16(p.y_base)
    lora.lora_build_and_apply(table, ws_a, ids, x, ya)
    lora.lora_build_segments(ws_b, ids)
    lora.lora_apply(table, ws_b, x, yb)
    torch.cuda.synchronize()
    return ya, yb


@pytest.mark.parametrize("case", ["decode", "one_token", "all_none", "bad_ids", "ragged_small", "stacked_16"])
def test_build_and_apply_equals_the_two_calls(case):
    """lora_build_and_apply (one launch for decode-sized batches) against lora_build_segments + lora_apply:
    the same output bits, the same segment table left in the workspace, the same status; a later
    lora_apply on that workspace reads the table it left."""
    if case == "stacked_16":
        q = synth.stacked("qkv", y_base="random")    # A blocks of 192 rows: one launch only up to 16 tokens
        p = synth.DenseProblem(**{**q.__dict__})
        p.ids, p.x, p.y_base, p.M = q.ids[:16].copy(), q.x[:16], q.y_base[:16], 16
    else:
        p = synth.decode(31, y_base="random")
        if case == "one_token":
            p.ids, p.x, p.y_base, p.M = p.ids[:1].copy(), p.x[:1], p.y_base[:1], 1
            p.ids[0] = 3
        elif case == "all_none":
            p.ids[:] = -1
        elif case == "bad_ids":
            p.ids[[1, 7]] = [p.L + 3, -9]
        elif case == "ragged_small":
            p.ids[:] = np.random.default_rng(5).integers(0, 3, p.M)   # a few groups of up to ~16 rows
    table = pack_dense(p)
    for path in PATHS:
        ws_a, ws_b = lora.Workspace(p.M, p.L), lora.Workspace(p.M, p.L)
        with forced_path(path):
            ya, yb = _fused_vs_separate(p, table, ws_a, ws_b)
            assert lora.lora_get_status(ws_a) == lora.lora_get_status(ws_b), "path %d" % path
            assert np.array_equal(host_bits(ya), host_bits(yb)), "path %d" % path
            sa, sb = ws_a.read_segments(), ws_b.read_segments()
            for k in ("M", "num_segments", "num_valid"):
                assert sa[k] == sb[k]
            assert np.array_equal(sa["perm"], sb["perm"]) and np.array_equal(sa["segments"], sb["segments"])
            # a later apply on the fused call's workspace uses the table it left
            yc = dev_bf16(p.y_base)
            lora.lora_apply(table, ws_a, dev_bf16(p.x), yc)
            torch.cuda.synchronize()
            assert np.array_equal(host_bits(yc), host_bits(yb)), "path %d" % path
    if case != "bad_ids":
        check_close(host_f64(ya), oracle_dense(p))
    table.destroy()


def test_build_and_apply_back_to_back_in_a_graph():
    """Fused decode steps with different ids, back to back on one workspace, eager and replayed from a
    CUDA graph: each equals its own two-call reference."""
    base = synth.decode(41, y_base="random")
    probs = [base]
    for sd in (42, 43):
        q = synth.decode(sd, y_base="random")
        r = synth.DenseProblem(**{**base.__dict__})
        r.ids, r.x, r.y_base = q.ids, q.x, q.y_base
        probs.append(r)
    table = pack_dense(base)
    ws = lora.Workspace(base.M, base.L)
    ids = [torch.from_numpy(p.ids).cuda() for p in probs]
    xs = [dev_bf16(p.x) for p in probs]
    ref = []
    for i, p in enumerate(probs):
        y = dev_bf16(p.y_base)
        w2 = lora.Workspace(p.M, p.L)
        lora.lora_build_segments(w2, ids[i])
        lora.lora_apply(table, w2, xs[i], y)
        ref.append(host_bits(y))
    ys = [dev_bf16(p.y_base) for p in probs]
    for i in range(len(probs)):
        lora.lora_build_and_apply(table, ws, ids[i], xs[i], ys[i])
    torch.cuda.synchronize()
    assert all(np.array_equal(host_bits(ys[i]), ref[i]) for i in range(len(probs)))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(len(probs)):
            lora.lora_build_and_apply(table, ws, ids[i], xs[i], ys[i])
    for i, p in enumerate(probs):
        ys[i].copy_(dev_bf16(p.y_base))
    g.replay()
    torch.cuda.synchronize()
    assert lora.lora_get_status(ws) == lora.LORA_OK
    assert all(np.array_equal(host_bits(ys[i]), ref[i]) for i in range(len(probs)))
    table.destroy()


@pytest.mark.parametrize("case", ["prefill_two_calls", "few_adapters_padded_ranks", "strided_rows"])
def test_build_and_apply_more_shapes(case):
    """lora_build_and_apply beyond the plain decode batch: a prefill batch (more than 32 tokens, so the
    two calls it stands for), fewer adapters than tokens with ranks that need padding (20, 40), and x / y
    with row strides past K and N (canary columns stay untouched)."""
    x_extra = y_extra = 0
    if case == "prefill_two_calls":
        p = synth.prefill(15, y_base="random")
    elif case == "few_adapters_padded_ranks":
        ids = np.random.default_rng(16).integers(-1, 4, 32).astype(np.int32)
        p = synth.make_dense("padded", 16, ids, 512, [264], [20, 40, 8, 64], y_base="random")
    else:
        p = synth.decode(17, y_base="random")
        x_extra, y_extra = 16, 24
    table = pack_dense(p)
    ws = lora.Workspace(p.M, p.L)
    ids = torch.from_numpy(p.ids).cuda()
    x = dev_bf16(padded(p.x, x_extra))
    y = dev_bf16(padded(p.y_base, y_extra))
    lora.lora_build_and_apply(table, ws, ids, x[:, :p.K] if x_extra else x, y[:, :p.N] if y_extra else y)
    torch.cuda.synchronize()
    assert lora.lora_get_status(ws) == lora.LORA_OK
    yb = host_bits(y)
    if y_extra:
        assert (yb[:, p.N:] == 0x7FC1).all()
    check_close(synth.bf16_bits_to_f32(yb[:, :p.N]).astype(np.float64), oracle_dense(p), case)
    none = p.ids < 0
    assert np.array_equal(yb[:, :p.N][none], p.y_base[none])
    seg = ws.read_segments()
    ws2 = lora.Workspace(p.M, p.L)
    lora.lora_build_segments(ws2, ids)
    ref = ws2.read_segments()
    assert np.array_equal(seg["perm"], ref["perm"]) and np.array_equal(seg["segments"], ref["segments"])
    table.destroy()
