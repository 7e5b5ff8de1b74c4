"""Pins for the dense oracle (CPU only).

Each test fixes the oracle's output by something other than the oracle:
the merged-weight identity W' = W + scale * B A ("vLLM-Ascend dynamic LoRA
fused operator", section 1.1), the -1 pass-through (section 3.4), token-order
invariance of the bucketed computation (section 2.3), the zero-padding rule
(section 4.3) and exact integer arithmetic.  ``test_pins_catch_planted_mistakes``
compiles altered copies of the oracle and checks that these pins reject them.
"""
import os
import subprocess
import ctypes

import numpy as np
import pytest

import oracle
from segmented_rank_gemm_lora_gb300 import synth

bf = synth.bf16_bits_to_f32


def merged_delta(p, ids=None):
    """x @ (scale_i * B_i A_i)^T per token, built from the merged weight matrix (float64)."""
    ids = p.ids if ids is None else ids
    x = bf(p.x).astype(np.float64)
    out = np.zeros((p.M, p.N))
    offs = np.concatenate([[0], np.cumsum(p.slice_n)])
    for i, r in enumerate(p.ranks):
        A = bf(p.A[i]).astype(np.float64)
        B = bf(p.B[i]).astype(np.float64)
        Wd = np.zeros((p.N, p.K))
        for s in range(len(p.slice_n)):
            sa = 0 if p.n_a == 1 else s
            Wd[offs[s]:offs[s + 1]] = p.scales[i] * (B[offs[s]:offs[s + 1]] @ A[sa * r:(sa + 1) * r])
        rows = np.nonzero(ids == i)[0]
        out[rows] = x[rows] @ Wd.T
    return out


def run(p, **kw):
    return oracle.lora_apply(p.ids, p.x, p.y_base, p.A, p.B, p.ranks, p.scales, p.slice_n, p.n_a, **kw)


SHAPES = [
    # (ids, K, slices, ranks, n_a)
    (np.array([0, 1, -1, 1, 0, 2, 2, -1, 0], np.int32), 24, [40], [8, 16, 4], None),
    (np.array([3, 0, 0, 2, 1, -1, 3, 3], np.int32), 32, [16, 8, 8], [8, 16, 8, 16], None),   # stacked, 3 blocks
    (np.array([1, 1, 0, 0, 1, 0], np.int32), 16, [24, 24], [16, 8], 1),                      # 2 slices share A
    (np.array([0], np.int32), 64, [64], [16], None),
]


@pytest.mark.parametrize("case", range(len(SHAPES)))
@pytest.mark.parametrize("base", ["zero", "random"])
def test_merged_weight_identity(case, base):
    ids, K, slices, ranks, n_a = SHAPES[case]
    p = synth.make_dense("pin", 100 + case, ids, K, slices, ranks, n_a=n_a, scale=1.75, y_base=base)
    p.scales = [1.75 + 0.25 * i for i in range(p.L)]
    y, bad = run(p)
    assert bad == 0
    ref = bf(p.y_base).astype(np.float64) + merged_delta(p)
    err = np.abs(y - ref).max()
    assert err <= 1e-12 * max(1.0, np.abs(ref).max()), err


def test_none_rows_and_bad_ids_pass_through_exactly():
    ids = np.array([0, -1, 5, 1, -2, -1, 1], np.int32)   # 5 and -2 are out of range for L=2
    p = synth.make_dense("pin", 7, ids, 32, [48], [8, 16], y_base="random")
    y, bad = run(p)
    assert bad == 2
    yb = bf(p.y_base).astype(np.float64)
    for t in (1, 2, 4, 5):
        assert np.array_equal(y[t], yb[t])
    for t in (0, 3, 6):
        assert not np.array_equal(y[t], yb[t])


def test_enabled_mask_behaves_like_none():
    ids = np.array([0, 1, 2, 1, 0], np.int32)
    p = synth.make_dense("pin", 8, ids, 16, [32], [8, 8, 16], y_base="random")
    en = np.array([1, 0, 1], np.uint8)
    y, _ = run(p, enabled=en)
    yb = bf(p.y_base).astype(np.float64)
    assert np.array_equal(y[1], yb[1]) and np.array_equal(y[3], yb[3])
    full, _ = run(p)
    for t in (0, 2, 4):
        assert np.array_equal(y[t], full[t])


def test_token_order_invariance():
    p = synth.tiny(seed=5, y_base="random")
    y, _ = run(p)
    perm = np.random.default_rng(0).permutation(p.M)
    q = synth.DenseProblem(**{**p.__dict__})
    q.ids, q.x, q.y_base = p.ids[perm], p.x[perm], p.y_base[perm]
    yq, _ = run(q)
    assert np.array_equal(yq, y[perm])


def test_zero_rank_padding_is_a_no_op():
    p = synth.make_dense("pin", 9, np.array([0, 1, 1, 0, -1, 1], np.int32), 40, [16, 24], [8, 12], y_base="random")
    y, _ = run(p)
    q = synth.DenseProblem(**{**p.__dict__})
    q.ranks, q.A, q.B = [], [], []
    for i, r in enumerate(p.ranks):
        rp = ((r + 15) // 16) * 16
        A = np.zeros((p.n_a * rp, p.K), np.uint16)
        for s in range(p.n_a):
            A[s * rp:s * rp + r] = p.A[i][s * r:(s + 1) * r]
        B = np.zeros((p.N, rp), np.uint16)
        B[:, :r] = p.B[i]
        q.ranks.append(rp)
        q.A.append(A)
        q.B.append(B)
    yq, _ = run(q)
    assert np.array_equal(yq, y)


def test_integer_problem_is_exact():
    ids = np.random.default_rng(3).integers(-1, 4, 40).astype(np.int32)
    p = synth.make_dense_int(11, ids, 128, [64, 32], [8, 16, 32, 16])
    y, _ = run(p)
    xi = bf(p.x).astype(np.int64)
    ref = bf(p.y_base).astype(np.int64).copy()
    offs = [0, 64, 96]
    for i, r in enumerate(p.ranks):
        A = bf(p.A[i]).astype(np.int64)
        B = bf(p.B[i]).astype(np.int64)
        for s in range(2):
            Wd = B[offs[s]:offs[s + 1]] @ A[s * r:(s + 1) * r]
            rows = ids == i
            ref[rows, offs[s]:offs[s + 1]] += xi[rows] @ Wd.T
    assert np.array_equal(y, ref.astype(np.float64))


# ----------------------------------------------------------------------------
# the pins above must reject plausible mistakes planted in a copy of the oracle
# ----------------------------------------------------------------------------
MUTANTS = {
    "drop_scale": ("y_out[(int64_t)t * N + n] += scale[i] * acc;", "y_out[(int64_t)t * N + n] += acc;"),
    "transposed_B": ("const uint16_t *brow = B[i] + (int64_t)n * r;", "const uint16_t *brow = B[i] + (int64_t)(n % r) * r;"),
    "always_first_block": ("int32_t sa = (n_a == 1) ? 0 : s;", "int32_t sa = 0;"),
    "skip_last_k": ("for (int32_t k = 0; k < K; ++k) acc += bf(x", "for (int32_t k = 0; k < K - 1; ++k) acc += bf(x"),
    "wrong_token_row": ("acc += bf(x[(int64_t)t * ldx + k])", "acc += bf(x[(int64_t)(t ^ 1) * ldx + k])"),
    "none_not_skipped": ("if (i == -1) continue;", "if (i == -1) i = 0;"),
}


def _compile_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "lora_oracle.c")).read()
    a, b = MUTANTS[name]
    assert a in src, name
    path = tmp_path / (name + ".c")
    path.write_text(src.replace(a, b))
    so = tmp_path / (name + ".so")
    subprocess.run(["gcc", "-std=c99", "-O1", "-ffp-contract=off", "-shared", "-fPIC", "-o", str(so), str(path)],
                   check=True)
    lib = ctypes.CDLL(str(so))
    lib.oracle_lora_apply.restype = ctypes.c_int
    lib.oracle_lora_apply.argtypes = oracle._load().oracle_lora_apply.argtypes
    return lib


def _pins_pass(lib_func):
    saved = oracle._lib.oracle_lora_apply
    ok = True
    try:
        oracle._lib.oracle_lora_apply = lib_func
        for case in range(len(SHAPES)):
            for base in ("zero", "random"):
                try:
                    test_merged_weight_identity(case, base)
                except AssertionError:
                    ok = False
        try:
            test_none_rows_and_bad_ids_pass_through_exactly()
        except AssertionError:
            ok = False
    finally:
        oracle._lib.oracle_lora_apply = saved
    return ok


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(tmp_path, name):
    oracle._load()
    lib = _compile_mutant(tmp_path, name)
    assert not _pins_pass(lib.oracle_lora_apply), "pins accepted the planted mistake " + name
