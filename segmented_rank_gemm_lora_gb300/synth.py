"""Seeded synthetic inputs for the multi-adapter LoRA workloads.

This module only draws numbers: adapter-id maps, activations, base outputs and
adapter weights, rounded to bf16.  It contains none of the LoRA arithmetic
(no shrink, no expand, no segmenting), so the CPU oracle and the CUDA path can
both consume its output without sharing any of the method's code.

Every array kind comes from its own counter-keyed numpy PCG64 stream
(``default_rng([seed, kind, index])``), so any subset of a workload can be drawn
without drawing the rest, and the same bytes come out on every machine.

bf16 arrays are returned as numpy ``uint16`` holding the bf16 bit patterns
(round-to-nearest-even from the fp32 draw).

Workloads (the adapter-id structure follows the operator description in
"vLLM-Ascend dynamic LoRA fused operator", section 3.2: decode maps are one
token per sequence, prefill maps are long runs of one id):

* ``tiny``     M=64, K=256, N=512, ranks (8,16,16,32), ids uniform in {-1..3}
* ``decode``   M=32, K=N=4096, 20 adapters, ranks cycling (16,32,64), 10 % of
               tokens set to -1
* ``prefill``  16 requests, lengths from a discrete power law l^-1.2 on
               [16,512], one adapter per request, K=N=4096, ranks cycling
* ``stacked``  M=1024 (512 decode tokens then prefill runs), 32 adapters of
               rank 64; projections qkv / gate_up / down
* ``moe``      M=512, top-2 of 8 experts, hidden 4096, intermediate 14336,
               8 adapters, ranks cycling (16,32,64)
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

# stream kinds for default_rng([seed, kind, index])
_K_STRUCT, _K_X, _K_W, _K_A, _K_B, _K_YBASE, _K_CACHE, _K_ROUTER = range(8)


# ----------------------------------------------------------------------------
# bf16 helpers (bit-pattern conversions only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 -> bf16 (nearest even), returned as uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 exactly."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def _rng(seed: int, kind: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(kind), int(index)])


# ----------------------------------------------------------------------------
# dense (token-level) problems
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class DenseProblem:
    """One LoRA-wrapped linear layer over one batch of tokens.

    A[i] has shape [n_a * rank[i], K] (n_a = 1 or n_slices; row block s is the
    shrink weight of output slice s), B[i] has shape [sum(slice_n), rank[i]].
    """
    name: str
    M: int
    K: int
    slice_n: List[int]
    n_a: int
    ranks: List[int]
    scales: List[float]
    ids: np.ndarray            # int32 [M], -1 = no adapter
    x: np.ndarray              # uint16 bf16 [M, K]
    A: List[np.ndarray]        # uint16 bf16 [n_a*r, K]
    B: List[np.ndarray]        # uint16 bf16 [N, r]
    y_base: Optional[np.ndarray] = None  # uint16 bf16 [M, N]
    W: Optional[np.ndarray] = None       # uint16 bf16 [N, K] (only when asked for)

    @property
    def N(self) -> int:
        return int(sum(self.slice_n))

    @property
    def L(self) -> int:
        return len(self.ranks)


def power_law_lengths(rng: np.random.Generator, count: int, lo: int = 16, hi: int = 512,
                      alpha: float = 1.2) -> np.ndarray:
    """Request lengths from P(l) ~ l^-alpha on [lo, hi] by inverse CDF."""
    ell = np.arange(lo, hi + 1, dtype=np.float64)
    pmf = ell ** (-alpha)
    cdf = np.cumsum(pmf) / pmf.sum()
    u = rng.random(count)
    idx = np.searchsorted(cdf, u, side="right")
    idx = np.minimum(idx, len(ell) - 1)
    return ell[idx].astype(np.int64)


def ids_tiny(seed: int = 0) -> np.ndarray:
    return _rng(seed, _K_STRUCT).integers(-1, 4, 64).astype(np.int32)


def ids_decode(seed: int, M: int = 32, L: int = 20, frac_none: float = 0.1) -> np.ndarray:
    rng = _rng(seed, _K_STRUCT)
    ids = rng.integers(0, L, M).astype(np.int32)
    n_none = int(round(frac_none * M))
    if n_none:
        ids[rng.choice(M, n_none, replace=False)] = -1
    return ids


def ids_prefill(seed: int, n_req: int = 16) -> np.ndarray:
    rng = _rng(seed, _K_STRUCT)
    lens = power_law_lengths(rng, n_req)
    return np.concatenate([np.full(int(n), j, np.int32) for j, n in enumerate(lens)])


def ids_stacked(seed: int, M: int = 1024, n_decode: int = 512, L: int = 32) -> np.ndarray:
    rng = _rng(seed, _K_STRUCT)
    parts = [rng.integers(0, L, n_decode).astype(np.int32)]
    have = n_decode
    while have < M:
        n = int(power_law_lengths(rng, 1)[0])
        n = min(n, M - have)
        parts.append(np.full(n, int(rng.integers(0, L)), np.int32))
        have += n
    return np.concatenate(parts)


def make_dense(name: str, seed: int, ids: np.ndarray, K: int, slice_n: Sequence[int], ranks: Sequence[int],
               n_a: Optional[int] = None, scale: float = 2.0, with_W: bool = False,
               y_base: str = "random") -> DenseProblem:
    """Draw one dense problem.

    x ~ N(0,1); A_i ~ N(0, 1/K); B_i ~ N(0, 1/r_i); all bf16.
    y_base: "xw" (bf16 of the fp32 product x @ W^T, W ~ N(0,1)), "zero"
    (delta-only runs), "random" (N(0, K) entries, the distribution of x @ W^T,
    drawn directly for sizes where the base GEMM is not worth running on the
    host), or "none".
    """
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    M = int(ids.shape[0])
    slice_n = [int(n) for n in slice_n]
    n_a = len(slice_n) if n_a is None else int(n_a)
    N = sum(slice_n)
    x = _normal_bf16(_rng(seed, _K_X), (M, K), 1.0)
    A = [_normal_bf16(_rng(seed, _K_A, i), (n_a * r, K), 1.0 / np.sqrt(K)) for i, r in enumerate(ranks)]
    B = [_normal_bf16(_rng(seed, _K_B, i), (N, r), 1.0 / np.sqrt(r)) for i, r in enumerate(ranks)]
    W = _normal_bf16(_rng(seed, _K_W), (N, K), 1.0) if with_W else None
    if y_base == "xw":
        if W is None:
            W = _normal_bf16(_rng(seed, _K_W), (N, K), 1.0)
        yb = f32_to_bf16_bits(bf16_bits_to_f32(x) @ bf16_bits_to_f32(W).T)
    elif y_base == "zero":
        yb = np.zeros((M, N), np.uint16)
    elif y_base == "random":
        yb = _normal_bf16(_rng(seed, _K_YBASE), (M, N), float(np.sqrt(K)))
    else:
        yb = None
    return DenseProblem(name=name, M=M, K=K, slice_n=slice_n, n_a=n_a, ranks=[int(r) for r in ranks],
                        scales=[float(scale)] * len(ranks), ids=ids, x=x, A=A, B=B, y_base=yb, W=W)


def cycle_ranks(L: int, cycle=(16, 32, 64)) -> List[int]:
    return [int(cycle[i % len(cycle)]) for i in range(L)]


def tiny(seed: int = 0, **kw) -> DenseProblem:
    return make_dense("tiny", seed, ids_tiny(seed), 256, [512], [8, 16, 16, 32], **kw)


def decode(seed: int = 1, **kw) -> DenseProblem:
    return make_dense("decode", seed, ids_decode(seed), 4096, [4096], cycle_ranks(20), **kw)


def prefill(seed: int = 2, **kw) -> DenseProblem:
    return make_dense("prefill", seed, ids_prefill(seed), 4096, [4096], cycle_ranks(16), **kw)


STACKED_PROJ = {
    # name: (K, slice widths, rows of A per slice block count)
    "qkv": (4096, [4096, 1024, 1024]),
    "gate_up": (4096, [14336, 14336]),
    "down": (14336, [4096]),
}


def stacked(proj: str, seed: int = 3, **kw) -> DenseProblem:
    K, slices = STACKED_PROJ[proj]
    sub = {"qkv": 0, "gate_up": 1, "down": 2}[proj]
    return make_dense("stacked_" + proj, seed * 16 + sub, ids_stacked(seed), K, slices, [64] * 32, **kw)


# ----------------------------------------------------------------------------
# MoE problems
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class MoEProblem:
    """LoRA deltas inside one MoE block.

    gate/up: A_gu[l] [E_A_gu, r, H], B_gu[l] [E_B_gu, 2I, r]
    down:    A_d[l]  [E_A_d,  r, I], B_d[l]  [E_B_d,  H, r]
    Pairs p = t*topk + k carry expert topk_ids[t, k].
    """
    M: int
    H: int
    I: int
    E: int
    topk: int
    block_m: int
    ranks: List[int]
    scales: List[float]
    ids: np.ndarray           # int32 [M]
    topk_ids: np.ndarray      # int32 [M, topk]
    topk_weights: np.ndarray  # float32 [M, topk]
    x: np.ndarray             # bf16 [M, H]
    cache1: np.ndarray        # bf16 [M*topk, 2I]  gate/up base output
    cache2: np.ndarray        # bf16 [M*topk, I]   SiLU(gate)*up input of the down projection
    cache3: np.ndarray        # bf16 [M*topk, H]   down base output
    A_gu: List[np.ndarray]
    B_gu: List[np.ndarray]
    A_d: List[np.ndarray]
    B_d: List[np.ndarray]

    @property
    def L(self) -> int:
        return len(self.ranks)


def router_topk(seed: int, M: int, E: int, topk: int):
    """Softmax router over N(0,1) logits; top-k by probability, lower expert id on ties."""
    logits = _rng(seed, _K_ROUTER).standard_normal((M, E), dtype=np.float32)
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z.astype(np.float64))
    p = p / p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :topk]
    w = np.take_along_axis(p, order, axis=1)
    return order.astype(np.int32), w.astype(np.float32)


def moe_routing(seed: int, M: int, E: int, topk: int, L: int, ids: Optional[np.ndarray] = None):
    """(ids, topk_ids, topk_weights) of an MoE batch: ids uniform over the L adapters."""
    if ids is None:
        ids = _rng(seed, _K_STRUCT).integers(0, L, M).astype(np.int32)
    topk_ids, topk_w = router_topk(seed, M, E, topk)
    return np.ascontiguousarray(ids, dtype=np.int32), topk_ids, topk_w


def make_moe(seed: int, M: int, H: int, I: int, E: int, topk: int, ranks: Sequence[int], block_m: int = 64,
             ids: Optional[np.ndarray] = None, shared_outer: bool = True, scale: float = 2.0,
             zero_base: bool = False) -> MoEProblem:
    """Draw one MoE LoRA problem.

    shared_outer=True gives A_gu [1, r, H] (shared by all experts) and
    B_d [1, H, r]; the expert-specific factors are B_gu [E, 2I, r] and
    A_d [E, r, I].  The base caches are drawn with unit variance (the scale
    of the base expert GEMM outputs with W ~ N(0, 1/in_features)); cache2 is
    SiLU(g)*u of two such draws.  zero_base=True zeroes cache1/cache3 for
    delta-only checks.
    """
    L = len(ranks)
    ids, topk_ids, topk_w = moe_routing(seed, M, E, topk, L, ids)
    P = M * topk
    x = _normal_bf16(_rng(seed, _K_X), (M, H), 1.0)
    if zero_base:
        c1 = np.zeros((P, 2 * I), np.uint16)
        c3 = np.zeros((P, H), np.uint16)
    else:
        c1 = _normal_bf16(_rng(seed, _K_CACHE, 1), (P, 2 * I), 1.0)
        c3 = _normal_bf16(_rng(seed, _K_CACHE, 3), (P, H), 1.0)
    rg = _rng(seed, _K_CACHE, 2)
    g = rg.standard_normal((P, I), dtype=np.float32)
    u = rg.standard_normal((P, I), dtype=np.float32)
    c2 = f32_to_bf16_bits(g / (1.0 + np.exp(-g)) * u)
    e_gu_a, e_d_b = (1, 1) if shared_outer else (E, E)
    A_gu = [_normal_bf16(_rng(seed, _K_A, 2 * l), (e_gu_a, r, H), 1.0 / np.sqrt(H)) for l, r in enumerate(ranks)]
    B_gu = [_normal_bf16(_rng(seed, _K_B, 2 * l), (E, 2 * I, r), 1.0 / np.sqrt(r)) for l, r in enumerate(ranks)]
    A_d = [_normal_bf16(_rng(seed, _K_A, 2 * l + 1), (E, r, I), 1.0 / np.sqrt(I)) for l, r in enumerate(ranks)]
    B_d = [_normal_bf16(_rng(seed, _K_B, 2 * l + 1), (e_d_b, H, r), 1.0 / np.sqrt(r)) for l, r in enumerate(ranks)]
    return MoEProblem(M=M, H=H, I=I, E=E, topk=topk, block_m=block_m, ranks=[int(r) for r in ranks],
                      scales=[float(scale)] * L, ids=ids, topk_ids=topk_ids, topk_weights=topk_w, x=x,
                      cache1=c1, cache2=c2, cache3=c3, A_gu=A_gu, B_gu=B_gu, A_d=A_d, B_d=B_d)


def moe(seed: int = 4, **kw) -> MoEProblem:
    return make_moe(seed, 512, 4096, 14336, 8, 2, cycle_ranks(8), block_m=64, **kw)


# ----------------------------------------------------------------------------
# small integer problems (every intermediate exactly representable in bf16)
# ----------------------------------------------------------------------------
def _small_ints(rng: np.random.Generator, shape, lo: int, hi: int, p_nonzero: float) -> np.ndarray:
    v = rng.integers(lo, hi + 1, shape).astype(np.float32)
    v *= (rng.random(shape) < p_nonzero).astype(np.float32)
    return f32_to_bf16_bits(v)


def make_dense_int(seed: int, ids: np.ndarray, K: int, slice_n: Sequence[int], ranks: Sequence[int],
                   n_a: Optional[int] = None) -> DenseProblem:
    """Integer-valued dense problem with scale 1.

    x in {-2..2} (half zero), A and B in {-1,0,1} (mostly zero), y_base in
    {-8..8}.  The caller checks that every partial sum stays an integer of
    magnitude <= 256, so bf16 and fp32 rounding are exact everywhere.
    """
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    M = int(ids.shape[0])
    slice_n = [int(n) for n in slice_n]
    n_a = len(slice_n) if n_a is None else int(n_a)
    N = sum(slice_n)
    x = _small_ints(_rng(seed, _K_X), (M, K), -2, 2, 0.5)
    A = [_small_ints(_rng(seed, _K_A, i), (n_a * r, K), -1, 1, 0.08) for i, r in enumerate(ranks)]
    B = [_small_ints(_rng(seed, _K_B, i), (N, r), -1, 1, 0.25) for i, r in enumerate(ranks)]
    yb = _small_ints(_rng(seed, _K_YBASE), (M, N), -8, 8, 1.0)
    return DenseProblem(name="int", M=M, K=K, slice_n=slice_n, n_a=n_a, ranks=[int(r) for r in ranks],
                        scales=[1.0] * len(ranks), ids=ids, x=x, A=A, B=B, y_base=yb)
