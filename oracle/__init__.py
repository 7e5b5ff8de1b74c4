"""CPU oracle for the multi-adapter LoRA hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its binding) never loads it, and this
package imports nothing from the product.

The arithmetic lives in ``lora_oracle.c`` (plain C99, fp64, per-token loops);
this module compiles it with gcc on first use and marshals numpy arrays into
it with ctypes.  Every function returns float64 results.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against values fixed independently of it (merged-weight identities, the MoE
merged-weight block identity, library sorts on the same keys, worked examples
from the pages under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile lora_oracle.c into oracle/_build/liboracle.so (gcc, no FP contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_lora_apply.restype = ctypes.c_int
            lib.oracle_lora_apply.argtypes = [_I32, _I32, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                              _P, _I64, _P, _I64, _P]
            lib.oracle_embedding_apply.restype = ctypes.c_int
            lib.oracle_embedding_apply.argtypes = [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _I64, _P]
            lib.oracle_matmul_bt.restype = None
            lib.oracle_matmul_bt.argtypes = [_I32, _I32, _I32, _P, _I64, _P, _I64, _P]
            lib.oracle_build_segments.restype = ctypes.c_int
            lib.oracle_build_segments.argtypes = [_I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P]
            lib.oracle_moe_align.restype = ctypes.c_int
            lib.oracle_moe_align.argtypes = [_I32, _I32, _I32, _I32, _I32, _P, _P, _P, _I32, _I32, _P, _P, _P]
            lib.oracle_moe_delta.restype = ctypes.c_int
            lib.oracle_moe_delta.argtypes = [_I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _I32, _I32, _P, _P,
                                             _P, _P, _P, _P, _I32, _P, _I64, _P, _I64, _P]
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr_array(arrs):
    keep = [_c(a, np.uint16) for a in arrs]
    table = (ctypes.c_void_p * max(1, len(keep)))(*[a.ctypes.data for a in keep])
    return table, keep


def lora_apply(ids, x, y_base, A: Sequence[np.ndarray], B: Sequence[np.ndarray], ranks, scales,
               slice_n, n_a: Optional[int] = None, enabled=None):
    """y = y_base + scale_i * (x A_i^T) B_i^T per token (float64 [M, N]); returns (y, bad_id_count).

    x: bf16 bits [M, K]; y_base: bf16 bits [M, N]; A[i]: [n_a*r_i, K]; B[i]: [N, r_i].
    """
    lib = _load()
    ids = _c(ids, np.int32)
    x = _c(x, np.uint16)
    y_base = _c(y_base, np.uint16)
    M, K = x.shape
    slice_n = _c(slice_n, np.int32)
    n_a = len(slice_n) if n_a is None else int(n_a)
    N = int(slice_n.sum())
    assert y_base.shape == (M, N) and ids.shape == (M,)
    ranks = _c(ranks, np.int32)
    scales = _c(scales, np.float64)
    for i, r in enumerate(ranks):
        assert A[i].shape == (n_a * r, K), (A[i].shape, n_a, r, K)
        assert B[i].shape == (N, r)
    pa, ka = _ptr_array(A)
    pb, kb = _ptr_array(B)
    en = None if enabled is None else _c(enabled, np.uint8)
    out = np.empty((M, N), np.float64)
    bad = lib.oracle_lora_apply(M, K, len(slice_n), _ptr(slice_n), n_a, len(ranks), _ptr(ranks), _ptr(scales),
                                pa, pb, _ptr(ids), _ptr(en), _ptr(x), K, _ptr(y_base), N, _ptr(out))
    return out, int(bad)


def matmul_bt(x, W):
    """Base projection x W^T (float64 [M, N]) of bf16 bits x [M, K] and W [N, K]."""
    lib = _load()
    x = _c(x, np.uint16)
    W = _c(W, np.uint16)
    M, K = x.shape
    N = W.shape[0]
    assert W.shape == (N, K)
    out = np.empty((M, N), np.float64)
    lib.oracle_matmul_bt(M, N, K, _ptr(x), K, _ptr(W), K, _ptr(out))
    return out


def lora_linear(ids, x, W, A: Sequence[np.ndarray], B: Sequence[np.ndarray], ranks, scales, slice_n,
                n_a: Optional[int] = None):
    """A LoRA linear layer ("vLLM-Ascend dynamic LoRA fused operator", section 3.3): the base projection
    x W^T plus every token's LoRA delta, as float64 [M, N]; returns (y, bad_id_count)."""
    M = np.asarray(x).shape[0]
    N = int(np.sum(slice_n))
    delta, bad = lora_apply(ids, x, np.zeros((M, N), np.uint16), A, B, ranks, scales, slice_n, n_a)
    return matmul_bt(x, W) + delta, bad


def embedding_apply(ids, vocab, y_base, A: Sequence[np.ndarray], B: Sequence[np.ndarray], ranks, scales):
    """Embedding LoRA ("[SGLang] LoRA Layers", VocabParallelEmbeddingWithLoRA): y = y_base + scale_i * B_i
    A_i[:, vocab[t]] per token (float64 [M, N]); returns (y, bad_count).  A[i]: bf16 bits [r_i, V];
    B[i]: [N, r_i]; y_base: bf16 bits [M, N]."""
    lib = _load()
    ids = _c(ids, np.int32)
    vocab = _c(vocab, np.int32)
    y_base = _c(y_base, np.uint16)
    M, N = y_base.shape
    ranks = _c(ranks, np.int32)
    scales = _c(scales, np.float64)
    V = A[0].shape[1]
    for i, r in enumerate(ranks):
        assert A[i].shape == (r, V) and B[i].shape == (N, r)
    pa, ka = _ptr_array(A)
    pb, kb = _ptr_array(B)
    out = np.empty((M, N), np.float64)
    bad = lib.oracle_embedding_apply(M, V, N, len(ranks), _ptr(ranks), _ptr(scales), pa, pb, _ptr(ids), _ptr(vocab),
                                     _ptr(y_base), N, _ptr(out))
    return out, int(bad)


def build_segments(ids, L: int, enabled=None):
    """Counting-sort segment table: dict(perm, seg_adapter, seg_start, seg_len, num_valid, bad)."""
    lib = _load()
    ids = _c(ids, np.int32)
    M = int(ids.shape[0])
    perm = np.empty(max(M, 1), np.int32)
    cap = max(1, min(L, M))
    sa = np.empty(cap, np.int32)
    ss = np.empty(cap, np.int32)
    sl = np.empty(cap, np.int32)
    ns = np.zeros(1, np.int32)
    nv = np.zeros(1, np.int32)
    en = None if enabled is None else _c(enabled, np.uint8)
    bad = lib.oracle_build_segments(M, L, _ptr(ids), _ptr(en), _ptr(perm), _ptr(sa), _ptr(ss), _ptr(sl),
                                    _ptr(ns), _ptr(nv))
    n = int(ns[0])
    return dict(perm=perm[:M].copy(), seg_adapter=sa[:n].copy(), seg_start=ss[:n].copy(), seg_len=sl[:n].copy(),
                num_segments=n, num_valid=int(nv[0]), bad=int(bad))


def moe_padded_sizes(M: int, topk: int, E: int, block_m: int):
    """(P_max, B_max): per-adapter capacity of the aligned pair list and its block count."""
    P_max = ((M * topk + E * (block_m - 1) + block_m - 1) // block_m) * block_m
    return P_max, P_max // block_m


def moe_align(ids, topk_ids, L: int, E: int, block_m: int, enabled=None):
    """(adapter, expert) alignment: dict(sorted_ids [L,P_max], expert_ids [L,B_max], ntpp [L], bad)."""
    lib = _load()
    ids = _c(ids, np.int32)
    topk_ids = _c(topk_ids, np.int32)
    M, topk = topk_ids.shape
    P_max, B_max = moe_padded_sizes(M, topk, E, block_m)
    srt = np.empty((L, P_max), np.int32)
    eid = np.empty((L, B_max), np.int32)
    ntpp = np.empty(L, np.int32)
    en = None if enabled is None else _c(enabled, np.uint8)
    bad = lib.oracle_moe_align(M, topk, E, L, block_m, _ptr(ids), _ptr(topk_ids), _ptr(en), P_max, B_max,
                               _ptr(srt), _ptr(eid), _ptr(ntpp))
    return dict(sorted_ids=srt, expert_ids=eid, ntpp=ntpp, P_max=P_max, B_max=B_max, bad=int(bad))


def moe_delta(ids, topk_ids, src, cache, A, B, ranks, scales, E: int, src_is_token: bool,
              topk_weights=None, enabled=None):
    """One MoE LoRA stage (gate/up: src = hidden [M,K], per token; down: src = [P,K], per pair).

    A[l]: [E_A, r, K]; B[l]: [E_B, N, r]; cache: [P, N].  Returns (float64 [P, N], bad).
    """
    lib = _load()
    ids = _c(ids, np.int32)
    topk_ids = _c(topk_ids, np.int32)
    M, topk = topk_ids.shape
    src = _c(src, np.uint16)
    cache = _c(cache, np.uint16)
    P, N = cache.shape
    K = src.shape[1]
    E_A = A[0].shape[0]
    E_B = B[0].shape[0]
    ranks = _c(ranks, np.int32)
    scales = _c(scales, np.float64)
    for l, r in enumerate(ranks):
        assert A[l].shape == (E_A, r, K) and B[l].shape == (E_B, N, r)
    pa, ka = _ptr_array(A)
    pb, kb = _ptr_array(B)
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    en = None if enabled is None else _c(enabled, np.uint8)
    out = np.empty((P, N), np.float64)
    bad = lib.oracle_moe_delta(M, topk, E, len(ranks), K, N, _ptr(ranks), _ptr(scales), E_A, E_B, pa, pb,
                               _ptr(ids), _ptr(topk_ids), _ptr(en), _ptr(w), 1 if src_is_token else 0,
                               _ptr(src), K, _ptr(cache), N, _ptr(out))
    return out, int(bad)
