"""Thin Python binding over the C ABI in include/lora.h.

Argument marshalling only: every step of the LoRA path runs in the CUDA
library (liblora.so).  torch supplies device memory and the current stream.
If the library is missing the calls raise; there is no fallback of any kind.
Function names match the C entry points.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build_lib

_c_i32, _c_i64, _c_f32, _c_sz, _c_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

STATUS = {0: "LORA_OK", 1: "LORA_ERR_INVALID_ARG", 2: "LORA_ERR_CUDA", 3: "LORA_ERR_OOM",
          4: "LORA_ERR_BAD_ADAPTER_ID", 5: "LORA_ERR_BAD_EXPERT_ID", 6: "LORA_ERR_TIMEOUT",
          7: "LORA_ERR_WORKSPACE", 8: "LORA_ERR_UNSUPPORTED"}
LORA_OK, LORA_ERR_INVALID_ARG, LORA_ERR_CUDA, LORA_ERR_OOM = 0, 1, 2, 3
LORA_ERR_BAD_ADAPTER_ID, LORA_ERR_BAD_EXPERT_ID, LORA_ERR_TIMEOUT, LORA_ERR_WORKSPACE, LORA_ERR_UNSUPPORTED = 4, 5, 6, 7, 8
LORA_MOE_GATE_UP, LORA_MOE_DOWN = 0, 1
LORA_OPT_PATH, LORA_OPT_TC_MIN_ROWS, LORA_OPT_WAIT_TIMEOUT_NS, LORA_OPT_GRID_CTAS, LORA_OPT_TEST_WITHHOLD_HANDOFF, \
    LORA_OPT_PDL = range(6)

EXPORTED = ["lora_pack_weights", "lora_table_destroy", "lora_table_info", "lora_table_stored_rank",
            "lora_workspace_bytes", "lora_workspace_layout", "lora_build_segments", "lora_apply",
            "lora_moe_delta", "lora_get_status", "lora_status_string", "lora_set_option", "lora_get_option",
            "lora_rank_padded", "lora_set_trace", "lora_apply_static_scratch", "lora_build_and_apply", "lora_linear",
            "lora_embedding_apply", "lora_table_set_adapter"]


class LoraError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__("%s: %s" % (where, STATUS.get(self.code, "status %d" % code)))


class AdapterDesc(ctypes.Structure):
    _fields_ = [("rank", _c_i32), ("scale", _c_f32), ("A", _c_p), ("B", _c_p)]


class ProjShape(ctypes.Structure):
    _fields_ = [("K", _c_i32), ("n_slices", _c_i32), ("slice_n", _c_i32 * 4), ("n_a", _c_i32), ("E_A", _c_i32),
                ("E_B", _c_i32)]


class WorkspaceDesc(ctypes.Structure):
    _fields_ = [("d_ptr", _c_p), ("bytes", _c_sz), ("max_M", _c_i32), ("L", _c_i32), ("topk", _c_i32),
                ("num_experts", _c_i32), ("block_m", _c_i32)]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, _c_sz) for n in ("header", "perm", "segments", "sorted_ids", "expert_ids", "ntpp",
                                      "moe_groups", "scratch")] + [("seg_capacity", _c_i32),
                                                                   ("moe_group_capacity", _c_i32)]


class TableInfo(ctypes.Structure):
    _fields_ = [(n, _c_i32) for n in ("L", "K", "N", "n_slices", "n_a", "E_A", "E_B", "num_rank_groups")] + \
               [("device_bytes", _c_i64), ("stored_rank_of_max", _c_i32)]


_lib = None


def library_path() -> str:
    return build_lib.LIB


def load(build_if_missing: bool = False):
    """Load liblora.so (in-tree).  Raises if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    path = build_lib.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError("liblora.so is not built (%s); run __graft_entry__.build() or "
                               "python -m segmented_rank_gemm_lora_gb300.build_lib" % path)
        build_lib.build()
    lib = ctypes.CDLL(path)
    P = _c_p
    sig = {
        "lora_pack_weights": (_c_i32, [P, _c_i32, P, P, P]),
        "lora_table_destroy": (_c_i32, [P]),
        "lora_table_info": (_c_i32, [P, P]),
        "lora_table_stored_rank": (_c_i32, [P, _c_i32]),
        "lora_workspace_bytes": (_c_sz, [_c_i32, _c_i32, _c_i32, _c_i32, _c_i32]),
        "lora_workspace_layout": (_c_i32, [P, P]),
        "lora_build_segments": (_c_i32, [P, P, _c_i32, P, P, P]),
        "lora_apply": (_c_i32, [P, P, P, _c_i64, P, _c_i64, P]),
        "lora_moe_delta": (_c_i32, [P, _c_i32, P, P, _c_i64, P, _c_i64, P, P]),
        "lora_get_status": (_c_i32, [P, P]),
        "lora_status_string": (ctypes.c_char_p, [_c_i32]),
        "lora_set_option": (_c_i32, [_c_i32, _c_i64]),
        "lora_get_option": (_c_i64, [_c_i32]),
        "lora_rank_padded": (_c_i32, [_c_i32]),
        "lora_set_trace": (_c_i32, [P, _c_sz]),
        "lora_apply_static_scratch": (_c_i32, [P, P, _c_i32, P, _c_i64, P, _c_i64, P]),
        "lora_build_and_apply": (_c_i32, [P, P, P, _c_i32, P, _c_i64, P, _c_i64, P]),
        "lora_linear": (_c_i32, [P, P, P, _c_i64, P, _c_i64, P, _c_i64, P]),
        "lora_embedding_apply": (_c_i32, [P, P, P, P, _c_i64, P]),
        "lora_table_set_adapter": (_c_i32, [P, _c_i32, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(code: int, where: str):
    if code != LORA_OK:
        raise LoraError(code, where)


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _bf16_dev(t: torch.Tensor, name: str):
    if not (t.is_cuda and t.dtype == torch.bfloat16):
        raise TypeError("%s must be a CUDA bfloat16 tensor" % name)


# ---------------------------------------------------------------------------
class Table:
    """Handle of a packed weight table (lora_table)."""

    def __init__(self, handle: int, L: int):
        self.handle = handle
        self.L = L

    def info(self) -> TableInfo:
        out = TableInfo()
        _check(load().lora_table_info(self.handle, ctypes.byref(out)), "lora_table_info")
        return out

    def stored_rank(self, adapter: int) -> int:
        return int(load().lora_table_stored_rank(self.handle, adapter))

    def destroy(self):
        if self.handle:
            _check(load().lora_table_destroy(self.handle), "lora_table_destroy")
            self.handle = None

    def __del__(self):
        try:
            if self.handle and _lib is not None:
                torch.cuda.synchronize()
                _lib.lora_table_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


def lora_pack_weights(A: Sequence[torch.Tensor], B: Sequence[torch.Tensor], ranks: Sequence[int],
                      scales: Sequence[float], K: int, slice_n: Sequence[int], n_a: Optional[int] = None,
                      E_A: int = 1, E_B: int = 1, stream=None) -> Table:
    """A[i]: bf16 [E_A, n_a*r, K] (or [n_a*r, K]); B[i]: bf16 [E_B, N, r] (or [N, r]); contiguous, on the GPU."""
    L = len(ranks)
    descs = (AdapterDesc * L)()
    for i in range(L):
        _bf16_dev(A[i], "A[%d]" % i)
        _bf16_dev(B[i], "B[%d]" % i)
        if not (A[i].is_contiguous() and B[i].is_contiguous()):
            raise ValueError("adapter weights must be contiguous")
        descs[i] = AdapterDesc(int(ranks[i]), float(scales[i]), A[i].data_ptr(), B[i].data_ptr())
    sh = ProjShape()
    sh.K = int(K)
    sh.n_slices = len(slice_n)
    for s, n in enumerate(slice_n):
        sh.slice_n[s] = int(n)
    sh.n_a = len(slice_n) if n_a is None else int(n_a)
    sh.E_A, sh.E_B = int(E_A), int(E_B)
    h = _c_p()
    _check(load().lora_pack_weights(descs, L, ctypes.byref(sh), _stream(stream), ctypes.byref(h)),
           "lora_pack_weights")
    return Table(h.value, L)


def lora_table_set_adapter(table: Table, index: int, A: torch.Tensor, B: torch.Tensor, rank: int, scale: float,
                           stream=None):
    """Hot-swap adapter `index` of a live table (shapes as in lora_pack_weights), in stream order."""
    _bf16_dev(A, "A")
    _bf16_dev(B, "B")
    if not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("adapter weights must be contiguous")
    desc = AdapterDesc(int(rank), float(scale), A.data_ptr(), B.data_ptr())
    _check(load().lora_table_set_adapter(table.handle, int(index), ctypes.byref(desc), _stream(stream)),
           "lora_table_set_adapter")


def lora_workspace_bytes(max_M: int, L: int, topk: int = 0, num_experts: int = 0, block_m: int = 0) -> int:
    return int(load().lora_workspace_bytes(max_M, L, topk, num_experts, block_m))


class Workspace:
    """A lora_workspace over a torch-allocated device buffer."""

    def __init__(self, max_M: int, L: int, topk: int = 0, num_experts: int = 0, block_m: int = 0, device=None,
                 buffer: Optional[torch.Tensor] = None):
        nbytes = lora_workspace_bytes(max_M, L, topk, num_experts, block_m)
        if nbytes == 0:
            raise LoraError(LORA_ERR_INVALID_ARG, "lora_workspace_bytes")
        if buffer is None:
            buffer = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-buffer.data_ptr()) % 256
        self.buffer = buffer
        self.desc = WorkspaceDesc(buffer.data_ptr() + off, buffer.numel() - off, max_M, L, topk, num_experts, block_m)
        self.offset = off
        self.built_M = None        # token count of the last lora_build_segments through this binding

    @property
    def ref(self):
        return ctypes.byref(self.desc)

    def layout(self) -> WorkspaceLayout:
        out = WorkspaceLayout()
        _check(load().lora_workspace_layout(self.ref, ctypes.byref(out)), "lora_workspace_layout")
        return out

    def _ints(self, byte_off: int, count: int) -> torch.Tensor:
        base = self.offset + byte_off
        return self.buffer[base:base + 4 * count].view(torch.int32)

    def read_segments(self) -> dict:
        """Copy the segment table (and MoE alignment, if built) to host numpy arrays."""
        lay = self.layout()
        h = self._ints(lay.header, 16).cpu().numpy()
        M, nseg, nval, nmoe = int(h[0]), int(h[1]), int(h[2]), int(h[3])
        out = dict(M=M, num_segments=nseg, num_valid=nval,
                   perm=self._ints(lay.perm, M).cpu().numpy(),
                   segments=self._ints(lay.segments, 4 * nseg).view(-1, 4).cpu().numpy())
        if self.desc.block_m > 0 and int(h[6]) > 0:
            L = self.desc.L
            P_max, B_max = int(h[7]), int(h[8])
            out.update(P_max=P_max, B_max=B_max,
                       sorted_ids=self._ints(lay.sorted_ids, L * P_max).view(L, P_max).cpu().numpy(),
                       expert_ids=self._ints(lay.expert_ids, L * B_max).view(L, B_max).cpu().numpy(),
                       ntpp=self._ints(lay.ntpp, L).cpu().numpy(),
                       moe_groups=self._ints(lay.moe_groups, 4 * nmoe).view(-1, 4).cpu().numpy())
        return out


def lora_build_segments(ws: Workspace, ids: torch.Tensor, topk_ids: Optional[torch.Tensor] = None,
                        enabled: Optional[torch.Tensor] = None, stream=None):
    if ids.dtype != torch.int32 or not ids.is_cuda or not ids.is_contiguous():
        raise TypeError("ids must be a contiguous CUDA int32 tensor")
    tk = 0
    if topk_ids is not None:
        if topk_ids.dtype != torch.int32 or not topk_ids.is_contiguous():
            raise TypeError("topk_ids must be a contiguous CUDA int32 tensor")
        tk = topk_ids.data_ptr()
    en = 0
    if enabled is not None:
        if enabled.dtype != torch.uint8:
            raise TypeError("enabled must be a CUDA uint8 tensor")
        en = enabled.data_ptr()
    _check(load().lora_build_segments(ws.ref, ids.data_ptr(), int(ids.numel()), tk or None, en or None,
                                      _stream(stream)), "lora_build_segments")
    ws.built_M = int(ids.numel())
    ws.built_topk = int(topk_ids.shape[1]) if topk_ids is not None and topk_ids.dim() == 2 else None


def lora_apply(table: Table, ws: Workspace, x: torch.Tensor, y: torch.Tensor, stream=None):
    """y (bf16 [M, N], holds y_base) += per-token LoRA delta of x (bf16 [M, K]); in place."""
    _bf16_dev(x, "x")
    _bf16_dev(y, "y")
    if x.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("x and y need unit column stride")
    if ws.built_M is not None and (x.shape[0] < ws.built_M or y.shape[0] < ws.built_M):
        raise ValueError("x and y need the %d rows of the last lora_build_segments" % ws.built_M)
    _check(load().lora_apply(table.handle, ws.ref, x.data_ptr(), x.stride(0), y.data_ptr(), y.stride(0),
                             _stream(stream)), "lora_apply")


def lora_build_and_apply(table: Table, ws: Workspace, ids: torch.Tensor, x: torch.Tensor, y: torch.Tensor,
                         stream=None):
    """lora_build_segments(ws, ids) then lora_apply(table, ws, x, y), in one launch for decode-sized batches."""
    if ids.dtype != torch.int32 or not ids.is_cuda or not ids.is_contiguous():
        raise TypeError("ids must be a contiguous CUDA int32 tensor")
    _bf16_dev(x, "x")
    _bf16_dev(y, "y")
    if x.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("x and y need unit column stride")
    M = int(ids.numel())
    if x.shape[0] < M or y.shape[0] < M:
        raise ValueError("x and y need a row for each of the %d ids" % M)
    _check(load().lora_build_and_apply(table.handle, ws.ref, ids.data_ptr(), M, x.data_ptr(), x.stride(0),
                                       y.data_ptr(), y.stride(0), _stream(stream)), "lora_build_and_apply")
    ws.built_M = M


def lora_moe_delta(table: Table, stage: int, ws: Workspace, inp: torch.Tensor, cache: torch.Tensor,
                   topk_weights: Optional[torch.Tensor] = None, stream=None):
    _bf16_dev(inp, "inp")
    _bf16_dev(cache, "cache")
    if ws.built_M is not None and ws.built_topk:
        pairs = ws.built_M * ws.built_topk
        need_in = ws.built_M if stage == LORA_MOE_GATE_UP else pairs
        if inp.shape[0] < need_in or cache.shape[0] < pairs:
            raise ValueError("MoE operands are smaller than the last alignment needs")
    w = None
    if topk_weights is not None:
        if topk_weights.dtype != torch.float32 or not topk_weights.is_contiguous():
            raise TypeError("topk_weights must be contiguous float32")
        w = topk_weights.data_ptr()
    _check(load().lora_moe_delta(table.handle, int(stage), ws.ref, inp.data_ptr(), inp.stride(0), cache.data_ptr(),
                                 cache.stride(0), w, _stream(stream)), "lora_moe_delta")


def lora_linear(table: Table, ws: Workspace, x: torch.Tensor, W: torch.Tensor, y: torch.Tensor, stream=None):
    """y (bf16 [M, N]) = x W^T + per-token LoRA delta of x (bf16 [M, K]), in one kernel; W bf16 [N, K]."""
    _bf16_dev(x, "x")
    _bf16_dev(W, "W")
    _bf16_dev(y, "y")
    if x.stride(1) != 1 or W.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("x, W and y need unit column stride")
    if ws.built_M is not None and (x.shape[0] < ws.built_M or y.shape[0] < ws.built_M):
        raise ValueError("x and y need the %d rows of the last lora_build_segments" % ws.built_M)
    _check(load().lora_linear(table.handle, ws.ref, x.data_ptr(), x.stride(0), W.data_ptr(), W.stride(0),
                              y.data_ptr(), y.stride(0), _stream(stream)), "lora_linear")


def lora_embedding_apply(table: Table, ws: Workspace, vocab: torch.Tensor, y: torch.Tensor, stream=None):
    """y (bf16 [M, N], the base embedding rows) += scale_i * B_i A_i[:, vocab[t]] per token (embedding LoRA)."""
    if vocab.dtype != torch.int32 or not vocab.is_cuda or not vocab.is_contiguous():
        raise TypeError("vocab must be a contiguous CUDA int32 tensor")
    _bf16_dev(y, "y")
    if y.stride(1) != 1:
        raise ValueError("y needs unit column stride")
    if ws.built_M is not None and (vocab.numel() < ws.built_M or y.shape[0] < ws.built_M):
        raise ValueError("vocab and y need the %d rows of the last lora_build_segments" % ws.built_M)
    _check(load().lora_embedding_apply(table.handle, ws.ref, vocab.data_ptr(), y.data_ptr(), y.stride(0),
                                       _stream(stream)), "lora_embedding_apply")


def lora_get_status(ws: Workspace, stream=None) -> int:
    """Synchronise the stream and return (and clear) the sticky device status code."""
    return int(load().lora_get_status(ws.ref, _stream(stream)))


def lora_set_option(option: int, value: int):
    _check(load().lora_set_option(int(option), int(value)), "lora_set_option")


def lora_get_option(option: int) -> int:
    return int(load().lora_get_option(int(option)))


def lora_set_trace(buf: Optional[torch.Tensor]):
    """Per-block phase stamps of later engine launches into buf (CUDA int64/uint8 tensor), or None to stop."""
    if buf is None:
        _check(load().lora_set_trace(None, 0), "lora_set_trace")
    else:
        _check(load().lora_set_trace(buf.data_ptr(), buf.numel() * buf.element_size()), "lora_set_trace")


def lora_rank_padded(rank: int) -> int:
    return int(load().lora_rank_padded(int(rank)))


def lora_status_string(code: int) -> str:
    return load().lora_status_string(int(code)).decode()
