"""Helpers shared by the GPU parity tests: move synthetic problems to the
device, run them through the C ABI, and compare with the CPU oracle."""
import numpy as np
import torch

import oracle
from segmented_rank_gemm_lora_gb300 import lora, synth

TOL = 1e-2   # max|y - y_ref| <= TOL * max|y_ref|, fp32 accumulation of bf16 inputs


def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t):
    return synth.bf16_bits_to_f32(host_bits(t)).astype(np.float64)


def pack_dense(p):
    A = [dev_bf16(a) for a in p.A]
    B = [dev_bf16(b) for b in p.B]
    t = lora.lora_pack_weights(A, B, p.ranks, p.scales, p.K, p.slice_n, p.n_a)
    torch.cuda.synchronize()
    return t


def padded(a, extra_cols, fill=0x7FC1):
    """Copy of a [rows, cols] bf16-bit array with extra canary columns (leading dim cols+extra)."""
    if extra_cols == 0:
        return a
    out = np.full((a.shape[0], a.shape[1] + extra_cols), fill, np.uint16)
    out[:, :a.shape[1]] = a
    return out


def run_dense(p, table=None, ws=None, x_extra=0, y_extra=0, build=True, y_base=None):
    """lora_build_segments + lora_apply on problem p; returns (y_device_full, table, ws)."""
    table = table or pack_dense(p)
    ws = ws or lora.Workspace(max(p.M, 1), p.L)
    ids = torch.from_numpy(p.ids).cuda()
    xh = padded(p.x, x_extra)
    yh = padded(p.y_base if y_base is None else y_base, y_extra)
    x = dev_bf16(xh)
    y = dev_bf16(yh)
    if build:
        lora.lora_build_segments(ws, ids)
    lora.lora_apply(table, ws, x[:, :p.K] if x_extra else x, y[:, :p.N] if y_extra else y)
    return y, table, ws


def oracle_dense(p, y_base=None):
    ref, bad = oracle.lora_apply(p.ids, p.x, p.y_base if y_base is None else y_base, p.A, p.B, p.ranks, p.scales,
                                 p.slice_n, p.n_a)
    return ref


def check_close(got, ref, what=""):
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    assert err <= TOL * scale, "%s: max err %.4g vs bound %.4g" % (what, err, TOL * scale)
    return err, scale


class forced_path:
    """Context manager: LORA_OPT_PATH = path inside the block (0 automatic: the persistent engine for dense
    workspaces of at most 32 tokens, else the streaming path; 1 the persistent engine on small tiles, 2 the
    persistent engine on 128-row tiles, 3 the streaming path on 16-row tiles)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        self.old = lora.lora_get_option(lora.LORA_OPT_PATH)
        lora.lora_set_option(lora.LORA_OPT_PATH, self.path)

    def __exit__(self, *exc):
        lora.lora_set_option(lora.LORA_OPT_PATH, self.old)


PATHS = (0, 1, 2, 3)
