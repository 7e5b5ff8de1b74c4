"""lora_apply_static_scratch: one step with no device memory from the caller.

This entry point serves callers that cannot allocate device memory (they can
only hand over their inputs and outputs): it keeps the segment table and the
hand-off scratch in a fixed array inside the library.  Its output must match
the workspace-based path (lora_build_segments + lora_apply) within the
tolerance every GPU test here uses, on consecutive calls that reuse the array.
This file is collected last so a failure here cannot hide any other test.
"""
import numpy as np
import pytest
import torch

from segmented_rank_gemm_lora_gb300 import lora, synth
from gpu_util import check_close, dev_bf16, host_f64, pack_dense, run_dense

pytestmark = pytest.mark.gpu


def static_apply(table, ids, x, y):
    lib = lora.load()
    return lib.lora_apply_static_scratch(table.handle, ids.data_ptr(), int(ids.numel()), x.data_ptr(), x.stride(0),
                                         y.data_ptr(), y.stride(0), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["decode", "decode_delta_only", "tiny", "prefill", "stacked_qkv_128"])
def test_static_scratch_matches_the_workspace_path_on_consecutive_calls(name):
    if name == "decode":
        p = synth.decode(1, y_base="random")
    elif name == "decode_delta_only":
        p = synth.decode(7, y_base="zero")
    elif name == "tiny":
        p = synth.tiny(0, y_base="xw")
    elif name == "prefill":
        p = synth.prefill(2, y_base="random")
    else:   # 128 tokens of the stacked batch keep the three-slice QKV within the fixed array
        q = synth.stacked("qkv", y_base="zero")
        p = synth.DenseProblem(**{**q.__dict__})
        p.ids, p.x, p.y_base, p.M = q.ids[384:512], q.x[384:512], q.y_base[384:512], 128
    table = pack_dense(p)
    y_ref, _, ws = run_dense(p, table=table)
    assert lora.lora_get_status(ws) == lora.LORA_OK
    ref = host_f64(y_ref)
    ids = torch.from_numpy(p.ids).cuda()
    x = dev_bf16(p.x)
    for call in range(2):
        y = dev_bf16(p.y_base)
        assert static_apply(table, ids, x, y) == lora.LORA_OK
        torch.cuda.synchronize()
        check_close(host_f64(y), ref, "%s call %d" % (name, call))
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
