"""The C-ABI library builds, loads and exports every entry point include/lora.h
declares; host-only calls behave without a GPU (no compute is launched here)."""
import ctypes
import os
import re

import pytest

from segmented_rank_gemm_lora_gb300 import build_lib, lora

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return lora.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "lora.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary_calls():
    names = header_functions()
    for n in ("lora_pack_weights", "lora_build_segments", "lora_apply", "lora_moe_delta", "lora_get_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(lora.EXPORTED) == names


def test_rank_padding_matches_the_pages(lib):
    rows = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "p1_rank_padding.txt"))
            if l.strip() and not l.startswith("#")]
    for r, pad in rows:
        assert lora.lora_rank_padded(int(r)) == int(pad)
    assert [lora.lora_rank_padded(r) for r in (1, 8, 17, 48, 64)] == [16, 16, 32, 48, 64]
    assert lora.lora_rank_padded(0) == -1 and lora.lora_rank_padded(65) == -1


def test_workspace_sizes(lib):
    a = lora.lora_workspace_bytes(32, 20)
    b = lora.lora_workspace_bytes(2048, 20)
    c = lora.lora_workspace_bytes(512, 8, 2, 8, 64)
    assert 0 < a < b and c > 0 and c % 256 == 0
    assert lora.lora_workspace_bytes(0, 4) == 0
    assert lora.lora_workspace_bytes(16, 0) == 0
    assert lora.lora_workspace_bytes(16, 4, 0, 8, 64) == 0


def test_options_roundtrip_and_validation(lib):
    old = lora.lora_get_option(lora.LORA_OPT_WAIT_TIMEOUT_NS)
    lora.lora_set_option(lora.LORA_OPT_WAIT_TIMEOUT_NS, 5_000_000)
    assert lora.lora_get_option(lora.LORA_OPT_WAIT_TIMEOUT_NS) == 5_000_000
    lora.lora_set_option(lora.LORA_OPT_WAIT_TIMEOUT_NS, old)
    assert lora.lora_get_option(lora.LORA_OPT_PDL) == 1          # on by default
    lora.lora_set_option(lora.LORA_OPT_PDL, 0)
    assert lora.lora_get_option(lora.LORA_OPT_PDL) == 0
    lora.lora_set_option(lora.LORA_OPT_PDL, 1)
    with pytest.raises(lora.LoraError):
        lora.lora_set_option(lora.LORA_OPT_PDL, 2)
    with pytest.raises(lora.LoraError):
        lora.lora_set_option(lora.LORA_OPT_PATH, 7)
    with pytest.raises(lora.LoraError):
        lora.lora_set_option(99, 1)


def test_status_strings(lib):
    for code in lora.STATUS:
        assert lora.lora_status_string(code)


def test_argument_errors_launch_nothing(lib):
    h = ctypes.c_void_p()
    sh = lora.ProjShape()
    assert lib.lora_pack_weights(None, 0, ctypes.byref(sh), None, ctypes.byref(h)) == lora.LORA_ERR_INVALID_ARG
    assert lib.lora_apply(None, None, None, 0, None, 0, None) == lora.LORA_ERR_INVALID_ARG
    assert lib.lora_build_segments(None, None, 0, None, None, None) == lora.LORA_ERR_INVALID_ARG
    ws = lora.WorkspaceDesc(0x1000, lora.lora_workspace_bytes(16, 4), 16, 4, 0, 0, 0)
    assert lib.lora_build_segments(ctypes.byref(ws), None, 4, None, None, None) == lora.LORA_ERR_INVALID_ARG
    small = lora.WorkspaceDesc(0x1000, 64, 16, 4, 0, 0, 0)
    assert lib.lora_build_segments(ctypes.byref(small), None, 0, None, None, None) == lora.LORA_ERR_WORKSPACE
    assert lib.lora_table_info(None, None) == lora.LORA_ERR_INVALID_ARG
