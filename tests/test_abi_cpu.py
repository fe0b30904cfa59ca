"""Host-side tests of the C ABI (no GPU needed): the library builds, loads, exports every
entry point declared in include/dh.h, and rejects bad arguments before launching anything.

Invalid calls must return their status without touching the device, so these run on a
machine without a GPU (fake, never dereferenced device addresses are passed).
"""
import ctypes
import os
import re

import pytest

import quantised_speculative_draft_gb300 as dh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dh.h")

FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    dh.build()
    return dh._load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dh_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for must in ("dh_quantize", "dh_workspace_bytes", "dh_forward", "dh_forward_debug",
                 "dh_forward_timed", "dh_set_coarse_path", "dh_coarse_path_for",
                 "dh_device_status", "dh_last_error", "dh_version"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(dh.library_path())
    for name in declared_functions():
        assert hasattr(so, name), f"{name} declared in dh.h but not exported"


def test_version(lib):
    assert dh.dh_version() >> 16 == 1


def _fwd(lib, M=4, H=1024, V=8192, kcand=8, rerank=32, topk=1, ws=1 << 40, **ptrs):
    p = dict(x=FAKE, packed=FAKE, scales=FAKE, zeros=FAKE, W=FAKE, idx=FAKE, logit=FAKE,
             ws=FAKE)
    if "ws_ptr" in ptrs:
        p["ws"] = ptrs.pop("ws_ptr")
    p.update(ptrs)
    return lib.dh_forward(p["x"], p["packed"], p["scales"], p["zeros"], p["W"], M, H, V, kcand,
                          rerank, topk, p["idx"], p["logit"], p["ws"], ws, None)


@pytest.mark.parametrize("kw, code", [
    (dict(x=None), -1), (dict(W=None), -1), (dict(ws=None), -1), (dict(idx=None), -1),
    (dict(M=0), -2), (dict(M=129), -2), (dict(H=256), -2), (dict(H=1000), -2), (dict(H=0), -2),
    (dict(V=0), -2),
    (dict(kcand=0), -3), (dict(kcand=65), -3),
    (dict(rerank=0), -3), (dict(rerank=1025), -3), (dict(topk=0), -3), (dict(topk=33), -3),
    (dict(V=100, kcand=64, rerank=101), -3),   # 64 + 36 valid candidates
    (dict(V=100, kcand=8, rerank=17), -3),     # 8 + 8 valid candidates
    (dict(x=FAKE + 8), -5), (dict(packed=FAKE + 4), -5), (dict(ws=FAKE + 2), -5),
    (dict(wsbytes=16), -4),
])
def test_forward_rejects_bad_arguments_before_launch(lib, kw, code):
    wsbytes = kw.pop("wsbytes", 1 << 40)
    rc = _fwd(lib, ws=wsbytes, **{("ws_ptr" if k == "ws" else k): v for k, v in kw.items()})
    assert rc == code, dh.dh_last_error()
    assert dh.dh_last_error() != ""


def test_boundary_selection_parameters_are_accepted_by_the_checks(lib):
    # V=100, kcand=64: exactly 100 valid candidates -> rerank 100 passes the checks and only
    # fails later on the (fake) workspace size
    assert _fwd(lib, V=100, kcand=64, rerank=100, topk=100, ws=16) == -4
    assert _fwd(lib, V=8192, kcand=8, rerank=1024, topk=1024, ws=16) == -4


def test_workspace_bytes(lib):
    assert dh.dh_workspace_bytes(1, 1024, 8192, 8, 32) > 0
    assert dh.dh_workspace_bytes(0, 1024, 8192, 8, 32) == 0
    assert dh.dh_workspace_bytes(1, 1000, 8192, 8, 32) == 0
    assert dh.dh_workspace_bytes(1, 1024, 8192, 8, 5000) == 0
    small = dh.dh_workspace_bytes(16, 5120, 124160, 8, 32)
    big = dh.dh_workspace_bytes(72, 5120, 248320, 8, 32)
    assert 0 < small < big
    # candidates dominate: M * nblk * kcand * 8 bytes
    assert big >= 72 * 3880 * 8 * 8


def test_quantize_rejects_bad_arguments(lib):
    q = lib.dh_quantize
    assert q(None, 10, 1024, FAKE, FAKE, FAKE, None) == -1
    assert q(FAKE, 0, 1024, FAKE, FAKE, FAKE, None) == -2
    assert q(FAKE, 10, 768, FAKE, FAKE, FAKE, None) == -2
    assert q(FAKE, 10, 1024, FAKE + 1, FAKE, FAKE, None) == -5


def test_forward_debug_and_timed_reject_bad_optional_pointers(lib):
    args = [FAKE] * 5 + [4, 1024, 8192, 8, 32, 1, FAKE, FAKE, FAKE, 1 << 40]
    assert lib.dh_forward_debug(*args, FAKE + 4, None, None, None, None, None) == -5
    assert lib.dh_forward_timed(*args, None, None) == -1
    arr = (ctypes.c_void_p * 6)(*([FAKE] * 5 + [0]))
    assert lib.dh_forward_timed(*args, arr, None) == -1


def test_coarse_path_setting(lib):
    prev = dh.dh_set_coarse_path(dh.PATH_WARP)
    try:
        assert dh.dh_coarse_path_for(16) == dh.PATH_WARP
        with pytest.raises(dh.DHError):
            dh.dh_set_coarse_path(7)
        with pytest.raises(dh.DHError):
            dh.dh_coarse_path_for(0)
    finally:
        dh.dh_set_coarse_path(prev)


def test_product_path_never_touches_the_oracle():
    """The CUDA library and its binding import, link and call nothing under oracle/."""
    pkg = os.path.join(ROOT, "quantised_speculative_draft_gb300")
    bad = re.compile(r"import\s+oracle|from\s+oracle|liboracle|dh_oracle|orc_[a-z]")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not bad.search(src), f


def test_fp8_head_entry_points_reject_bad_arguments(lib):
    # dh_quantize_fp8(W8, row_scale, V, H, packed, scales, zeros, stream)
    assert lib.dh_quantize_fp8(FAKE, None, 16, 1024, FAKE, FAKE, FAKE, None) == -1
    assert lib.dh_quantize_fp8(FAKE, FAKE, 16, 1000, FAKE, FAKE, FAKE, None) == -2
    assert lib.dh_quantize_fp8(FAKE, FAKE, 0, 1024, FAKE, FAKE, FAKE, None) == -2
    assert lib.dh_quantize_fp8(FAKE, FAKE + 2, 16, 1024, FAKE, FAKE, FAKE, None) == -5
    assert lib.dh_quantize_fp8(FAKE + 8, FAKE, 16, 1024, FAKE, FAKE, FAKE, None) == -5
    # dh_forward_fp8w(x, packed, S, ZS, W8, row_scale, M, H, V, kcand, R, k, idx, logit, ws, n)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1024, 8192, 8, 32, 1, FAKE, FAKE, FAKE,
            1 << 40, None]
    bad = list(args)
    bad[5] = None
    assert lib.dh_forward_fp8w(*bad) == -1
    bad = list(args)
    bad[5] = FAKE + 2
    assert lib.dh_forward_fp8w(*bad) == -5
    bad = list(args)
    bad[7] = 1000
    assert lib.dh_forward_fp8w(*bad) == -2
    bad = list(args)
    bad[11] = 33
    assert lib.dh_forward_fp8w(*bad) == -3
    bad = list(args)
    bad[15] = 16
    assert lib.dh_forward_fp8w(*bad) == -4


def test_4bit_head_entry_points_reject_bad_arguments(lib):
    assert lib.dh_quantize4(FAKE, 16, 1024, None, FAKE, FAKE, None) == -1
    assert lib.dh_quantize4(FAKE, 16, 768, FAKE, FAKE, FAKE, None) == -2   # H % 512
    assert lib.dh_quantize4(FAKE + 4, 16, 1024, FAKE, FAKE, FAKE, None) == -5
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1024, 8192, 1, 32, 1, FAKE, FAKE, FAKE, 1 << 40,
            None]
    bad = list(args)
    bad[4] = None
    assert lib.dh_forward4(*bad) == -1
    bad = list(args)
    bad[6] = 1000
    assert lib.dh_forward4(*bad) == -2
    bad = list(args)
    bad[14] = 16
    assert lib.dh_forward4(*bad) == -4
    # the debug twin checks its optional outputs' alignment
    assert lib.dh_forward4_debug(*args[:15], FAKE + 4, None, None, None, None, None) == -5


def test_c4_entry_points_reject_bad_arguments(lib):
    assert lib.dh_quantize_c4(FAKE, 16, 1024, None, FAKE, FAKE, None) == -1
    assert lib.dh_quantize_c4(FAKE, 16, 768, FAKE, FAKE, FAKE, None) == -2
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1024, 8192, 8, 32, 1, FAKE, FAKE, FAKE, 1 << 40]
    assert lib.dh_forward_c4_debug(*args, FAKE + 4, None, None, None, None, None, None) == -5
    events = (ctypes.c_void_p * 6)(FAKE, FAKE, None, FAKE, FAKE, FAKE)
    assert lib.dh_forward_c4_debug(*args, None, None, None, None, None, events, None) == -1
    bad = list(args)
    bad[6] = 1000
    assert lib.dh_forward_c4_debug(*bad, None, None, None, None, None, None, None) == -2


def test_g64_entry_points_reject_bad_arguments(lib):
    assert lib.dh_quantize_g64(FAKE, 16, 1024, None, FAKE, FAKE, None) == -1
    assert lib.dh_quantize_g64(FAKE, 16, 768, FAKE, FAKE, FAKE, None) == -2
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1024, 8192, 8, 32, 1, FAKE, FAKE, FAKE, 1 << 40]
    assert lib.dh_forward_g64_debug(*args, FAKE + 4, None, None, None, None, None, None) == -5
    bad = list(args)
    bad[10] = 0
    assert lib.dh_forward_g64_debug(*bad, None, None, None, None, None, None, None) == -3


def test_wside_entry_point_rejects_bad_arguments(lib):
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1024, 8192, 8, 32, 1, FAKE, FAKE, FAKE, 1 << 40]
    assert lib.dh_forward_wside_debug(*args, FAKE + 4, None, None, None, None, None, None) == -5
    bad = list(args)
    bad[3] = None
    assert lib.dh_forward_wside_debug(*bad, None, None, None, None, None, None, None) == -1


def test_draft_head_rejects_bad_heads_on_the_host():
    import torch
    W = torch.zeros(64, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        dh.DraftHead(W, bits=3)                                   # no such width
    with pytest.raises(ValueError):
        dh.DraftHead(W.to(torch.uint8), bits=4, row_scale=torch.ones(64))  # 4-bit fp8 head
    with pytest.raises(ValueError):
        dh.DraftHead(W)                                           # not a CUDA tensor
    with pytest.raises(ValueError):
        dh.DraftHead(W.to(torch.uint8), row_scale=torch.ones(64))  # fp8 head off the device


def test_forward_host_rejects_missing_buffers_before_any_cuda_call(lib):
    # dh_forward_host(x, packed, scales, zeros, W, M, H, V, kcand, rerank, topk, idx, logit,
    #                 workspace, ws_bytes, stream): NULL host buffers or workspace -> -1
    args = [FAKE] * 5 + [4, 1024, 8192, 8, 32, 1, FAKE, FAKE, FAKE, 1 << 40]
    for i in (0, 11, 12, 13):
        bad = list(args)
        bad[i] = None
        assert lib.dh_forward_host(*bad, None) == -1


def test_every_width_up_to_14336_has_a_coarse_path(lib):
    """Launch counts (staging + coarse launches + selection) from the host-side plan: the 8-bit
    path runs 32-row launches up to H = 7168 and 16-row launches above, at any batch size; wider
    rows have no path, and the forward refuses them before any CUDA call."""
    count = dh.dh_forward_launch_count
    assert count(100, 5120, 248320, 8, 32) == 1 + 4 + 1      # 32 + 32 + 32 + 4 rows
    assert count(100, 8192, 248320, 8, 32) == 1 + 7 + 1      # 16-row launches
    assert count(128, 14336, 248320, 8, 32) == 1 + 8 + 1
    assert count(1, 16384, 248320, 8, 32) == 0
    args = [FAKE] * 5 + [4, 16384, 8192, 8, 32, 1, FAKE, FAKE, FAKE, 1 << 40]
    assert lib.dh_forward(*args, None) == -8
    assert "no coarse path" in dh.dh_last_error()
