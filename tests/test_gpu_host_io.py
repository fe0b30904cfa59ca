"""GPU tests of dh_forward_host: x, idx and logit in pinned host memory.

The call runs the same kernels as dh_forward; on the 8-bit tcgen05 path the staging kernel
reads x across the host link and keeps a device copy for the rerank, on the other coarse paths
x is copied to the device first, and the last kernel writes idx and logit into the host
buffers.  Each case checks the host results bit for bit against dh_forward on the same inputs
and, for the full comparison, against the oracle's forward.  Unpinned host buffers are
rejected before anything runs.
"""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth
from oracle import oracle as orc

from parity import check_result, gpu_quantize, host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


def _both(M, H, V, kcand, R, topk, path=None, seed=0):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, seed, DEV), synth.make_w(wl, seed, DEV)
    packed, S, ZS = gpu_quantize(W)
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, kcand, R), dtype=torch.uint8, device=DEV)
    idx = torch.empty(M, topk, dtype=torch.int32, device=DEV)
    logit = torch.empty(M, topk, dtype=torch.float32, device=DEV)
    xh = x.cpu().pin_memory()
    ih = torch.full((M, topk), -7, dtype=torch.int32).pin_memory()
    lh = torch.full((M, topk), float("nan"), dtype=torch.float32).pin_memory()
    prev = dh.dh_set_coarse_path(path) if path is not None else None
    try:
        dh.dh_forward(x, packed, S, ZS, W, kcand, R, topk, idx, logit, ws)
        torch.cuda.synchronize()
        ws.random_(0, 255)                       # nothing may carry over from the first call
        dh.dh_forward_host(xh, packed, S, ZS, W, kcand, R, topk, ih, lh, ws)
        torch.cuda.synchronize()
    finally:
        if prev is not None:
            dh.dh_set_coarse_path(prev)
    assert dh.dh_device_status(reset=True) == 0
    assert torch.equal(ih, idx.cpu())
    assert torch.equal(lh.view(torch.int32), logit.cpu().view(torch.int32))
    return x, W, packed, S, ZS, ih.numpy(), lh.numpy()


@pytest.mark.parametrize("M, H, V, kcand, R, topk", [
    (16, 5120, 40000 + 37, 8, 32, 1),     # the default path, fused selection, ragged tail
    (33, 1536, 6144, 4, 24, 5),           # two staging chunks (32 + 16 rows)
    (72, 1024, 9000, 8, 64, 16),          # three chunks; the two-launch selection (R = 64)
    (1, 512, 70, 64, 70, 7),              # whole blocks as candidates, everything reranked
])
def test_host_buffers_match_device_buffers(M, H, V, kcand, R, topk):
    _both(M, H, V, kcand, R, topk)


@pytest.mark.parametrize("path", [dh.PATH_WARP, dh.PATH_CORE])
def test_host_buffers_on_the_copy_paths(path):
    """Coarse paths without the staging kernel's copy: x goes to the device by one copy."""
    try:
        _both(4, 1024, 8192 + 37, 8, 32, 4, path=path)
    except dh.DHError as e:
        pytest.skip(f"path {path} does not take these sizes: {e}")


def test_host_buffers_against_the_oracle():
    M, H, V, kcand, R, topk = 8, 2048, 20000 + 9, 8, 32, 4
    x, W, packed, S, ZS, ih, lh = _both(M, H, V, kcand, R, topk, seed=3)
    ref = orc.forward(host(x), host(packed), host(S), host(ZS), host(W), kcand, R, topk)
    check_result({"idx": ih, "logit": lh}, ref, kcand, topk, host(x), host(W))


def test_unpinned_host_buffers_are_rejected():
    M, H, V, kcand, R, topk = 2, 512, 1000, 8, 32, 1
    wl = synth.custom(M, H, V)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, kcand, R), dtype=torch.uint8, device=DEV)
    xh = x.cpu()                                  # pageable
    ih = torch.empty(M, topk, dtype=torch.int32).pin_memory()
    lh = torch.empty(M, topk, dtype=torch.float32).pin_memory()
    args = [dh._p(xh), dh._p(packed), dh._p(S), dh._p(ZS), dh._p(W), M, H, V, kcand, R, topk,
            dh._p(ih), dh._p(lh), dh._p(ws), ws.numel()]
    rc = dh._load().dh_forward_host(*args, dh._stream(None))
    assert rc == -8                               # DH_ERR_ARG
    assert "pinned" in dh.dh_last_error()
    with pytest.raises(ValueError):
        dh.dh_forward_host(xh, packed, S, ZS, W, kcand, R, topk, ih, lh, ws)
    torch.cuda.synchronize()
    assert dh.dh_device_status(reset=True) == 0


def test_draft_head_takes_a_pinned_host_x():
    M, H, V = 5, 1024, 9000 + 13
    wl = synth.custom(M, H, V, hot_rows=V // 50, hot_scale=4.0)
    x, W = synth.make_x(wl, 1, DEV), synth.make_w(wl, 1, DEV)
    head = dh.DraftHead(W, kcand=8, rerank=32)
    idx, logit = head.forward(x, topk=4)
    hidx, hlogit = head.forward(x.cpu().pin_memory(), topk=4)
    assert not hidx.is_cuda and hidx.is_pinned()
    assert torch.equal(hidx, idx.cpu())
    assert torch.equal(hlogit.view(torch.int32), logit.cpu().view(torch.int32))
    with pytest.raises(ValueError):
        head.forward(x.cpu(), topk=4)                # pageable
