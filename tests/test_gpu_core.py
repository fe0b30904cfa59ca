"""GPU parity of the CUDA-core coarse path (batches of up to 4 rows) against the CPU oracle.

The path builds each fp32 weight from the packed bits with integer ops and accumulates x w with
fp32 FMAs; every forward here runs it through dh_forward_debug and applies all of parity.py's
checks (coarse values, block candidates, the top-R selection, exact values, indices).  The
sizes reach the kernel's edges: M padded to 1, 2 and 4 rows, ragged tail blocks, KCAND 1..64,
H from one chunk per plane (512) to 5120, and heads with more blocks than the grid has warps,
so that warps take several items from the work counter.
"""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth

from parity import full_compare, gpu_forward, gpu_quantize, rows_compare
from test_gpu_outliers import wide_range_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


def _inputs(M, H, V, seed=0, **kw):
    wl = synth.custom(M, H, V, **kw)
    return synth.make_x(wl, seed, DEV), synth.make_w(wl, seed, DEV)


def test_core_path_takes_small_batches_only():
    prev = dh.dh_set_coarse_path(dh.PATH_CORE)
    try:
        for M in (1, 2, 3, 4):
            assert dh.dh_coarse_path_for(M) == dh.PATH_CORE
        for M in (5, 16):
            try:
                got = dh.dh_coarse_path_for(M)
            except dh.DHError:
                got = None
            assert got != dh.PATH_CORE
    finally:
        dh.dh_set_coarse_path(prev)


@pytest.mark.parametrize("M, H, V, kcand, rerank, topk", [
    (1, 1024, 8192, 8, 32, 1),          # the tiny workload's sizes
    (2, 512, 3017, 8, 32, 4),           # one chunk per plane, tail block of 9
    (3, 1536, 4099, 3, 40, 5),          # M padded to 4, tail block of 3 < kcand
    (4, 5120, 40037, 8, 32, 1),         # the full width, 626 blocks, ragged tail
    (1, 512, 70, 64, 70, 7),            # whole blocks as candidates, rerank everything
    (4, 2048, 1, 1, 1, 1),              # a one-row head
    (1, 512, 200003, 8, 32, 16),        # 3126 blocks: more than the grid's warps
    (2, 1024, 130005, 8, 64, 16),       # 2032 blocks, the two-launch selection (R = 64)
    (4, 512, 100029, 2, 32, 4),         # 1563 blocks with 8 warps per CTA
])
def test_core_forward(M, H, V, kcand, rerank, topk):
    x, W = _inputs(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    packed, S, ZS = gpu_quantize(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, rerank, topk, path=dh.PATH_CORE)
    print((M, H, V, kcand, rerank, topk), rep["coarse_worst"], rep["exact_worst"],
          "tie rows", len(rep["ties"]))


def test_core_wide_range_rows():
    """A 2^10 outlier, a 2^12 outlier, a row spanning 2^-20 .. 2^4 and an RMS-normalised row
    with 100x channels: the fold's rescaling of plane 0 by 64 stays inside the tolerance."""
    M, H, V = 4, 5120, 40000 + 37
    wl = synth.custom(M, H, V, hot_rows=V // 50, hot_scale=4.0)
    W = synth.make_w(wl, 0, DEV)
    x = wide_range_rows(M, H)
    packed, S, ZS = gpu_quantize(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, 8, 32, 4, path=dh.PATH_CORE)
    print("core wide-range", rep["coarse_worst"], rep["exact_worst"], "tie rows", len(rep["ties"]))


@pytest.mark.parametrize("M", [1, 4])
def test_core_full_head_sampled(M):
    """The full 248320 x 5120 head (the small-M points of the sweep): every check on the whole
    batch against the oracle's full path for these rows."""
    wl = synth.full(M)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    prev = dh.dh_set_coarse_path(dh.PATH_CORE)
    try:
        gpu = gpu_forward(x, packed, S, ZS, W, 8, 32, 1)
    finally:
        dh.dh_set_coarse_path(prev)
    rep, _ = rows_compare(gpu, np.arange(M), x, W, packed, S, ZS, 8, 32, 1)
    print("core full head M", M, rep["coarse_worst"], "tie rows", len(rep["ties"]))

