"""GPU parity of the 8-bit tcgen05 path at the widest hidden sizes it takes.

At H = 8192 the tile's S/ZS copies leave room for fewer TMA stages, above 7168 the batch runs in
16-row launches whatever its size, and above 8192 the x staging kernel holds a second 16-byte
slice of the row per thread.  Each case runs every check of
parity.py against the oracle on the tcgen05 path explicitly; a size the path does not take is
skipped (the automatic choice would run another path there).
"""
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth

from parity import full_compare, gpu_quantize

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


@pytest.mark.parametrize("M, H, V, kcand, rerank, topk", [
    (16, 8192, 20000 + 37, 8, 32, 1),   # fewer stages; 157 tiles: some CTAs run two
    (33, 6144, 9000, 8, 32, 4),         # 32-row and 16-row launches at H = 6144
    (16, 12288, 9000, 8, 32, 1),        # the staging kernel's second slice per thread
    (40, 8192, 9000 + 5, 8, 32, 4),     # wider than a 32-row launch holds: 16 + 16 + 8 rows
])
def test_wide_rows_on_the_tensor_path(M, H, V, kcand, rerank, topk):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    try:
        rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, rerank, topk, path=dh.PATH_TC)
    except dh.DHError as e:
        pytest.skip(f"the tcgen05 path does not take M={M}, H={H}: {e}")
    print((M, H, V), rep["coarse_worst"], rep["exact_worst"], "tie rows", len(rep["ties"]))
