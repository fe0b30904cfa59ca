"""GPU parity of the weight-side dequant variant (the page's scale-placement ablation): the
forward whose coarse pass dots x with bf16(S (1 + v/4) - ZS) per weight, judged by the rules in
parity.py against the oracle's weight-side forward, and its coarse values against the
activation-side head within the coarse tolerance."""
import numpy as np
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


@pytest.mark.parametrize("M, H, V, kcand, R, k", [
    (1, 1024, 8192, 8, 32, 1),
    (5, 1024, 8192 + 37, 8, 32, 4),       # ragged tail block
    (16, 5120, 12288, 8, 32, 1),
    (40, 1536, 6144, 4, 24, 5),           # N = 48 launch
    (16, 5120, 40000 + 37, 8, 32, 1),     # 313 tiles of 128 rows: every CTA runs two or more
])
def test_forward_wside_matches_the_oracle(M, H, V, kcand, R, k):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = gpu_quantize(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, k, bits="wside")
    print("wside", M, H, V, rep["coarse_worst"], "tie rows", len(rep["ties"]))
