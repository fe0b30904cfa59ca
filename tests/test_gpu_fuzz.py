"""GPU parity on seeded random configurations: every check of parity.py against the oracle.

The hand-picked cases elsewhere cover the edges one at a time; these draw the batch size,
hidden size, vocabulary size, KCAND, RERANK and top-k together (seed 2024), on whichever coarse
path the library chooses for the sizes, so that combinations nobody wrote down are exercised
too: ragged tail blocks with small KCAND, RERANK above 32 (the radix selection and the
standalone rerank) next to batch chunks, wide rows with small heads.  The product M H V is
capped so that the oracle finishes each case in seconds.
"""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth

from parity import full_compare, gpu_quantize

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _valid_candidates(V, kcand):
    full, tail = divmod(V, 64)
    return full * kcand + min(tail, kcand)


def _cases(n=14, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 17, 24, 32, 33, 48, 64, 72, 100, 128]))
        H = 512 * int(rng.integers(1, 17))
        V = int(rng.integers(64, 30000))
        if M * H * V > 4e9:
            continue
        kcand = int(rng.integers(1, 65))
        top = min(_valid_candidates(V, kcand), 1024, V)
        if rng.random() < 0.6:
            R = int(rng.integers(1, min(top, 32) + 1))
        else:
            R = int(rng.integers(1, top + 1))
        topk = int(rng.integers(1, min(R, 32) + 1))
        out.append((M, H, V, kcand, R, topk))
    return out


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


@pytest.mark.parametrize("M, H, V, kcand, R, topk", _cases())
def test_random_configuration(M, H, V, kcand, R, topk):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, M + V, DEV), synth.make_w(wl, H + V, DEV)
    packed, S, ZS = gpu_quantize(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, topk)
    print((M, H, V, kcand, R, topk), "path", dh.dh_coarse_path_for(M), rep["coarse_worst"],
          rep["exact_worst"], "tie rows", len(rep["ties"]))
