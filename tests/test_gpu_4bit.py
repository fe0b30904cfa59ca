"""GPU parity of the 4-bit head (the page's BITS = 4 variant: 15 levels, half-split packing,
bias 16): dh_quantize4 bit-exact with the oracle's quantiser, and dh_forward4 judged by the
rules in parity.py against the oracle's 4-bit forward, on the sizes and KCAND values the
variant is used with (KCAND = 1 is the page's 4-bit setting)."""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth
from oracle import oracle as orc

from parity import full_compare, gpu_forward, host, check_coarse, rows_compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


def _quantize4(W):
    V, H = W.shape
    packed = torch.empty(V, H // 2, dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // 128, dtype=torch.bfloat16, device=DEV)
    ZS = torch.empty_like(S)
    dh.dh_quantize4(W, packed, S, ZS)
    return packed, S, ZS


@pytest.mark.parametrize("V, H", [(4096, 1024), (1000, 512), (2003, 1536), (777, 5120), (1, 512)])
def test_quantize4_bit_exact(V, H):
    wl = synth.custom(1, H, V, hot_rows=min(V, 37), hot_scale=4.0)
    W = synth.make_w(wl, 0, DEV)
    W[0, :128] = 0.25                                   # constant group
    if V > 2:
        W[1, 128:256] = W[1, 128:256].abs() + 0.01      # all-positive group
        W[2, :128] = -W[2, :128].abs() - 0.01           # all-negative group
    packed, S, ZS = _quantize4(W)
    torch.cuda.synchronize()
    rp, rS, rZS = orc.quantize4(host(W))
    assert np.array_equal(host(packed), rp)
    assert np.array_equal(host(S), rS)
    assert np.array_equal(host(ZS), rZS)


@pytest.mark.parametrize("M, H, V, kcand, R, k", [
    (1, 1024, 8192, 1, 32, 1),            # the page's 4-bit setting: KCAND = 1
    (5, 1024, 8192 + 37, 1, 32, 4),       # ragged tail block
    (16, 5120, 12288 + 64 * 3 + 5, 1, 32, 1),
    (16, 2048, 16384, 8, 32, 1),          # KCAND = 8 on the 4-bit head
    (32, 5120, 4096, 1, 32, 1),           # two launches of 16 rows
    (33, 1536, 6144, 4, 24, 5),           # three batch chunks (16 + 16 + 1 rows)
    (64, 1024, 4096, 8, 64, 16),          # RERANK 64, top-16
    (16, 5120, 40000 + 37, 1, 32, 1),     # 313 tiles of 128 rows: every CTA runs two or more
    (128, 1024, 4096 + 64 * 2 + 9, 1, 32, 1),  # eight 16-row chunks: one staging launch for all
    (113, 512, 3000, 4, 32, 3),           # eight chunks, the last of one row
])
def test_forward4_matches_the_oracle(M, H, V, kcand, R, k):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = _quantize4(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, k, bits=4)
    print("4-bit", M, H, V, kcand, rep["coarse_worst"], rep["exact_worst"], "tie rows",
          len(rep["ties"]), "differing", sum(t[4] for t in rep["ties"]))


def test_forward4_rejects_sizes_and_paths_it_cannot_run():
    M, H, V = 32, 16384, 4096                           # 64 blocks: 64 valid candidates
    x = torch.zeros(M, H, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(V, H, dtype=torch.bfloat16, device=DEV)
    packed, S, ZS = _quantize4(W)
    nws = dh.dh_workspace_bytes(M, H, V, 1, 32)
    assert nws > 0
    ws = torch.empty(nws, dtype=torch.uint8, device=DEV)
    idx = torch.empty(M, 1, dtype=torch.int32, device=DEV)
    logit = torch.empty(M, 1, dtype=torch.float32, device=DEV)
    with pytest.raises(dh.DHError) as e:  # at H = 16384 the S / ZS tile copies alone need 128 KB
        dh.dh_forward4(x, packed, S, ZS, W, 1, 32, 1, idx, logit, ws)
    assert e.value.code == -8
    prev = dh.dh_set_coarse_path(dh.PATH_WARP)
    try:
        with pytest.raises(dh.DHError) as e:
            dh.dh_forward4(x[:4], packed, S, ZS, W, 1, 32, 1, idx[:4], logit[:4], ws)
        assert e.value.code == -8
    finally:
        dh.dh_set_coarse_path(prev)
    torch.cuda.synchronize()
    assert dh.dh_device_status(reset=True) == 0


def test_draft_head_class_builds_the_4bit_head():
    M, H, V = 3, 1024, 4096
    wl = synth.custom(M, H, V)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    head = dh.DraftHead(W, kcand=1, rerank=32, bits=4)
    idx, logit = head.forward(x, topk=2)
    packed, S, ZS = _quantize4(W)
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, 1, 32), dtype=torch.uint8, device=DEV)
    i2 = torch.empty_like(idx)
    l2 = torch.empty_like(logit)
    dh.dh_forward4(x, packed, S, ZS, W, 1, 32, 2, i2, l2, ws)
    torch.cuda.synchronize()
    assert torch.equal(head.packed, packed)
    assert torch.equal(idx, i2) and torch.equal(logit, l2)


def test_forward4_full_head_sampled():
    """The 4-bit head at full size (M=16, H=5120, V=248320, KCAND 1): coarse values of 2000
    sampled vocabulary rows (plus every reranked one and the last) for the whole batch against
    the oracle's 4-bit coarse value, then three whole batch rows through the oracle's path."""
    wl = synth.full(16)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = _quantize4(W)
    gpu = gpu_forward(x, packed, S, ZS, W, 1, 32, 1, bits=4)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([rng.choice(wl.V, 2000, replace=False),
                                     gpu["sel_idx"].ravel(), [wl.V - 1]]))
    rows_t = torch.from_numpy(rows).to(DEV)
    ref_c = orc.coarse4(host(x), host(packed[rows_t]), host(S[rows_t]), host(ZS[rows_t]))
    worst = check_coarse(gpu["coarse"][:, rows], ref_c)
    rep, _ = rows_compare(gpu, [0, 7, 15], x, W, packed, S, ZS, 1, 32, 1, bits=4)
    print("4-bit full head: sampled coarse worst", worst, "rows", rep["coarse_worst"],
          "tie rows", len(rep["ties"]))
