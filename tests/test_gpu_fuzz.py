"""GPU parity on seeded random configurations: every check of parity.py against the oracle.

The hand-picked cases elsewhere cover the edges one at a time; these draw the batch size,
hidden size, vocabulary size, KCAND, RERANK and top-k together (seeded), on whichever coarse
path the library chooses for the sizes -- for the bf16 2-bit head, the 4-bit head and the fp8
head -- so that combinations nobody wrote down are exercised
too: ragged tail blocks with small KCAND, RERANK above 32 (the radix selection and the
standalone rerank) next to batch chunks, wide rows with small heads.  The product M H V is
capped so that the oracle finishes each case in seconds.
"""
import numpy as np
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth

from oracle import oracle as orc
from parity import check_result, full_compare, gpu_quantize, host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _valid_candidates(V, kcand):
    full, tail = divmod(V, 64)
    return full * kcand + min(tail, kcand)


def _cases(n=14, seed=2024, max_h=8192):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 17, 24, 32, 33, 48, 64, 72, 100, 128]))
        H = 512 * int(rng.integers(1, max_h // 512 + 1))
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


@pytest.mark.parametrize("M, H, V, kcand, R, topk", _cases() + _cases(8, seed=7, max_h=15360))
def test_random_configuration(M, H, V, kcand, R, topk):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, M + V, DEV), synth.make_w(wl, H + V, DEV)
    packed, S, ZS = gpu_quantize(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, topk)
    print((M, H, V, kcand, R, topk), "path", dh.dh_coarse_path_for(M), rep["coarse_worst"],
          rep["exact_worst"], "tie rows", len(rep["ties"]))


@pytest.mark.parametrize("M, H, V, kcand, R, topk", _cases(6, seed=11, max_h=11264))
def test_random_configuration_4bit_head(M, H, V, kcand, R, topk):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, M + V, DEV), synth.make_w(wl, H + V, DEV)
    packed = torch.empty(V, H // 2, dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // 128, dtype=torch.bfloat16, device=DEV)
    ZS = torch.empty_like(S)
    dh.dh_quantize4(W, packed, S, ZS)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, topk, bits=4)
    print((M, H, V, kcand, R, topk), "4-bit", rep["coarse_worst"], "tie rows", len(rep["ties"]))


@pytest.mark.parametrize("M, H, V, kcand, R, topk", _cases(6, seed=13))
def test_random_configuration_fp8_head(M, H, V, kcand, R, topk):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x = synth.make_x(wl, M + V, DEV)
    W8, rs = synth.make_w_fp8(wl, H + V, DEV)
    packed = torch.empty(V, H // 4, dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // 128, dtype=torch.bfloat16, device=DEV)
    ZS = torch.empty_like(S)
    dh.dh_quantize_fp8(W8, rs, packed, S, ZS)
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, kcand, R), dtype=torch.uint8, device=DEV)
    idx = torch.empty(M, topk, dtype=torch.int32, device=DEV)
    logit = torch.empty(M, topk, dtype=torch.float32, device=DEV)
    dh.dh_forward_fp8w(x, packed, S, ZS, W8, rs, kcand, R, topk, idx, logit, ws)
    torch.cuda.synchronize()
    assert dh.dh_device_status(reset=True) == 0
    xb, W8h, rsh = host(x), W8.cpu().numpy(), rs.cpu().numpy()
    ref = orc.forward_fp8(xb, host(packed), host(S), host(ZS), W8h, rsh, kcand, R, topk)
    ties = check_result({"idx": idx.cpu().numpy(), "logit": logit.cpu().numpy()}, ref, kcand,
                        topk, xb, None, rerank_fn=lambda xr, ix: orc.rerank_fp8(xr, W8h, rsh, ix))
    print((M, H, V, kcand, R, topk), "fp8", "tie rows", len(ties))


def _forced_cases():
    out = []
    for path, Ms in ((dh.PATH_CORE, [1, 2, 3, 4]), (dh.PATH_TC_BF16, [1, 5, 16, 17, 40]),
                     (dh.PATH_WARP, [1, 7, 16, 33, 64])):
        rng = np.random.default_rng(100 + path)
        for _ in range(4):
            M = int(rng.choice(Ms))
            H = 512 * int(rng.integers(1, 13))
            V = int(rng.integers(64, 20000))
            kcand = int(rng.integers(1, 65))
            top = min(_valid_candidates(V, kcand), 1024, V)
            R = int(rng.integers(1, min(top, 64) + 1))
            topk = int(rng.integers(1, min(R, 16) + 1))
            out.append((path, M, H, V, kcand, R, topk))
    return out


@pytest.mark.parametrize("path, M, H, V, kcand, R, topk", _forced_cases())
def test_random_configuration_forced_path(path, M, H, V, kcand, R, topk):
    """The other coarse implementations, each forced, on sizes it takes (skipped otherwise)."""
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, M + V, DEV), synth.make_w(wl, H + V, DEV)
    packed, S, ZS = gpu_quantize(W)
    try:
        rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, topk, path=path)
    except dh.DHError as e:
        pytest.skip(f"path {path} does not take M={M}, H={H}: {e}")
    print((path, M, H, V, kcand, R, topk), rep["coarse_worst"], "tie rows", len(rep["ties"]))


@pytest.mark.parametrize("M, H, V, kcand, R, topk", _cases(6, seed=17))
def test_random_configuration_entry_points_agree(M, H, V, kcand, R, topk):
    """dh_forward, dh_forward_host and dh_forward_noalloc run the same kernels: bit for bit."""
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, M + V, DEV), synth.make_w(wl, H + V, DEV)
    packed, S, ZS = gpu_quantize(W)
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, kcand, R), dtype=torch.uint8, device=DEV)
    idx = torch.empty(M, topk, dtype=torch.int32, device=DEV)
    logit = torch.empty(M, topk, dtype=torch.float32, device=DEV)
    dh.dh_forward(x, packed, S, ZS, W, kcand, R, topk, idx, logit, ws)
    ih = torch.empty(M, topk, dtype=torch.int32).pin_memory()
    lh = torch.empty(M, topk, dtype=torch.float32).pin_memory()
    dh.dh_forward_host(x.cpu().pin_memory(), packed, S, ZS, W, kcand, R, topk, ih, lh, ws)
    torch.cuda.synchronize()
    assert torch.equal(ih, idx.cpu())
    assert torch.equal(lh.view(torch.int32), logit.cpu().view(torch.int32))
    if ws.numel() <= dh.NOALLOC_WORKSPACE_BYTES:
        i2, l2 = torch.empty_like(idx), torch.empty_like(logit)
        dh.dh_forward_noalloc(x, packed, S, ZS, W, kcand, R, topk, i2, l2)
        torch.cuda.synchronize()
        assert torch.equal(i2, idx) and torch.equal(l2.view(torch.int32), logit.view(torch.int32))
    assert dh.dh_device_status(reset=True) == 0


def _shard_cases(n=5, seed=23):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        P = int(rng.integers(2, 5))
        M = int(rng.choice([1, 3, 16, 17, 40]))
        H = 512 * int(rng.integers(1, 11))
        kcand = int(rng.integers(1, 17))
        R = int(rng.integers(1, 65))
        topk = int(rng.integers(1, min(R, 16) + 1))
        # every shard holds at least R valid candidates
        V = int(rng.integers(P * 64 * (R // kcand + 2), 30000))
        if M * H * V > 2e9:
            continue
        out.append((P, M, H, V, kcand, R, topk))
    return out


@pytest.mark.parametrize("P, M, H, V, kcand, R, topk", _shard_cases())
def test_random_configuration_sharded_head(P, M, H, V, kcand, R, topk):
    """P sequential vocabulary shards through the C ABI equal the unsharded forward bit for
    bit."""
    from quantised_speculative_draft_gb300.sharded import (DeviceShard,
                                                           sharded_forward_sequential, split_rows)
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, M + V, DEV), synth.make_w(wl, H + V, DEV)
    packed, S, ZS = gpu_quantize(W)
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, kcand, R), dtype=torch.uint8, device=DEV)
    idx = torch.empty(M, topk, dtype=torch.int32, device=DEV)
    logit = torch.empty(M, topk, dtype=torch.float32, device=DEV)
    dh.dh_forward(x, packed, S, ZS, W, kcand, R, topk, idx, logit, ws)
    shards = [DeviceShard(packed[a:b], S[a:b], ZS[a:b], W[a:b], a, kcand, R)
              for a, b in split_rows(V, P)]
    sidx, slogit = sharded_forward_sequential(x, shards, topk)
    torch.cuda.synchronize()
    assert dh.dh_device_status(reset=True) == 0
    assert torch.equal(sidx, idx)
    assert torch.equal(slogit.view(torch.int32), logit.view(torch.int32))


@pytest.mark.parametrize("layout", ["c4", "g64"])
@pytest.mark.parametrize("case", range(3))
def test_random_configuration_packing_ablations(layout, case):
    """The contiguous-4 and group-64 heads on random sizes they take (skipped otherwise)."""
    rng = np.random.default_rng(31 + case + (10 if layout == "g64" else 0))
    M = int(rng.choice([1, 5, 16] if layout == "g64" else [1, 5, 16, 17, 33]))
    H = 512 * int(rng.integers(1, 11))
    V = int(rng.integers(64, 20000))
    kcand = int(rng.integers(1, 65))
    R = int(rng.integers(1, min(_valid_candidates(V, kcand), 64, V) + 1))
    topk = int(rng.integers(1, min(R, 16) + 1))
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, M + V, DEV), synth.make_w(wl, H + V, DEV)
    G = 64 if layout == "g64" else 128
    packed = torch.empty(V, H // 4, dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // G, dtype=torch.bfloat16, device=DEV)
    ZS = torch.empty_like(S)
    (dh.dh_quantize_g64 if layout == "g64" else dh.dh_quantize_c4)(W, packed, S, ZS)
    try:
        rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, topk, bits=layout)
    except dh.DHError as e:
        pytest.skip(f"{layout} does not take M={M}, H={H}: {e}")
    print((layout, M, H, V, kcand, R, topk), rep["coarse_worst"], "tie rows", len(rep["ties"]))


@pytest.mark.parametrize("M, H, V, kcand, R, topk", [
    (2, 1024, 70000, 16, 1024, 1024),   # the largest RERANK, every reranked entry returned
    (5, 2048, 20011, 64, 700, 333),     # a large top-k from a ragged head
    (17, 512, 9000, 8, 100, 65),        # top-k just above two warps' worth
])
def test_large_topk(M, H, V, kcand, R, topk):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, M + V, DEV), synth.make_w(wl, H + V, DEV)
    packed, S, ZS = gpu_quantize(W)
    rep, gpu, ref = full_compare(x, W, packed, S, ZS, kcand, R, topk)
    print((M, H, V, kcand, R, topk), rep["coarse_worst"], "tie rows", len(rep["ties"]))


def _quant_shapes(n=6, seed=41):
    rng = np.random.default_rng(seed)
    return [(int(rng.choice([1, 2, 3, 7, int(rng.integers(8, 5000))])),
             512 * int(rng.integers(1, 21))) for _ in range(n)]


@pytest.mark.parametrize("kind", ["quarter", "half4", "c4", "g64", "fp8"])
@pytest.mark.parametrize("V, H", _quant_shapes())
def test_random_quantiser_shapes(kind, V, H):
    """Every quantiser bit-exact with the oracle on random head shapes: tiny heads, odd span
    counts per row (the two-span work items end on one span), widths up to 10240."""
    from parity import host as hbits
    wl = synth.custom(1, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    G = 64 if kind == "g64" else 128
    packed = torch.empty(V, H // (2 if kind == "half4" else 4), dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // G, dtype=torch.bfloat16, device=DEV)
    ZS = torch.empty_like(S)
    if kind == "fp8":
        W8, rs = synth.make_w_fp8(wl, V + H, DEV)
        dh.dh_quantize_fp8(W8, rs, packed, S, ZS)
        ref = orc.quantize_fp8(W8.cpu().numpy(), rs.cpu().numpy())
    else:
        W = synth.make_w(wl, V + H, DEV)
        fn, rf = {"quarter": (dh.dh_quantize, orc.quantize),
                  "half4": (dh.dh_quantize4, orc.quantize4),
                  "c4": (dh.dh_quantize_c4, orc.quantize_c4),
                  "g64": (dh.dh_quantize_g64, orc.quantize_g64)}[kind]
        fn(W, packed, S, ZS)
        ref = rf(hbits(W))
    torch.cuda.synchronize()
    rp, rS, rZS = ref
    assert np.array_equal(hbits(packed), rp)
    assert np.array_equal(hbits(S), rS)
    assert np.array_equal(hbits(ZS), rZS)
