"""Vocabulary-parallel head on one GPU: the head split into shards run one after another
through the sharded entry points (dh_shard_candidates / dh_shard_rerank / dh_shard_topk), the
exchanges done by stacking, must return exactly what the unsharded dh_forward returns, and
that result is judged against the oracle by the rules in parity.py."""
import pytest
import torch

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth
from oracle import oracle as orc
from quantised_speculative_draft_gb300.sharded import (DeviceShard, sharded_forward_sequential,
                                                       split_rows)

from parity import check_result, host

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _build():
    dh.build()
    torch.cuda.init()


def _quantize(W):
    V, H = W.shape
    packed = torch.empty(V, H // 4, dtype=torch.uint8, device=DEV)
    S = torch.empty(V, H // 128, dtype=torch.bfloat16, device=DEV)
    ZS = torch.empty_like(S)
    dh.dh_quantize(W, packed, S, ZS)
    return packed, S, ZS


@pytest.mark.parametrize("P, M, H, V, kcand, R, k", [
    (2, 5, 1024, 8192 + 37, 8, 32, 4),    # ragged tail block in the last shard
    (3, 16, 1024, 16384, 8, 32, 1),       # argmax caller
    (4, 16, 512, 12288, 8, 64, 16),       # RERANK 64: the multi-pass selection with offsets
    (2, 33, 1536, 6144, 4, 24, 5),        # several batch chunks
])
def test_sequential_shards_equal_the_unsharded_forward(P, M, H, V, kcand, R, k):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = _quantize(W)
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, kcand, R), dtype=torch.uint8, device=DEV)
    idx = torch.empty(M, k, dtype=torch.int32, device=DEV)
    logit = torch.empty(M, k, dtype=torch.float32, device=DEV)
    dh.dh_forward(x, packed, S, ZS, W, kcand, R, k, idx, logit, ws)
    shards = [DeviceShard(packed[a:b], S[a:b], ZS[a:b], W[a:b], a, kcand, R)
              for a, b in split_rows(V, P)]
    sidx, slogit = sharded_forward_sequential(x, shards, k)
    torch.cuda.synchronize()
    assert dh.dh_device_status(reset=True) == 0
    assert torch.equal(sidx, idx)
    assert torch.equal(slogit, logit)
    xb, Wb = host(x), host(W)
    ref = orc.forward(xb, host(packed), host(S), host(ZS), Wb, kcand, R, k)
    ties = check_result({"idx": sidx.cpu().numpy(), "logit": slogit.cpu().numpy()}, ref,
                        kcand, k, xb, Wb)
    print("sharded", P, M, V, "tie rows", len(ties), "differing", sum(t[4] for t in ties))


def test_shard_candidates_are_the_shard_slice_of_the_coarse_pass():
    """A shard's candidates carry global ids and the coarse values of the unsharded pass."""
    M, H, V, kcand, R = 4, 1024, 4096, 8, 32
    wl = synth.custom(M, H, V)
    x, W = synth.make_x(wl, 0, DEV), synth.make_w(wl, 0, DEV)
    packed, S, ZS = _quantize(W)
    nblk = (V + 63) // 64
    ws = torch.empty(dh.dh_workspace_bytes(M, H, V, kcand, R), dtype=torch.uint8, device=DEV)
    coarse = torch.empty(M, V, dtype=torch.float32, device=DEV)
    cval = torch.empty(M, nblk * kcand, dtype=torch.float32, device=DEV)
    cidx = torch.empty(M, nblk * kcand, dtype=torch.int32, device=DEV)
    idx = torch.empty(M, 1, dtype=torch.int32, device=DEV)
    logit = torch.empty(M, 1, dtype=torch.float32, device=DEV)
    dh.dh_forward_debug(x, packed, S, ZS, W, kcand, R, 1, idx, logit, ws, coarse=coarse,
                        cand_val=cval, cand_idx=cidx)
    a, b = 1024, 3072
    shard = DeviceShard(packed[a:b], S[a:b], ZS[a:b], W[a:b], a, kcand, R)
    val, gid = shard.candidates(x)
    torch.cuda.synchronize()
    assert ((gid >= a) & (gid < b)).all()
    assert torch.equal(val, torch.gather(coarse, 1, gid.long()))
    # rank order: values descending, equal values by lower id
    v, g = val.cpu(), gid.cpu()
    for m in range(M):
        for j in range(R - 1):
            assert v[m, j] > v[m, j + 1] or (v[m, j] == v[m, j + 1] and g[m, j] < g[m, j + 1])
