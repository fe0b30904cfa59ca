"""Vocabulary-parallel head on the CPU (no GPU): the row split, the host-side argument checks
of the sharded entry points, and the exchange protocol itself run as gloo ranks with every
step computed by the oracle on that rank's shard -- the sharded result must equal the
oracle's unsharded forward exactly.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import quantised_speculative_draft_gb300 as dh
from quantised_speculative_draft_gb300 import synth
from quantised_speculative_draft_gb300.sharded import (sharded_forward, split_rows,
                                                       torch_all_gather)
from oracle import oracle as orc

FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def test_split_rows_covers_the_head_in_whole_blocks():
    for V, P in [(1000, 2), (1000, 3), (8192 + 37, 3), (64, 1), (640, 10)]:
        parts = split_rows(V, P)
        assert len(parts) == P and parts[0][0] == 0 and parts[-1][1] == V
        for (a, b), (c, _) in zip(parts, parts[1:]):
            assert b == c
        assert all(a % 64 == 0 and b > a for a, b in parts)
    with pytest.raises(ValueError):
        split_rows(100, 3)  # two blocks cannot make three shards


@pytest.fixture(scope="module")
def lib():
    dh.build()
    return dh._load()


def test_shard_entry_points_reject_bad_arguments(lib):
    # vocab_offset not a multiple of 64, then a null output
    assert lib.dh_shard_candidates(FAKE, FAKE, FAKE, FAKE, 4, 1024, 4096, 32, 8, 32, FAKE, FAKE,
                                   FAKE, 1 << 40, None) == -2
    assert lib.dh_shard_candidates(FAKE, FAKE, FAKE, FAKE, 4, 1024, 4096, 64, 8, 32, None, FAKE,
                                   FAKE, 1 << 40, None) == -1
    # rerank above the shard's valid candidates
    assert lib.dh_shard_candidates(FAKE, FAKE, FAKE, FAKE, 4, 1024, 64, 0, 8, 32, FAKE, FAKE,
                                   FAKE, 1 << 40, None) == -3
    assert lib.dh_shard_rerank_workspace_bytes(4, 64, 32) > 0
    assert lib.dh_shard_rerank_workspace_bytes(4, 16, 32) == 0   # rerank > gathered entries
    assert lib.dh_shard_rerank_workspace_bytes(0, 64, 32) == 0
    assert lib.dh_shard_rerank(FAKE, FAKE, 4, 1024, 4096, 0, FAKE, FAKE, 64, 32, FAKE, FAKE,
                               FAKE, 16, None) == -4           # workspace too small
    assert lib.dh_shard_rerank(FAKE, None, 4, 1024, 4096, 0, FAKE, FAKE, 64, 32, FAKE, FAKE,
                               FAKE, 1 << 40, None) == -1
    assert lib.dh_shard_rerank(FAKE, FAKE, 4, 1000, 4096, 0, FAKE, FAKE, 64, 32, FAKE, FAKE,
                               FAKE, 1 << 40, None) == -2      # H not a multiple of 512
    assert lib.dh_shard_topk(FAKE, FAKE, 2, 4, 32, 33, FAKE, FAKE, None) == -3
    assert lib.dh_shard_topk(FAKE, FAKE, 0, 4, 32, 1, FAKE, FAKE, None) == -8
    assert lib.dh_shard_topk(FAKE, None, 2, 4, 32, 1, FAKE, FAKE, None) == -1


class OracleShard:
    """The three steps of one rank, computed by the oracle on the rank's rows."""

    def __init__(self, packed, S, ZS, W, offset, kcand, rerank):
        self.packed, self.S, self.ZS, self.W = packed, S, ZS, W
        self.offset, self.kcand, self.R = offset, kcand, rerank

    def candidates(self, x):
        cf = orc.coarse(x.numpy(), self.packed, self.S, self.ZS).astype(np.float32)
        cval, cidx, _ = orc.block_topk(cf, self.kcand)
        cidx = np.where(cidx >= 0, cidx + self.offset, -1).astype(np.int32)
        sel, val = orc.select_topr(cval, cidx, self.R)
        return torch.from_numpy(val), torch.from_numpy(sel)

    def rerank(self, x, all_val, all_idx):
        sel, _ = orc.select_topr(all_val.numpy(), all_idx.numpy(), self.R)
        local = sel - self.offset
        own = (local >= 0) & (local < self.W.shape[0])
        e = orc.rerank(x.numpy(), self.W, np.where(own, local, 0).astype(np.int32))
        e[~own] = -np.inf
        return torch.from_numpy(sel), torch.from_numpy(e)

    def topk(self, parts, sel, k):
        idx, val = orc.topk(parts.max(dim=0).values.numpy(), sel.numpy(), k)
        return torch.from_numpy(idx), torch.from_numpy(val)


def _inputs(M, H, V):
    wl = synth.custom(M, H, V, hot_rows=max(1, V // 50), hot_scale=4.0)
    x, W = synth.make_x(wl, 0, "cpu"), synth.make_w(wl, 0, "cpu")
    return synth.bits(x), synth.bits(W)


def _rank(rank, world, port, M, H, V, kcand, R, k):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        xb, Wb = _inputs(M, H, V)
        packed, S, ZS = orc.quantize(Wb)
        a, b = split_rows(V, world)[rank]
        shard = OracleShard(packed[a:b], S[a:b], ZS[a:b], Wb[a:b], a, kcand, R)
        idx, logit = sharded_forward(torch.from_numpy(xb), shard, torch_all_gather(), k)
        ref = orc.forward(xb, packed, S, ZS, Wb, kcand, R, k)
        assert np.array_equal(idx.numpy(), ref["idx"])
        assert np.array_equal(logit.numpy(), ref["logit"])
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world, M, H, V, kcand, R, k", [
    (2, 3, 512, 1000, 4, 8, 3),
    (3, 5, 1024, 2048 + 37, 8, 32, 4),
])
def test_sharded_protocol_matches_the_unsharded_oracle(world, M, H, V, kcand, R, k):
    orc.build()
    mp.spawn(_rank, args=(world, _free_port(), M, H, V, kcand, R, k), nprocs=world, join=True)
