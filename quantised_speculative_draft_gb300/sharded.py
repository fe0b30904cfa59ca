"""Vocabulary-parallel draft head: each rank holds a contiguous shard of the head's rows.

radiance_drafthead.py runs the draft head on a vocab-parallel lm_head (every tensor-parallel
rank owns a slice of the vocabulary).  The exact sharded result needs two small exchanges:

1. every rank computes its shard's top-RERANK candidates (coarse value, global vocabulary id);
2. the lists are all-gathered; every rank takes the same global top-RERANK (the union of the
   shards' top-RERANK lists contains it, so it equals the unsharded selection) and computes the
   exact logits of the selected ids it owns (-inf for the others);
3. the partial exact logits are all-gathered and merged into the top-k.

Each step runs on the device through the C ABI (``DeviceShard``).  The exchange is a callable
``all_gather(t) -> stacked [P, *t.shape]``: ``torch_all_gather`` wraps torch.distributed (one
process per GPU), and ``sharded_forward_sequential`` runs several shards in one process, which
is how the result is checked bit for bit against the unsharded head on one GPU.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def split_rows(V: int, parts: int, align: int = 64):
    """Row ranges [(start, stop), ...] covering [0, V) in `parts` shards whose starts are
    multiples of `align` (the selection blocks then coincide with the unsharded head's)."""
    nblk = (V + align - 1) // align
    if parts < 1 or parts > nblk:
        raise ValueError(f"cannot split {V} rows into {parts} shards of whole {align}-row blocks")
    bounds = [min(V, (nblk * i // parts) * align) for i in range(parts + 1)]
    return [(bounds[i], bounds[i + 1]) for i in range(parts)]


def sharded_forward(x, shard, all_gather, topk: int):
    """One rank's part of the sharded forward.  `shard` provides candidates(x),
    rerank(x, all_val, all_idx) and topk(parts, sel_idx, topk); returns (idx, logit) [M, topk],
    identical on every rank."""
    val, idx = shard.candidates(x)                      # [M, R] each
    M, R = val.shape
    all_val = all_gather(val).permute(1, 0, 2).reshape(M, -1).contiguous()
    all_idx = all_gather(idx).permute(1, 0, 2).reshape(M, -1).contiguous()
    sel_idx, exact = shard.rerank(x, all_val, all_idx)  # [M, R] each
    parts = all_gather(exact).contiguous()               # [P, M, R]
    return shard.topk(parts, sel_idx, topk)


def sharded_forward_sequential(x, shards, topk: int):
    """All shards in one process (one device), the exchanges done by stacking."""
    cands = [s.candidates(x) for s in shards]
    M = x.shape[0]
    all_val = torch.stack([c[0] for c in cands]).permute(1, 0, 2).reshape(M, -1).contiguous()
    all_idx = torch.stack([c[1] for c in cands]).permute(1, 0, 2).reshape(M, -1).contiguous()
    reranked = [s.rerank(x, all_val, all_idx) for s in shards]
    parts = torch.stack([r[1] for r in reranked]).contiguous()
    return shards[0].topk(parts, reranked[0][0], topk)


def torch_all_gather(group=None):
    """all_gather over a torch.distributed process group, stacked along a new leading axis."""
    import torch.distributed as dist

    def gather(t):
        out = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
        dist.all_gather(out, t.contiguous(), group=group)
        return torch.stack(out)

    return gather


@dataclass
class DeviceShard:
    """Rows [vocab_offset, vocab_offset + Vs) of a quantised head on this device.

    packed/scales/zeros are the shard's dh_quantize outputs, W its bf16 rows (kept by
    reference for the rerank)."""
    packed: torch.Tensor
    scales: torch.Tensor
    zeros: torch.Tensor
    W: torch.Tensor
    vocab_offset: int
    kcand: int = 8
    nrerank: int = 32

    def candidates(self, x):
        from . import dh_shard_candidates, dh_workspace_bytes
        M, H = x.shape
        Vs = self.packed.shape[0]
        ws = torch.empty(dh_workspace_bytes(M, H, Vs, self.kcand, self.nrerank),
                         dtype=torch.uint8, device=x.device)
        val = torch.empty(M, self.nrerank, dtype=torch.float32, device=x.device)
        idx = torch.empty(M, self.nrerank, dtype=torch.int32, device=x.device)
        dh_shard_candidates(x, self.packed, self.scales, self.zeros, self.vocab_offset,
                            self.kcand, self.nrerank, val, idx, ws)
        return val, idx

    def rerank(self, x, all_val, all_idx):
        from . import dh_shard_rerank, dh_shard_rerank_workspace_bytes
        M = x.shape[0]
        n = dh_shard_rerank_workspace_bytes(M, all_val.shape[1], self.nrerank)
        ws = torch.empty(n, dtype=torch.uint8, device=x.device)
        sel = torch.empty(M, self.nrerank, dtype=torch.int32, device=x.device)
        exact = torch.empty(M, self.nrerank, dtype=torch.float32, device=x.device)
        dh_shard_rerank(x, self.W, self.vocab_offset, all_val, all_idx, self.nrerank, sel, exact,
                        ws)
        return sel, exact

    def topk(self, parts, sel_idx, topk):
        from . import dh_shard_topk
        M = sel_idx.shape[0]
        idx = torch.empty(M, topk, dtype=torch.int32, device=sel_idx.device)
        logit = torch.empty(M, topk, dtype=torch.float32, device=sel_idx.device)
        dh_shard_topk(parts, sel_idx, topk, idx, logit)
        return idx, logit
