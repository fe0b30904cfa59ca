"""Seeded synthetic workloads for the draft head (inputs only: no step of the method here).

The pages measure on hidden states captured from a live serve and on a trained head; neither
exists here, so these generators stand in for them with the shapes and value distributions
the workloads name:

* ``tiny``      M=1,  H=1024, V=8192:   x ~ N(0,1); W ~ N(0, 0.02)
* ``shard``     M=16 (or 64), H=5120, V=124160: x ~ N(0,1) with every row scaled to RMS 1;
                W ~ N(0, 0.02) with 512 seeded rows at 4x (hot rows that create near-ties)
* ``full``      H=5120, V=248320, any M: x ~ N(0,1); W ~ N(0, 0.02) with 1 % of the rows
                (2483) drawn at 3x the standard deviation
* ``topk``      M=16, H=5120, V=248320: x ~ N(0,1); W ~ N(0, 0.02) with 2048 rows at 4x

``make_w_fp8`` gives any of these heads as an fp8 checkpoint (e4m3 rows, per-row fp32 scale).

All draws come from one ``torch.Generator`` seeded with ``seed`` (0 by default) on the
requested device; values are drawn in fp32 and rounded once to bf16.  The same tensors feed
the CUDA path and (copied to the host) the CPU oracle.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    H: int
    V: int
    x_rms_norm: bool = False
    hot_rows: int = 0          # rows of W scaled by hot_scale
    hot_scale: float = 1.0
    w_std: float = 0.02
    kcand: int = 8
    rerank: int = 32
    topk: int = 1


def tiny(M: int = 1) -> Workload:
    return Workload("tiny head", M=M, H=1024, V=8192)


def shard(M: int = 16) -> Workload:
    return Workload("one-shard head", M=M, H=5120, V=124160, x_rms_norm=True, hot_rows=512,
                    hot_scale=4.0)


def full(M: int = 16) -> Workload:
    return Workload("full-vocab head", M=M, H=5120, V=248320, hot_rows=2483, hot_scale=3.0)


def topk_caller(rerank: int = 32) -> Workload:
    return Workload("top-k caller", M=16, H=5120, V=248320, hot_rows=2048, hot_scale=4.0,
                    rerank=rerank, topk=16)


def custom(M: int, H: int, V: int, **kw) -> Workload:
    return Workload("custom", M=M, H=H, V=V, **kw)


def make_x(wl: Workload, seed: int = 0, device: str = "cpu") -> torch.Tensor:
    """Hidden states x [M, H] bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 17)
    x = torch.randn(wl.M, wl.H, generator=g, device=device, dtype=torch.float32)
    if wl.x_rms_norm:
        x = x / x.pow(2).mean(dim=1, keepdim=True).sqrt()
    return x.to(torch.bfloat16).contiguous()


def make_w(wl: Workload, seed: int = 0, device: str = "cpu", chunk_rows: int = 16384
           ) -> torch.Tensor:
    """Head weight W [V, H] bf16 (row n = vocabulary entry n)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 29)
    W = torch.empty(wl.V, wl.H, dtype=torch.bfloat16, device=device)
    scale = torch.full((wl.V,), wl.w_std, dtype=torch.float32, device=device)
    if wl.hot_rows:
        hot = torch.randperm(wl.V, generator=g, device=device)[: wl.hot_rows]
        scale[hot] *= wl.hot_scale
    for r0 in range(0, wl.V, chunk_rows):
        r1 = min(wl.V, r0 + chunk_rows)
        blk = torch.randn(r1 - r0, wl.H, generator=g, device=device, dtype=torch.float32)
        W[r0:r1] = (blk * scale[r0:r1, None]).to(torch.bfloat16)
    return W


def make_w_fp8(wl: Workload, seed: int = 0, device: str = "cpu", chunk_rows: int = 16384):
    """An fp8 head standing in for a checkpoint stored as e4m3 rows with one fp32 scale per
    row: the fp32 draws of make_w (before their bf16 rounding), each row scaled so that its
    largest magnitude maps to 448 (the largest finite e4m3 value) and rounded to e4m3.
    Returns (codes [V, H] uint8, row_scale [V] fp32); no code is a NaN code."""
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 29)
    codes = torch.empty(wl.V, wl.H, dtype=torch.uint8, device=device)
    row_scale = torch.empty(wl.V, dtype=torch.float32, device=device)
    scale = torch.full((wl.V,), wl.w_std, dtype=torch.float32, device=device)
    if wl.hot_rows:
        hot = torch.randperm(wl.V, generator=g, device=device)[: wl.hot_rows]
        scale[hot] *= wl.hot_scale
    for r0 in range(0, wl.V, chunk_rows):
        r1 = min(wl.V, r0 + chunk_rows)
        blk = torch.randn(r1 - r0, wl.H, generator=g, device=device, dtype=torch.float32)
        blk = blk * scale[r0:r1, None]
        rs = blk.abs().amax(dim=1).clamp_min(1e-30) / 448.0
        q = (blk / rs[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        codes[r0:r1] = q.view(torch.uint8)
        row_scale[r0:r1] = rs
    return codes, row_scale


def bits(t: torch.Tensor):
    """A bf16 tensor's raw bit patterns as a host uint16 numpy array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
