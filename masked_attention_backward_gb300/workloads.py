"""Seeded synthetic workloads for masked attention backward.

This module only draws random inputs and block masks; it holds none of the
attention arithmetic.  Both the oracle side (tests, CPU baseline) and the CUDA
side (tests, bench) take their inputs from here, so they see the same values.

Recipe (one ``torch.Generator('cpu')`` per workload, seeded with the workload's
seed): draw q, k, v, dO as float32 N(0,1) in that order and round them to the
workload's dtype (round to nearest even); then the per-head sink logits as
float32 N(0,1) when the workload has a sink; then the random numbers of the
block mask; then, for a variable-length workload, the valid query rows of
each batch element, uniform integers in [ceil(varlen_min * Sq), Sq], and the
valid keys the same way (the query lengths again under a causal or sliding
mask, where each element is one self-attention sequence).

The five named workloads mirror the mask families and sizes of the pages'
suites: GQA with a sink and a causal sliding window (tilelang-ascend PR #1
"Add GQA Sink Backward BHSD", Summary), and block-sparse MHA with a uint8
block mask whose block sizes may differ per axis and need not divide S
(cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook, task features:
causal / window / bigbird / random / dense patterns, non-divisible S).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

MASK_NONE, MASK_CAUSAL, MASK_SLIDING, MASK_BLOCK = 0, 1, 2, 3


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f16" or "bf16"
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int = 128
    mask_kind: int = MASK_NONE
    window: int = 0
    bx: int = 1
    by: int = 1
    block_pattern: str = ""   # "random", "bigbird", "ones", "diag" for MASK_BLOCK
    density: float = 0.0      # Bernoulli rate of the "random" pattern
    sink: bool = False
    seed: int = 0
    varlen: bool = False      # per-batch valid lengths (the padded variable-length batch)
    varlen_min: float = 0.0   # shortest length as a fraction of S

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "f16" else torch.bfloat16

    @property
    def nqb(self) -> int:
        return -(-self.Sq // self.bx)

    @property
    def nkb(self) -> int:
        return -(-self.Skv // self.by)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = [
    Workload("gqa_sink_swa64_tiny", "f16", B=1, Hq=2, Hkv=1, Sq=256, Skv=256,
             mask_kind=MASK_SLIDING, window=64, sink=True, seed=0),
    Workload("gqa_sink_swa128_s4096", "bf16", B=2, Hq=32, Hkv=8, Sq=4096, Skv=4096,
             mask_kind=MASK_SLIDING, window=128, sink=True, seed=1),
    Workload("blocksparse_random30_s8192", "f16", B=1, Hq=16, Hkv=16, Sq=8192, Skv=8192,
             mask_kind=MASK_BLOCK, bx=64, by=64, block_pattern="random", density=0.3,
             seed=2),
    Workload("blocksparse_bigbird_5000x7000", "f16", B=2, Hq=8, Hkv=8, Sq=5000, Skv=7000,
             mask_kind=MASK_BLOCK, bx=48, by=80, block_pattern="bigbird", seed=3),
    Workload("gqa_sink_causal_s16384", "bf16", B=1, Hq=64, Hkv=8, Sq=16384, Skv=16384,
             mask_kind=MASK_CAUSAL, sink=True, seed=4),
]
# Variable-length GQA-sink backward: 8 sequences of 256..2048 tokens, 64 query
# heads in groups of 16 (tilelang-ascend examples table, "GQA Sink Backward
# VarLen": batch 8, heads 64, groups 16, sequence 2048, dim 128, fp16).
VARLEN_WORKLOADS = [
    Workload("gqa_sink_varlen_causal_b8_s2048", "f16", B=8, Hq=64, Hkv=4, Sq=2048, Skv=2048,
             mask_kind=MASK_CAUSAL, sink=True, seed=6, varlen=True, varlen_min=0.125),
]
# A smaller member of the causal GQA-sink family (inputs still larger than L2),
# used for detailed hardware-counter captures.
PROFILE_WORKLOADS = [
    Workload("gqa_sink_causal_s16384_h16", "bf16", B=1, Hq=16, Hkv=2, Sq=16384, Skv=16384,
             mask_kind=MASK_CAUSAL, sink=True, seed=5),
]
BY_NAME = {w.name: w for w in WORKLOADS + PROFILE_WORKLOADS + VARLEN_WORKLOADS}


@dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dO: torch.Tensor
    sink: Optional[torch.Tensor]          # float32 [Hq] or None
    block_mask: Optional[torch.Tensor]    # uint8 [B,Hq,nQB,nKB] or None
    extra: dict = field(default_factory=dict)
    seqlen_q: Optional[torch.Tensor] = None   # int32 [B]: valid query rows, or None
    seqlen_k: Optional[torch.Tensor] = None   # int32 [B]: valid keys, or None


def _normal(gen, shape, dtype):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def _block_mask(wl: Workload, gen) -> torch.Tensor:
    B, H, nqb, nkb = wl.B, wl.Hq, wl.nqb, wl.nkb
    if wl.block_pattern == "ones":
        return torch.ones((B, H, nqb, nkb), dtype=torch.uint8)
    if wl.block_pattern == "diag":
        m = torch.zeros((B, H, nqb, nkb), dtype=torch.uint8)
        for i in range(min(nqb, nkb)):
            m[:, :, i, i] = 1
        return m
    if wl.block_pattern == "random":
        # off-diagonal Bernoulli(density), diagonal always on
        u = torch.rand((B, H, nqb, nkb), generator=gen)
        m = (u < wl.density).to(torch.uint8)
        idx = torch.arange(min(nqb, nkb))
        m[:, :, idx, idx] = 1
        return m
    if wl.block_pattern == "bigbird":
        # per query block i: global first key block, a 3-block band around the
        # key block that holds row i*bx, and 2 distinct random blocks not yet on
        m = torch.zeros((B, H, nqb, nkb), dtype=torch.uint8)
        for b in range(B):
            for h in range(H):
                for i in range(nqb):
                    row = m[b, h, i]
                    row[0] = 1
                    c = min((i * wl.bx) // wl.by, nkb - 1)
                    for cc in (c - 1, c, c + 1):
                        if 0 <= cc < nkb:
                            row[cc] = 1
                    off = torch.nonzero(row == 0).flatten()
                    if off.numel() > 0:
                        pick = torch.randperm(off.numel(), generator=gen)[:2]
                        row[off[pick]] = 1
        return m
    if wl.block_pattern == "bernoulli":
        u = torch.rand((B, H, nqb, nkb), generator=gen)
        return (u < wl.density).to(torch.uint8)
    raise ValueError(f"unknown block pattern {wl.block_pattern!r}")


def make_inputs(wl: Workload, seed: Optional[int] = None) -> Inputs:
    """Seeded CPU tensors of the workload's shapes, in its dtype."""
    gen = torch.Generator("cpu")
    gen.manual_seed(wl.seed if seed is None else seed)
    dt = wl.torch_dtype
    q = _normal(gen, (wl.B, wl.Hq, wl.Sq, wl.D), dt)
    k = _normal(gen, (wl.B, wl.Hkv, wl.Skv, wl.D), dt)
    v = _normal(gen, (wl.B, wl.Hkv, wl.Skv, wl.D), dt)
    dO = _normal(gen, (wl.B, wl.Hq, wl.Sq, wl.D), dt)
    sink = torch.randn((wl.Hq,), generator=gen, dtype=torch.float32) if wl.sink else None
    bm = _block_mask(wl, gen) if wl.mask_kind == MASK_BLOCK else None
    lq = lk = None
    if wl.varlen:
        lq = torch.randint(math.ceil(wl.varlen_min * wl.Sq), wl.Sq + 1, (wl.B,), generator=gen,
                           dtype=torch.int32)
        if wl.mask_kind in (MASK_CAUSAL, MASK_SLIDING):
            lk = lq.clone()
        else:
            lk = torch.randint(math.ceil(wl.varlen_min * wl.Skv), wl.Skv + 1, (wl.B,),
                               generator=gen, dtype=torch.int32)
    return Inputs(wl, q, k, v, dO, sink, bm, seqlen_q=lq, seqlen_k=lk)
