"""Shared helpers for the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare them under the acceptance gate.

Gate (per output tensor): no non-finite element, and
|gpu - ref| <= atol + rtol * |ref| on at least 99.9 % of the elements, with
atol = rtol = 2e-3 for fp16 inputs and 1.6e-2 for bf16 inputs.  The oracle
reference is float64 computed from the very values the GPU received (inputs
rounded to the working dtype, O rounded to the dtype, LSE rounded to fp32).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import oracle
from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import (MASK_BLOCK, MASK_NONE, MASK_SLIDING, Inputs,
                                                        Workload, make_inputs)

TOL = {"f16": 2e-3, "bf16": 1.6e-2}
MIN_FRAC = 0.999


def oracle_problem(wl: Workload, inp: Inputs) -> oracle.Problem:
    return oracle.Problem(
        B=wl.B, Hq=wl.Hq, Hkv=wl.Hkv, Sq=wl.Sq, Skv=wl.Skv, D=wl.D, scale=wl.scale,
        mask_kind=wl.mask_kind, window=wl.window, bx=wl.bx, by=wl.by,
        block_mask=None if inp.block_mask is None else inp.block_mask.numpy(),
        sink=None if inp.sink is None else inp.sink.double().numpy(),
        seqlen_q=None if inp.seqlen_q is None else inp.seqlen_q.numpy(),
        seqlen_k=None if inp.seqlen_k is None else inp.seqlen_k.numpy())


def gpu_mask(wl: Workload, inp: Inputs, device="cuda") -> mab.Mask:
    bm = inp.block_mask.to(device) if inp.block_mask is not None else None
    lq = inp.seqlen_q.to(device) if inp.seqlen_q is not None else None
    lk = inp.seqlen_k.to(device) if inp.seqlen_k is not None else None
    return mab.Mask(kind=wl.mask_kind, window=wl.window, bx=wl.bx, by=wl.by, block_mask=bm,
                    seqlen_q=lq, seqlen_k=lk)


def forward_stats(wl: Workload, inp: Inputs, pb=None):
    """Oracle forward; returns (O rounded to the dtype, LSE rounded to fp32)."""
    pb = pb or oracle_problem(wl, inp)
    O, lse = oracle.forward(pb, inp.q, inp.k, inp.v)
    return torch.from_numpy(O).to(wl.torch_dtype), torch.from_numpy(lse).to(torch.float32)


def compare(name: str, got, ref, dtype: str, min_frac: float = MIN_FRAC):
    """Assert the gate; returns a small report dict."""
    g = got.detach().to("cpu").double().numpy() if hasattr(got, "detach") else np.asarray(got)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    nonfinite = int(np.size(g) - np.isfinite(g).sum())
    assert nonfinite == 0, f"{name}: {nonfinite} non-finite elements"
    tol = TOL[dtype]
    err = np.abs(g - r)
    ok = err <= tol + tol * np.abs(r)
    frac = float(ok.mean()) if ok.size else 1.0
    rep = {"name": name, "frac": frac, "max_err": float(err.max()) if err.size else 0.0,
           "n": int(ok.size)}
    assert frac >= min_frac, f"{name}: only {frac:.5f} within tolerance (max err {rep['max_err']:.3g})"
    return rep


def load_gate(path=None) -> dict:
    """The fp16 precision gate printed for the GQA-sink backward example's
    test suite (tests/golden/fp16_precision_gate.txt, with its citation)."""
    import os
    path = path or os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                                "fp16_precision_gate.txt")
    gate = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if len(line) == 2:
                gate[line[0]] = float(line[1])
    return gate


# The page prints atol and rtol to three figures; they are read as 2^-14 and
# 2^-9 (6.1035e-5, 1.9531e-3), which tests/test_golden.py checks.
_GATE = load_gate()
TIGHT_ATOL, TIGHT_RTOL = 2.0 ** -14, 2.0 ** -9
TIGHT_FRAC, TIGHT_MAX = _GATE["required_ratio"], _GATE["max_abs_limit"]


def tight_gate(name: str, got, ref) -> float:
    g = got.detach().double().cpu().numpy()
    err = np.abs(g - np.asarray(ref, dtype=np.float64))
    frac = float((err <= TIGHT_ATOL + TIGHT_RTOL * np.abs(ref)).mean())
    assert frac >= TIGHT_FRAC, f"{name}: {frac:.5f} of the elements within the tight gate"
    assert float(err.max()) <= TIGHT_MAX, f"{name}: max error {err.max():.3e}"
    return frac


@dataclass
class GpuRun:
    dq: torch.Tensor
    dk: torch.Tensor
    dv: torch.Tensor
    dsink: torch.Tensor
    ws: torch.Tensor


def run_gpu_bwd(wl: Workload, inp: Inputs, O, lse, poison: bool = True,
                compensated: bool = False, single_pass: bool = False) -> GpuRun:
    dev = "cuda"
    q, k, v, dO = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.dO))
    o, l = O.to(dev), lse.to(dev)
    sink = inp.sink.to(dev) if inp.sink is not None else None
    mask = gpu_mask(wl, inp, dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dsink = torch.empty_like(sink) if sink is not None else None
    if poison:  # every output element must be written
        for t in (dq, dk, dv):
            t.fill_(float("nan"))
        if dsink is not None:
            dsink.fill_(float("nan"))
    flags = mab.ATTN_FLAG_SINGLE_PASS if single_pass else 0
    ws = mab.workspace(mab.shape_of(q, k, flags), mask, dev)
    mab.bwd(q, k, v, o, dO, l, sink, mask, wl.scale, ws=ws, out=(dq, dk, dv, dsink),
            compensated=compensated, single_pass=single_pass)
    torch.cuda.synchronize()
    st = mab.device_status(ws)
    assert st == mab.ATTN_OK, mab.attn_status_string(st)
    return GpuRun(dq, dk, dv, dsink, ws)


def full_parity(wl: Workload, seed=None, single_pass: bool = False):
    """Element-by-element parity of dq, dk, dv (and dsink) against the oracle."""
    inp = make_inputs(wl, seed)
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    run = run_gpu_bwd(wl, inp, O, lse, single_pass=single_pass)
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    reps = [compare("dq", run.dq, ref["dq"], wl.dtype),
            compare("dk", run.dk, ref["dk"], wl.dtype),
            compare("dv", run.dv, ref["dv"], wl.dtype)]
    if inp.sink is not None:
        reps.append(compare("dsink", run.dsink, ref["dsink"], wl.dtype, min_frac=1.0))
    return reps, run, ref


# Tile sizes of the CUDA kernels (key tile / query sub-tile of the dK-dV walk,
# query tile / key sub-tile of the dQ walk) and the workspace layout that the
# library carves; mirrored here so that tests can read the device tables.
KV_TILE, KV_SUB, Q_TILE, Q_SUB, PREP_ROWS = 128, 64, 128, 64, 128
PREP_BLOCK_ROWS = 64  # rows per preprocess block: one dSink partial each


def _a256(x):
    return (x + 255) // 256 * 256


def tile_pair_visible(wl: Workload, i0: int, i1: int, j0: int, j1: int) -> bool:
    """Whether query rows [i0, i1) and keys [j0, j1) hold a visible pair under
    a closed-form mask: causal j <= i, sliding window 0 <= i - j < W, or none.
    The differences i - j the two ranges can form are [i0 - (j1 - 1),
    (i1 - 1) - j0]; a pair is visible when that interval meets the mask's."""
    if wl.mask_kind == MASK_NONE:
        return True
    lo, hi = i0 - (j1 - 1), (i1 - 1) - j0
    w = wl.window if wl.mask_kind == MASK_SLIDING else 1 << 40
    return hi >= 0 and lo <= w - 1


def single_pass_steps_head(wl: Workload) -> int:
    """dq partial slots per query head of the single-pass backward: the
    (key tile, query sub-tile) pairs holding a visible pair at the full
    lengths, every pair for block masks."""
    cdiv = lambda a, b: -(-a // b)
    nkt, nqt = cdiv(wl.Skv, KV_TILE), cdiv(wl.Sq, KV_SUB)
    if wl.mask_kind == MASK_BLOCK:
        return nkt * nqt
    return sum(tile_pair_visible(wl, r * KV_SUB, min((r + 1) * KV_SUB, wl.Sq), t * KV_TILE,
                                 min((t + 1) * KV_TILE, wl.Skv))
               for t in range(nkt) for r in range(nqt))


def ws_layout(wl: Workload, single_pass: bool = False) -> dict:
    cdiv = lambda a, b: -(-a // b)
    Sq_pad = cdiv(wl.Sq, PREP_ROWS) * PREP_ROWS
    BH = wl.B * wl.Hq
    L = {"status": 0}
    off = _a256(24)  # the status word
    L["nlse2"] = off; off = _a256(off + BH * Sq_pad * 4)
    L["delta"] = off; off = _a256(off + BH * Sq_pad * 4)
    L["dsink_part"] = off; off = _a256(off + wl.Hq * wl.B * (Sq_pad // PREP_BLOCK_ROWS) * 4)
    d = {"Sq_pad": Sq_pad, "nQT_k": cdiv(wl.Sq, KV_SUB), "nKT_k": cdiv(wl.Skv, KV_TILE),
         "nQT_q": cdiv(wl.Sq, Q_TILE), "nKT_q": cdiv(wl.Skv, Q_SUB)}
    if wl.mask_kind == MASK_BLOCK:
        L["maskT"] = off; off = _a256(off + BH * wl.nqb * wl.nkb)
        L["sel_k"] = off; off = _a256(off + BH * d["nKT_k"] * d["nQT_k"] * 4)
        L["cnt_k"] = off; off = _a256(off + BH * d["nKT_k"] * 4)
        L["sel_q"] = off; off = _a256(off + BH * d["nQT_q"] * d["nKT_q"] * 4)
        L["cnt_q"] = off; off = _a256(off + BH * d["nQT_q"] * 4)
    if single_pass:
        slots = BH * single_pass_steps_head(wl)
        L["dq_flag"] = off; off = _a256(off + slots)
        L["dq_part"] = off; off = _a256(off + slots * KV_SUB * 128 * 4)
    L["total"] = off
    L.update(d)
    return L


def ws_view(ws: torch.Tensor, off: int, count: int, dtype) -> torch.Tensor:
    nbytes = count * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)
