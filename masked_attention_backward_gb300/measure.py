"""Work units of the backward pass, for throughput reporting.

The unit is a visible (b, h, i, j) token pair.  The count does not depend on
the kernels' tile sizes, so work spent on masked positions inside partially
visible tiles earns no credit.  Per visible pair the five contractions of the
backward (S = QK^T, dP = dO V^T, dV += P^T dO, dK += dS^T Q, dQ += dS K) cost
2*D flops each:

  end-to-end         10 * D * pairs
  dK/dV kernel        8 * D * pairs   (S, dP, dV, dK)
  dQ kernel           6 * D * pairs   (S, dP, dQ; S and dP are recomputed)
"""
from __future__ import annotations

import numpy as np

from .workloads import MASK_BLOCK, MASK_CAUSAL, MASK_NONE, MASK_SLIDING, Workload


def visible_pairs(wl: Workload, block_mask=None, seqlen_q=None, seqlen_k=None) -> int:
    if seqlen_q is not None or seqlen_k is not None:
        # one batch element at a time, cut to its valid rows and keys
        lq = [wl.Sq] * wl.B if seqlen_q is None else [int(x) for x in seqlen_q]
        lk = [wl.Skv] * wl.B if seqlen_k is None else [int(x) for x in seqlen_k]
        total = 0
        for b in range(wl.B):
            Lq, Lk = max(0, min(lq[b], wl.Sq)), max(0, min(lk[b], wl.Skv))
            if Lq == 0 or Lk == 0:
                continue
            cut = wl.with_(B=1, Sq=Lq, Skv=Lk, varlen=False)
            bm = None
            if block_mask is not None:
                bm = np.asarray(block_mask.cpu().numpy() if hasattr(block_mask, "cpu")
                                else block_mask)[b:b + 1, :, :cut.nqb, :cut.nkb]
            total += visible_pairs(cut, bm)
        return total
    heads = wl.B * wl.Hq
    S = wl.Sq
    if wl.mask_kind == MASK_NONE:
        return heads * wl.Sq * wl.Skv
    if wl.mask_kind == MASK_CAUSAL:
        assert wl.Sq == wl.Skv
        return heads * S * (S + 1) // 2
    if wl.mask_kind == MASK_SLIDING:
        W = wl.window
        if W >= S:
            return heads * S * (S + 1) // 2
        return heads * (W * (W + 1) // 2 + (S - W) * W)
    if wl.mask_kind == MASK_BLOCK:
        m = np.asarray(block_mask.cpu().numpy() if hasattr(block_mask, "cpu") else block_mask,
                       dtype=np.int64)
        rows = np.minimum(wl.bx, wl.Sq - np.arange(wl.nqb) * wl.bx)
        cols = np.minimum(wl.by, wl.Skv - np.arange(wl.nkb) * wl.by)
        return int(np.einsum("bhqk,q,k->", m, rows, cols))
    raise ValueError(wl.mask_kind)


def flops(wl: Workload, pairs: int) -> dict:
    D = wl.D
    # the forward's two contractions (S = Q K^T, O = P V) at 2 D per pair
    return {"total": 10 * D * pairs, "dkdv": 8 * D * pairs, "dq": 6 * D * pairs,
            "fwd": 4 * D * pairs}


def algorithmic_bytes(wl: Workload, block_mask_bytes: int = 0, seqlen_q=None,
                      seqlen_k=None) -> dict:
    """Bytes each tensor must cross HBM once: q, k, v, o, dO, lse read; dq, dk,
    dv written (plus sink / dsink and the block mask).  With per-batch lengths
    only the rows and keys inside them count."""
    e = 2
    rows_q = wl.B * wl.Sq if seqlen_q is None else int(sum(min(max(int(x), 0), wl.Sq)
                                                           for x in seqlen_q))
    rows_k = wl.B * wl.Skv if seqlen_k is None else int(sum(min(max(int(x), 0), wl.Skv)
                                                            for x in seqlen_k))
    q = wl.Hq * rows_q * wl.D * e
    kv = wl.Hkv * rows_k * wl.D * e
    lse = wl.Hq * rows_q * 4
    read = 3 * q + 2 * kv + lse + block_mask_bytes
    write = q + 2 * kv
    return {"read": read, "write": write, "total": read + write,
            # preprocess alone: reads o, dO, lse; writes Delta and lse*log2(e)
            "preprocess": 2 * q + lse + 2 * lse}
