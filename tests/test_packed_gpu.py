"""The packed variable-length layout (cumulative sequence offsets) against the
oracle, element by element.

The inputs are the seeded padded tensors of a variable-length workload; the
GPU receives them packed token-major (sequence b's first L_b rows, back to
back: q, o, dO [T_q, Hq, 128], k, v [T_k, Hkv, 128], lse [Hq, T_q]).  Its
outputs are unpacked again and compared with the oracle's results for the
padded problem with the same per-batch lengths, whose rows and keys past
each length are zero.  Outputs start as NaN, so every token must be written.
Packing and unpacking only move rows.
"""
import numpy as np
import pytest
import torch

import oracle
from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import (BY_NAME, MASK_BLOCK, MASK_CAUSAL,
                                                        MASK_NONE, MASK_SLIDING, Workload,
                                                        make_inputs)
from parity import compare, forward_stats, oracle_problem

pytestmark = pytest.mark.gpu


def pack(x, lens):
    """[B, H, S, ...] -> [sum(lens), H, ...]"""
    return torch.cat([x[b, :, :L].transpose(0, 1) for b, L in enumerate(lens)], dim=0).contiguous()


def unpack(y, lens, S):
    """[T, H, ...] -> [B, H, S, ...], zeros past each length"""
    B = len(lens)
    out = torch.zeros((B, y.shape[1], S) + tuple(y.shape[2:]), dtype=y.dtype)
    t = 0
    for b, L in enumerate(lens):
        out[b, :, :L] = y[t:t + L].transpose(0, 1)
        t += L
    return out


def pack_lse(lse, lens):
    """[B, Hq, S] -> [Hq, T]"""
    return torch.cat([lse[b, :, :L] for b, L in enumerate(lens)], dim=1).contiguous()


def unpack_lse(y, lens, S):
    B = len(lens)
    out = torch.full((B, y.shape[0], S), float("inf"), dtype=y.dtype)
    t = 0
    for b, L in enumerate(lens):
        out[b, :, :L] = y[:, t:t + L]
        t += L
    return out


CASES = [
    # causal GQA with a sink, a zero-length and a one-token sequence
    (Workload("packed_causal_f16", "f16", B=4, Hq=8, Hkv=2, Sq=300, Skv=300,
              mask_kind=MASK_CAUSAL, sink=True, seed=61), [300, 1, 0, 173], None),
    (Workload("packed_swa_bf16", "bf16", B=3, Hq=4, Hkv=1, Sq=257, Skv=257,
              mask_kind=MASK_SLIDING, window=50, sink=True, seed=62), [257, 64, 190], None),
    # block mask with different query and key lengths per sequence
    (Workload("packed_bigbird_f16", "f16", B=3, Hq=2, Hkv=2, Sq=500, Skv=700,
              mask_kind=MASK_BLOCK, bx=48, by=80, block_pattern="bigbird", seed=63),
     [500, 123, 1], [650, 700, 37]),
    (Workload("packed_dense_bf16", "bf16", B=2, Hq=4, Hkv=2, Sq=200, Skv=260, mask_kind=MASK_NONE,
              sink=True, seed=64), [131, 200], [260, 77]),
]


def _setup(wl, lq, lk):
    lk = lq if lk is None else lk
    inp = make_inputs(wl)
    inp.seqlen_q = torch.tensor(lq, dtype=torch.int32)
    inp.seqlen_k = torch.tensor(lk, dtype=torch.int32)
    pb = oracle_problem(wl, inp)
    dev = "cuda"
    bm = inp.block_mask.to(dev) if inp.block_mask is not None else None
    mask = mab.packed_mask(wl.mask_kind, lq, lk, dev, window=wl.window, bx=wl.bx, by=wl.by,
                           block_mask=bm)
    mask.max_seqlen_q, mask.max_seqlen_k = wl.Sq, wl.Skv   # the padded shape's lengths
    return inp, pb, mask, lk


@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_packed_backward_matches_oracle(cuda_lib, case):
    wl, lq, lk = case
    inp, pb, mask, lk = _setup(wl, lq, lk)
    O, lse = forward_stats(wl, inp, pb)
    dev = "cuda"
    q, o, dO = (pack(x, lq).to(dev) for x in (inp.q, O, inp.dO))
    k, v = (pack(x, lk).to(dev) for x in (inp.k, inp.v))
    l = pack_lse(lse, lq).to(dev)
    sink = inp.sink.to(dev) if inp.sink is not None else None
    out = [torch.full_like(q, float("nan")), torch.full_like(k, float("nan")),
           torch.full_like(v, float("nan")),
           torch.full_like(sink, float("nan")) if sink is not None else None]
    mab.bwd(q, k, v, o, dO, l, sink, mask, wl.scale, out=out)
    torch.cuda.synchronize()
    ref = oracle.backward(pb, inp.q, inp.k, inp.v, O, inp.dO, lse)
    compare("dq", unpack(out[0].cpu(), lq, wl.Sq), ref["dq"], wl.dtype)
    compare("dk", unpack(out[1].cpu(), lk, wl.Skv), ref["dk"], wl.dtype)
    compare("dv", unpack(out[2].cpu(), lk, wl.Skv), ref["dv"], wl.dtype)
    if sink is not None:
        compare("dsink", out[3], ref["dsink"], wl.dtype, min_frac=1.0)


@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_packed_forward_matches_oracle(cuda_lib, case):
    wl, lq, lk = case
    inp, pb, mask, lk = _setup(wl, lq, lk)
    O_ref, lse_ref = oracle.forward(pb, inp.q, inp.k, inp.v)
    dev = "cuda"
    q = pack(inp.q, lq).to(dev)
    k, v = (pack(x, lk).to(dev) for x in (inp.k, inp.v))
    sink = inp.sink.to(dev) if inp.sink is not None else None
    o, lse = mab.fwd(q, k, v, sink, mask, wl.scale)
    torch.cuda.synchronize()
    assert tuple(lse.shape) == (wl.Hq, sum(lq))
    compare("o", unpack(o.cpu(), lq, wl.Sq), O_ref, wl.dtype)
    g = unpack_lse(lse.cpu(), lq, wl.Sq).double().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.all(np.abs(g[fin] - lse_ref[fin]) <= 1e-4 * (1 + np.abs(lse_ref[fin])))


def test_packed_equals_padded_bitwise(cuda_lib):
    # the same problem in both layouts runs the same arithmetic on the same
    # rows: the packed gradients are the padded ones, bit for bit
    wl, lq, lk = CASES[0]
    inp, pb, mask, lk = _setup(wl, lq, lk)
    O, lse = forward_stats(wl, inp, pb)
    dev = "cuda"
    pad_mask = mab.Mask(kind=wl.mask_kind, window=wl.window,
                        seqlen_q=inp.seqlen_q.to(dev), seqlen_k=inp.seqlen_k.to(dev))
    sink = inp.sink.to(dev)
    a = mab.bwd(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), O.to(dev), inp.dO.to(dev),
                lse.to(dev), sink, pad_mask, wl.scale)
    b = mab.bwd(pack(inp.q, lq).to(dev), pack(inp.k, lk).to(dev), pack(inp.v, lk).to(dev),
                pack(O, lq).to(dev), pack(inp.dO, lq).to(dev), pack_lse(lse, lq).to(dev), sink,
                mask, wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(unpack(b[0].cpu(), lq, wl.Sq), a[0].cpu())
    assert torch.equal(unpack(b[1].cpu(), lk, wl.Skv), a[1].cpu())
    assert torch.equal(unpack(b[2].cpu(), lk, wl.Skv), a[2].cpu())
    assert torch.equal(b[3], a[3])


def test_packed_fullsize_varlen_sampled(cuda_lib):
    # the variable-length GQA-sink workload (8 sequences of 256..2048 tokens,
    # 64 query heads in groups of 16) in the packed layout: dq on sampled rows,
    # dk, dv on sampled key rows, dsink of every head
    wl = BY_NAME["gqa_sink_varlen_causal_b8_s2048"]
    inp = make_inputs(wl)
    lq = [int(x) for x in inp.seqlen_q]
    pb = oracle_problem(wl, inp)
    O, lse = forward_stats(wl, inp, pb)
    dev = "cuda"
    mask = mab.packed_mask(wl.mask_kind, lq, lq, dev)
    mask.max_seqlen_q = mask.max_seqlen_k = wl.Sq
    q, o, dO = (pack(x, lq).to(dev) for x in (inp.q, O, inp.dO))
    k, v = (pack(x, lq).to(dev) for x in (inp.k, inp.v))
    dq, dk, dv, dsink = mab.bwd(q, k, v, o, dO, pack_lse(lse, lq).to(dev), inp.sink.to(dev), mask,
                                wl.scale)
    torch.cuda.synchronize()
    dq_p, dk_p, dv_p = unpack(dq.cpu(), lq, wl.Sq), unpack(dk.cpu(), lq, wl.Skv), \
        unpack(dv.cpu(), lq, wl.Skv)
    rng = np.random.default_rng(0)
    rows = rng.choice(wl.B * wl.Hq * wl.Sq, size=2048, replace=False)
    cols = rng.choice(wl.B * wl.Hkv * wl.Skv, size=1024, replace=False)
    q64, k64, v64, dO64 = (oracle._f64(t) for t in (inp.q, inp.k, inp.v, inp.dO))
    dl = oracle.delta(pb, O, dO64)
    compare("dq", dq_p.reshape(-1, wl.D)[rows], oracle.dq_rows(pb, q64, k64, v64, dO64, lse, dl,
                                                              rows), wl.dtype)
    rk, rv = oracle.dkdv_cols(pb, q64, k64, v64, dO64, lse, dl, cols)
    compare("dk", dk_p.reshape(-1, wl.D)[cols], rk, wl.dtype)
    compare("dv", dv_p.reshape(-1, wl.D)[cols], rv, wl.dtype)
    compare("dsink", dsink, oracle.dsink(pb, lse, dl), wl.dtype, min_frac=1.0)
